// fused_stream_cluster.cu -- the decode-sized fused MoE-LoRA shrink+expand on
// CUDA cores, streamed through persistent thread-block clusters (sm_103a).
//
// Computes, for every block b of every listed slot (l = lora_ids[z],
// e = expert_ids[l][b]), every adapter slice s and every pair f of that block
// (input row x_f: row f / topk, or row f with one row per pair; router weight
// w_f, 1 without weights):
//     t[j]    = sum_k x_f[k] * A_s[l][e][j][k]                (fp32)
//     y[f][off + s*N + n] = bf16((add_inputs ? y_in : 0) + w_f * sum_j B_s[l][e][n][j] * t[j])
// (prhub.com.cn summary of vLLM PR #42290, "Implementation breakdown" step 1:
// shrink by lora_a and expand by lora_b in one kernel, the rank dimension kept
// on chip.)  With naive block assignment (the summary's "Key source snippets":
// one program per pair) every pair is its own block, its LoRA and expert read
// from token_lora_mapping and topk_ids.
//
// At decode sizes a block holds one or a few real pairs, so the work is a
// skinny GEMV bound by streaming A[l,e] (r x K) and B[l,e] (N x r) from HBM.
// Design:
//   * work items are NPG pairs of one unit (block, slice): NPG = 1 for the
//     naive assignment and for decode batches (a block's second pair re-reads
//     the block's adapters, mostly from L2), NPG = 2 otherwise.
//   * a cluster of C CTAs (C = 1 with NPG = 1, up to 4 with NPG = 2) works on
//     one item at a time; CTA c owns the K columns [k_lo(c), k_hi(c)) of the
//     shrink and the output rows [n_lo(c), n_hi(c)) of the expand, so every
//     adapter byte of the item is read once, by one CTA.
//   * the items of aligned blocks come from a balanced list that every
//     cluster builds the same way (each block's real pairs counted, the items
//     ordered by pair count and dealt to the clusters in a snake); beyond
//     what the list covers, units are taken in turn (vLLM PR #32005: the work
//     list covers the active LoRAs only).
//   * two producer warps stream each item's share through a ring of 16 KB
//     stages: A boxes of r rows x kc columns by TMA (3-D tensor map), with
//     the kc columns of the pairs' x rows by bulk copies beside them; then B
//     rows by bulk copies, with the matching y_in pieces.  They run ahead
//     across items as far as the ring allows.
//   * eight consumer warps copy each stage to registers and hand it back,
//     then accumulate each CTA's partial t over its K columns; with C > 1 the
//     partial (fp32) goes into every peer's shared memory by st.async
//     (completion counted on the peer's mbarrier) and each CTA sums the C
//     partials in rank order (deterministic).  They then expand the item's
//     N rows.  t never leaves shared memory or registers.
// Every wait is bounded.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "device_utils.cuh"
#include "internal.h"
#include "stream_pipeline.cuh"

namespace cg = cooperative_groups;

namespace moe_lora {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarps = 2;           // ring stage st is filled by producer warp st % 2
constexpr int kThreads = kConsumers + kProducerWarps * 32;
constexpr int kNPG = 2;                     // most pairs a work item holds (NPG: 1 or kNPG)
constexpr int kDesc = 8;                    // work-item descriptors in flight
constexpr int kMaxStages = 24;
constexpr int kMaxCluster = 8;
constexpr int kMaxSlots = 128;              // listed slots the work list indexes
constexpr int kListCap = 32;                // work items a cluster takes from the balanced list
constexpr int kScanPerThread = 4;           // blocks a thread counts when the list is built
constexpr int kStageVecs = 1024;            // 16-byte adapter vectors per ring stage (16 KB)
constexpr int kRowsPerThread = 4;           // B rows per consumer thread and stage (one 8-column piece each)
constexpr int kVecsPerThread = kStageVecs / kConsumers;
static_assert(kRowsPerThread == kVecsPerThread, "a stage's B vectors are four per consumer thread");
constexpr int kCtasPerSm = 2;               // two rings and 16 consumer warps per SM

struct CsCfg {
  int C;             // CTAs per cluster
  int kc;            // A box columns per stage (power of two, <= 256)
  int lg_va;         // log2(kc / 8): vectors per A row
  int nb;            // B rows per stage
  int lg_vr;         // log2(r / 8): vectors per B row
  int stages;
  int stage_bytes;
  int npg;           // pairs per work item (the kernel's NPG)
  int a_bytes;       // r * kc * 2: the A box; npg x pieces of kc * 2 bytes follow
  int b_bytes;       // nb * r * 2: the B rows; npg y_in pieces of nb * 2 bytes follow
  int off_rbuf;      // fp32 [2][C][npg][r]: partial t received from each CTA
  int off_tfull;     // fp32 [2][npg][r]: summed t
  int off_stg;       // fp32 [npg][r]: this CTA's partial t
  int off_meta;
  int smem_bytes;
  int k_lo[kMaxCluster], k_hi[kMaxCluster], n_lo[kMaxCluster], n_hi[kMaxCluster];
};

// The A tensor map of every slice ([L*E, r, K], boxes of kc x r).
struct CsMaps {
  CUtensorMap a[kMaxSlices];
};

struct Desc {
  int s, le, ng;     // slice, flat (LoRA, expert) index, pairs (0: no more work)
  int f[kNPG];       // the pairs' flat indices
  int xrow[kNPG];    // their rows of x
  float w[kNPG];     // their router weights
};

struct CsMeta {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t dfull[kDesc], dempty[kDesc];
  uint64_t t_ready[2], t_free[2];
  Desc desc[kDesc];
  int prefix[kMaxSlots + 1];
  int lids[kMaxSlots];                  // lora_ids (the naive assignment: -1 where disabled)
  int pf[kProducerWarps][128];          // each producer: the current block's real pairs
  int scan[kThreads / 32][kNPG];        // per-warp item counts by pair count (list building)
  int list[kListCap];                   // this cluster's work items: (block, group, slice)
  int nlist;                            // their number, or -1: no list (every unit in turn)
  int abort;
};

// Bounded wait used when draining: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return;
}

// Row sums over a group of G consecutive lanes (G a power of two up to 32),
// each lane holding partial sums of the same V rows.  While a lane holds more
// than one row, a step with lane distance d hands half of its rows to the
// partner and keeps the other half plus the partner's share of it; once one
// row is left, the remaining steps are plain butterflies.  A lane ends with
// rows_reduce_out() consecutive row sums, starting at row rows_reduce_base().
template <int G, int V>
__host__ __device__ constexpr int rows_reduce_out() {
  return G >= V ? 1 : V / G;
}
template <int G, int V>
__device__ __forceinline__ int rows_reduce_base(int lane) {
  int base = 0, n = V;
#pragma unroll
  for (int d = G / 2; d >= 1; d >>= 1)
    if (n > 1) {
      n >>= 1;
      if (lane & d) base += n;
    }
  return base;
}
// Of the lanes holding the same sums, the one that writes them.
template <int G, int V>
__device__ __forceinline__ bool rows_reduce_keeper(int lane) {
  return G <= V || (lane & (G / V - 1)) == 0;
}
template <int G, int V>
__device__ __forceinline__ void rows_reduce(float (&v)[V], int lane) {
  int n = V;
#pragma unroll
  for (int d = G / 2; d >= 1; d >>= 1) {
    if (n > 1) {
      const int h = n >> 1;
      const bool up = (lane & d) != 0;
#pragma unroll
      for (int k = 0; k < V / 2; ++k)
        if (k < h) {
          const float send = up ? v[k] : v[k + h];
          const float keep = up ? v[k + h] : v[k];
          v[k] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], d);
    }
  }
}

__device__ __forceinline__ int find_slot(const int *prefix, int nact, int item) {
  int lo = 0, hi = nact;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid;
  }
  return lo;
}

// The sorted blocks' work as a balanced list, built by all threads of one CTA
// per cluster from the same inputs (so every cluster sees the same order).  Block b
// holds n_b real pairs, applied NPG at a time: n_b / NPG items of NPG pairs
// and one of n_b % NPG pairs (if any), each once per slice.  The items are
// ordered by their pair count (most first), then by block, group and slice,
// and dealt out to the G clusters in a snake (0 .. G-1, G-1 .. 0, ...): each
// cluster gets floor or ceil(items / G) of them, one per round, and the
// heavy ones are spread.  Entry `round` of cluster g's list encodes
// (block << 8) | (group << 2) | slice.  No list (nlist = -1) when the blocks
// outnumber what the threads count in one pass or a share exceeds kListCap;
// the units are then taken in turn.
template <int NPG>
__device__ void build_item_list(CsMeta &meta, const FusedArgs &p, int nact, int S, int P, int G, int g, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int nblk = meta.prefix[nact];
  if (nblk > kThreads * kScanPerThread) {
    if (tid == 0) meta.nlist = -1;
    __syncthreads();
    return;
  }
  // this thread's blocks: a contiguous run, so that the scan follows block order
  const int per = (nblk + kThreads - 1) / kThreads;
  const int b0 = tid * per;
  int nbk[kScanPerThread];
  int cnt[NPG];   // this thread's items with k + 1 pairs
#pragma unroll
  for (int k = 0; k < NPG; ++k) cnt[k] = 0;
#pragma unroll
  for (int i = 0; i < kScanPerThread; ++i) {
    nbk[i] = 0;
    const int b = b0 + i;
    if (i < per && b < nblk) {
      const int z = find_slot(meta.prefix, nact, b);
      const int l = meta.lids[z];
      const int32_t *ids =
          p.sorted_token_ids + (size_t)l * p.max_num_tokens_padded + (size_t)(b - meta.prefix[z]) * p.block_size;
      // In the align's layout a block's real pairs come first and the
      // sentinel fills its tail, so the count stops at the first entry that
      // is not a pair: a decode block takes one 16-byte read.  (The producers
      // flag a block that breaks this layout.)
      int n = 0;
      if ((reinterpret_cast<uintptr_t>(ids) & 15) == 0 && (p.block_size & 3) == 0) {
        for (int k = 0; k < p.block_size; k += 4) {
          const int4 v = __ldg(reinterpret_cast<const int4 *>(ids + k));
          const unsigned m4 = (v.x >= 0 && v.x < P) | (v.y >= 0 && v.y < P) << 1 | (v.z >= 0 && v.z < P) << 2 |
                              (v.w >= 0 && v.w < P) << 3;
          if (m4 & (m4 + 1u)) flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);   // a pair after a sentinel
          const int c4 = __popc(m4);
          n += c4;
          if (c4 < 4) break;
        }
      } else {
        for (int k = 0; k < p.block_size; ++k) {
          const int f = __ldg(ids + k);
          if (f < 0 || f >= P) break;
          ++n;
        }
      }
      nbk[i] = n;
      // (unrolled selects, not an index: the counts stay in registers)
#pragma unroll
      for (int k = 0; k < NPG; ++k) cnt[k] += (k == NPG - 1 ? n / NPG : 0) + (n % NPG == k + 1 ? 1 : 0);
    }
  }
  // exclusive scan of the counts over the threads (block order)
  int incl[NPG];
#pragma unroll
  for (int k = 0; k < NPG; ++k) {
    int v = cnt[k];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += o;
    }
    incl[k] = v;
    if (lane == 31) meta.scan[warp][k] = v;
  }
  __syncthreads();
  int run[NPG], off[NPG];
  long long items = 0;
#pragma unroll
  for (int k = NPG - 1; k >= 0; --k) {
    int before = 0, all = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const int v = meta.scan[w][k];
      if (w < warp) before += v;
      all += v;
    }
    run[k] = before + incl[k] - cnt[k];   // rank of this thread's first item with k + 1 pairs
    off[k] = (int)items;                   // items with more pairs come first
    items += all;
  }
  const long long total = items * S;
  const long long rounds = (total + G - 1) / G;
  if (rounds > kListCap) {
    if (tid == 0) meta.nlist = -1;
    __syncthreads();
    return;
  }
  // this cluster's count: one per full round, and one in the last partial
  // round when the snake's direction there covers it
  const long long full = total / G, rest = total - full * G;
  const bool in_last = rest > 0 && ((full & 1) ? g >= G - rest : g < rest);
  if (tid == 0) meta.nlist = (int)(full + (in_last ? 1 : 0));
#pragma unroll
  for (int i = 0; i < kScanPerThread; ++i) {
    const int n = nbk[i], b = b0 + i;
    const int groups = n / NPG + (n % NPG ? 1 : 0);
    for (int j = 0; j < groups; ++j) {
      const int kk = (j < n / NPG ? NPG : n % NPG) - 1;
      int rank_k = 0;
#pragma unroll
      for (int k = 0; k < NPG; ++k)
        if (k == kk) rank_k = off[k] + run[k]++;
      const long long idx0 = (long long)rank_k * S;
      for (int s = 0; s < S; ++s) {
        const long long idx = idx0 + s, round = idx / G, pos = idx - round * G;
        if (((round & 1) ? G - 1 - pos : pos) == g) meta.list[round] = (b << 8) | (j << 2) | s;
      }
    }
  }
  __syncthreads();
}

// log2 of the 16-byte vectors per A box row: the box has min(256, 8192 / r)
// columns (at most kStageVecs vectors), r = 8 << LG_VR.
template <int LG_VR>
constexpr int kLgVa = (7 - LG_VR) < 5 ? (7 - LG_VR) : 5;

// LG_VR = log2(rank / 8): the rank (8 .. 128) fixes every per-thread loop.
template <bool NAIVE, int LG_VR, int NPG>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    fused_cluster_stream_kernel(const __grid_constant__ CsMaps maps, const FusedArgs p, const CsCfg cfg) {
  extern __shared__ __align__(1024) uint8_t smem[];
  CsMeta &meta = *reinterpret_cast<CsMeta *>(smem + cfg.off_meta);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = cfg.C;
  const int c = (int)cg::this_cluster().block_rank();
  const int r = p.rank, K = p.K, N = p.N, E = p.num_experts, P = p.M * p.topk;
  const int nact = p.num_active_loras, S = p.num_slices;
  const int kc = cfg.kc, nb = cfg.nb, NS = cfg.stages;
  volatile int *abort = &meta.abort;
  uint8_t *ring = smem;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&meta.full[s], 1);
      mbar_init(&meta.empty[s], kConsumerWarps);
    }
    for (int d = 0; d < kDesc; ++d) {
      mbar_init(&meta.dfull[d], 1);
      mbar_init(&meta.dempty[d], kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&meta.t_ready[b], 1);
      mbar_init(&meta.t_free[b], C);
    }
    meta.abort = 0;
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane < S) prefetch_tensor_map(&maps.a[lane]);
  // peers arrive on and write to this CTA's barriers and buffers: every CTA of
  // the cluster has initialised them before any CTA goes on
  cluster_arrive_release();
  cluster_wait();

  wait_for_prior_grid();   // align outputs (and every other input) are read from here on
  long long units;
  if (!NAIVE) {
    // blocks per listed slot and their prefix sum; the slots' LoRA ids.  With
    // at most 2 x 128 LoRAs, every LoRA's block count is read beside lora_ids
    // (one round trip, not two), staged in the producers' pair lists.
    int *nbl = &meta.pf[0][0];
    const bool staged = p.max_loras <= kProducerWarps * 128;
    if (staged) {
      for (int l = tid; l < p.max_loras; l += blockDim.x) {
        int nb_l = -1;   // -1: disabled
        if (!p.adapter_enabled || __ldg(p.adapter_enabled + l) != 0)
          nb_l = max(0, min(__ldg(p.num_tokens_post_padded + l) / p.block_size, p.max_num_m_blocks));
        nbl[l] = nb_l;
      }
    }
    int lz[(kMaxSlots + kThreads - 1) / kThreads];
#pragma unroll
    for (int i = 0; i < (kMaxSlots + kThreads - 1) / kThreads; ++i) {
      const int z = tid + i * kThreads;
      lz[i] = z < nact ? __ldg(p.lora_ids + z) : 0;
    }
    if (staged) __syncthreads();
#pragma unroll
    for (int i = 0; i < (kMaxSlots + kThreads - 1) / kThreads; ++i) {
      const int z = tid + i * kThreads;
      if (z >= nact) continue;
      const int l = lz[i];
      int nb_z = 0;
      if (l < 0 || l >= p.max_loras) {
        if (blockIdx.x == 0) flag_error(p.err, MOE_LORA_DEVERR_LORA_ID);
      } else if (staged) {
        nb_z = max(0, nbl[l]);
      } else if (!p.adapter_enabled || __ldg(p.adapter_enabled + l) != 0) {
        nb_z = __ldg(p.num_tokens_post_padded + l) / p.block_size;
        nb_z = max(0, min(nb_z, p.max_num_m_blocks));
      }
      meta.prefix[z + 1] = nb_z;
      meta.lids[z] = l;   // a slot with blocks has a valid id
    }
    __syncthreads();
    if (tid == 0) {
      meta.prefix[0] = 0;
      for (int z = 0; z < nact; ++z) meta.prefix[z + 1] += meta.prefix[z];
    }
    __syncthreads();
    units = (long long)meta.prefix[nact] * S;
  } else {
    for (int z = tid; z < nact; z += blockDim.x) {
      const int l = __ldg(p.lora_ids + z);
      if (l < 0 || l >= p.max_loras) {
        if (blockIdx.x == 0) flag_error(p.err, MOE_LORA_DEVERR_LORA_ID);
        meta.lids[z] = -1;
      } else {
        meta.lids[z] = (!p.adapter_enabled || __ldg(p.adapter_enabled + l) != 0) ? l : -1;
      }
    }
    __syncthreads();
    units = (long long)P * S;
  }
  const int G = gridDim.x / C, g = blockIdx.x / C;
  if (!NAIVE) {
    // the cluster's CTAs take the same items: rank 0 builds the list and
    // writes it into the others' shared memory
    if (c == 0) {
      build_item_list<NPG>(meta, p, nact, S, P, G, g, tid);
      for (int i = tid; i < (kListCap + 1) * (C - 1); i += kThreads) {
        const int dst = 1 + i / (kListCap + 1), k = i - (dst - 1) * (kListCap + 1);
        int *src = k < kListCap ? &meta.list[k] : &meta.nlist;
        st_cluster_u32(cluster_map(smem_addr(src), dst), (uint32_t)*src);
      }
    }
    if (C > 1) {
      cluster_arrive_release();
      cluster_wait();
    }
  }
  const int k_lo = cfg.k_lo[c], k_hi = cfg.k_hi[c], n_lo = cfg.n_lo[c], n_hi = cfg.n_hi[c];

  if (warp >= kConsumerWarps) {
    // ================================================= producer warps
    // Both walk the same work items; producer pw fills the ring stages whose
    // index is pw (mod 2), and producer 0 writes the work-item descriptors.
    // Stage order: A(0), A(1), B(0), A(2), B(1), ..., B(n-1): the consumers
    // shrink item i + 1 while item i's partial t is exchanged.
    const int pw = warp - kConsumerWarps;
    int *pf = meta.pf[pw];
    uint32_t it = 0, issued = 0, item = 0;   // it, issued: lane 0's count of stages (all / issued)
    const bool lead = lane == 0;
    // the previous item (its B stages follow the current item's A stages)
    bool have_prev = false;
    int pv_s = 0, pv_le = 0, pv_ng = 0, pv_f[NPG];
    auto issue_b = [&](int s_, int le_, int ng_, const int (&f_)[NPG]) {
      if (!lead) return;
      const uint16_t *Bm = slice_b(p, s_) + (size_t)le_ * N * r;
      const int col0 = p.y_offset + s_ * N;
      for (int n0 = n_lo; n0 < n_hi; n0 += nb, ++it) {
        if (((it % NS) & 1) != (uint32_t)pw || *abort) continue;
        const int st = it % NS;
        if (it >= (uint32_t)NS && !mbar_wait(&meta.empty[st], ((it / NS) - 1) & 1, abort, p.err)) continue;
        issued = it + 1;
        uint8_t *stage = ring + (size_t)st * cfg.stage_bytes;
        const int rows = min(nb, n_hi - n0);
        const uint32_t bb = (uint32_t)rows * r * 2, yb = (uint32_t)rows * 2;
        mbar_arrive_expect_tx(&meta.full[st], bb + (p.add_inputs ? ng_ * yb : 0));
        bulk_g2s(stage, Bm + (size_t)n0 * r, bb, &meta.full[st]);
        if (p.add_inputs) {
#pragma unroll
          for (int q = 0; q < NPG; ++q)
            if (q < ng_)
              bulk_g2s(stage + cfg.b_bytes + q * nb * 2, p.y + (size_t)f_[q] * p.ldy + col0 + n0, yb, &meta.full[st]);
        }
      }
    };
    // the units in turn (u = g, g + G, ...), or this cluster's entries of the
    // balanced list (one group of one block's pairs each)
    const int nlist = NAIVE ? -1 : meta.nlist;
    const long long nwork = nlist >= 0 ? nlist : (units > g ? (units - 1 - g) / G + 1 : 0);
    for (long long w = 0; w < nwork; ++w) {
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
      long long u = g + w * G;
      int jsel = -1;   // the one group this entry takes (-1: all of the unit's)
      if (nlist >= 0) {
        const int code = meta.list[w];
        jsel = (code >> 2) & 63;
        u = (long long)(code >> 8) * S + (code & 3);
      }
      int s, le, np = 0;
      if (!NAIVE) {
        const int gb = (int)(u / S);
        s = (int)(u - (long long)gb * S);
        const int z = find_slot(meta.prefix, nact, gb);
        const int l = meta.lids[z];
        const int b = gb - meta.prefix[z];
        const int e = __ldg(p.expert_ids + (size_t)l * p.max_num_m_blocks + b);
        if (e < 0 || e >= E) {
          if (lead && pw == 0 && c == 0 && s == 0) flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
          continue;
        }
        le = l * E + e;
        const int32_t *ids = p.sorted_token_ids + (size_t)l * p.max_num_tokens_padded + (size_t)b * p.block_size;
        bool gap = false;   // an entry that is not a pair has been seen
        for (int i0 = 0; i0 < p.block_size; i0 += 32) {
          const int f = i0 + lane < p.block_size ? __ldg(ids + i0 + lane) : P;
          const bool real = f >= 0 && f < P;
          if ((f < 0 || f > P) && pw == 0 && c == 0 && s == 0) flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);
          const unsigned bal = __ballot_sync(0xffffffffu, real);
          // the align's layout: real pairs first, then the sentinel (the
          // balanced list counts on it)
          if (((gap && bal) || (bal & (bal + 1u))) && lead && pw == 0 && c == 0 && s == 0)
            flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);
          gap = gap || bal != 0xffffffffu;
          if (real) pf[np + __popc(bal & ((1u << lane) - 1u))] = f;
          np += __popc(bal);
        }
        __syncwarp();
      } else {
        const int f = (int)(u / S);
        s = (int)(u - (long long)f * S);
        const int l = __ldg(p.token_lora_mapping + f / p.topk);
        const int e = __ldg(p.topk_ids + f);
        bool listed = false;
        for (int z = lane; z < nact; z += 32) listed |= l >= 0 && meta.lids[z] == l;
        if (!__any_sync(0xffffffffu, listed)) continue;
        if (e < 0 || e >= E) {
          if (lead && pw == 0 && c == 0 && s == 0) flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
          continue;
        }
        le = l * E + e;
        if (lead) pf[0] = f;
        __syncwarp();
        np = 1;
      }
      const int g_first = jsel < 0 ? 0 : jsel * NPG, g_end = jsel < 0 ? np : min(np, g_first + NPG);
      for (int g0 = g_first; g0 < g_end; g0 += NPG) {
        const int ng = min(NPG, np - g0);
        int fq = -1, xq = 0;
        if (lane < ng) {
          fq = pf[g0 + lane];
          xq = x_row(p, fq);
        }
        if (pw == 0) {
          const int d = item % kDesc;
          if (item >= kDesc) mbar_wait(&meta.dempty[d], ((item / kDesc) - 1) & 1, abort, p.err);
          Desc &ds = meta.desc[d];
          if (lane < ng) {
            ds.f[lane] = fq;
            ds.xrow[lane] = xq;
            ds.w[lane] = route_weight(p, fq);
          }
          if (lead) {
            ds.s = s;
            ds.le = le;
            ds.ng = ng;
          }
          __syncwarp();
          if (lead) mbar_arrive(&meta.dfull[d]);
        }
        // the pairs' rows, in every lane (lane q < ng holds pair q)
        int xr[NPG], fr[NPG];
#pragma unroll
        for (int q = 0; q < NPG; ++q) {
          xr[q] = __shfl_sync(0xffffffffu, xq, q);
          fr[q] = __shfl_sync(0xffffffffu, fq, q);
        }
        // Lane 0 issues this producer's stages.  After an abort it issues
        // nothing more; `issued` bounds the drain below.
        // A boxes (r x kc) of this item with the pairs' x pieces beside them
        if (lead) {
          for (int k0 = k_lo; k0 < k_hi; k0 += kc, ++it) {
            if (((it % NS) & 1) != (uint32_t)pw || *abort) continue;
            const int st = it % NS;
            if (it >= (uint32_t)NS && !mbar_wait(&meta.empty[st], ((it / NS) - 1) & 1, abort, p.err)) continue;
            issued = it + 1;
            uint8_t *stage = ring + (size_t)st * cfg.stage_bytes;
            const uint32_t xb = (uint32_t)min(kc, k_hi - k0) * 2;
            mbar_arrive_expect_tx(&meta.full[st], (uint32_t)cfg.a_bytes + ng * xb);
            tma_load_3d(stage, &maps.a[s], k0, 0, le, &meta.full[st]);
#pragma unroll
            for (int q = 0; q < NPG; ++q)
              if (q < ng) bulk_g2s(stage + cfg.a_bytes + q * kc * 2, p.x + (size_t)xr[q] * K + k0, xb, &meta.full[st]);
          }
        }
        // then the B rows of the previous item
        if (have_prev) issue_b(pv_s, pv_le, pv_ng, pv_f);
        have_prev = true;
        pv_s = s;
        pv_le = le;
        pv_ng = ng;
#pragma unroll
        for (int q = 0; q < NPG; ++q) pv_f[q] = fr[q];
        ++item;
        __syncwarp();
      }
    }
    // end of the work: a descriptor with no pairs.  It goes out before the
    // last item's B stages: the consumers read it before they expand that
    // item, and those stages may be more than the ring holds.
    if (pw == 0) {
      const int d = item % kDesc;
      if (item >= kDesc) mbar_wait(&meta.dempty[d], ((item / kDesc) - 1) & 1, abort, p.err);
      if (lead) {
        meta.desc[d].ng = 0;
        mbar_arrive(&meta.dfull[d]);
      }
    }
    __syncwarp();
    if (have_prev) issue_b(pv_s, pv_le, pv_ng, pv_f);
    __syncwarp();
    // every copy this producer issued has landed before the CTA exits (its
    // stages are those with index = pw mod 2, so the last fill it issued to a
    // stage is that stage's last fill)
    if (lead)
      for (int st = pw; st < NS && (uint32_t)st < issued; st += kProducerWarps) {
        const uint32_t last = st + (uint32_t)NS * ((issued - 1 - st) / NS);
        drain_wait(&meta.full[st], (last / NS) & 1);
      }
    __syncwarp();
  } else {
    // ================================================= consumer warps
    // Shrink: thread tid owns the A vectors g = i * 256 + tid (i < 4) of a
    // stage: row g / va, column vector g % va; a warp reads 512 contiguous
    // bytes per step.  Expand: thread tid owns column vector tid % vr of the
    // four B rows 4 (tid / vr) .. + 3 (a quarter warp reads 128 contiguous
    // bytes); the vr lanes of a row group then sum each row between them.
    constexpr int lg_vr = LG_VR, vr = 1 << LG_VR;
    constexpr int lg_va = kLgVa<LG_VR>, va = 1 << lg_va;
    constexpr int kOut = rows_reduce_out<vr, kRowsPerThread>();           // row sums a lane ends with
    const int cv_a = (tid & (va - 1)) * 8;                                // this thread's A column (elements)
    const int cv_b = tid & (vr - 1);                                      // its B column vector
    const int erow0 = (tid >> lg_vr) * kRowsPerThread;                    // its first B row in a stage
    const int obase = rows_reduce_base<vr, kRowsPerThread>(lane);         // its first summed row (of erow0 ..)
    const bool store_lane = rows_reduce_keeper<vr, kRowsPerThread>(lane); // it writes those rows
    float *rbuf = reinterpret_cast<float *>(smem + cfg.off_rbuf);
    float *tfull = reinterpret_cast<float *>(smem + cfg.off_tfull);
    float *stg = reinterpret_cast<float *>(smem + cfg.off_stg);
    uint32_t it = 0;
    uint32_t cst = 0, cph = 0;   // it % NS and (it / NS) & 1, kept without a division
    auto advance = [&] {
      ++it;
      if (++cst == (uint32_t)NS) {
        cst = 0;
        cph ^= 1;
      }
    };
    // the previous item, whose exchange overlaps this item's shrink
    bool have_prev = false;
    uint32_t pv_item = 0;

    // Wait for the C partials of item `itm`, sum them (rank order), free the
    // receive buffer on every CTA, and expand the item's output rows.
    auto finish = [&](uint32_t itm) {
      const int d = itm % kDesc, b = itm & 1;
      const Desc &ds = meta.desc[d];
      const int ng = min(ds.ng, NPG);
      const int s = ds.s;
      float wq[NPG];
      int fq[NPG];
#pragma unroll
      for (int q = 0; q < NPG; ++q) {
        wq[q] = q < ng ? ds.w[q] : 0.f;
        fq[q] = q < ng ? ds.f[q] : 0;
      }
      if (tid == 0) mbar_wait_cluster(&meta.t_ready[b], (itm >> 1) & 1, abort, p.err);
      named_barrier(1, kConsumers);
      float *tf = tfull + (size_t)b * NPG * r;
      for (int i = tid; i < ng * r; i += kConsumers) {
        float sum = 0.f;
        for (int q = 0; q < C; ++q) sum += rbuf[(size_t)(b * C + q) * NPG * r + i];
        tf[i] = sum;
      }
      named_barrier(1, kConsumers);
      // this CTA's buffer b is free again: tell every CTA of the cluster.  The
      // reads of rbuf above are complete (their sums were stored before the
      // barrier), so the arrive needs no release, which would first wait for
      // this thread's y stores still in flight.
      if (tid == 0)
        for (int dst = 0; dst < C; ++dst) mbar_arrive_remote_relaxed(cluster_map(smem_addr(&meta.t_free[b]), dst));
      // ---- expand: this CTA's output rows
      const int col0 = p.y_offset + s * N;
      for (int n0 = n_lo; n0 < n_hi; n0 += nb, advance()) {
        const int st = cst;
        mbar_wait(&meta.full[st], cph, abort, p.err);
        const uint8_t *stage = ring + (size_t)st * cfg.stage_bytes;
        const int rows = min(nb, n_hi - n0);
        // B vectors and y_in values to registers, then the stage goes back
        uint4 bv[kRowsPerThread];
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j)
          bv[j] = erow0 + j < rows ? *reinterpret_cast<const uint4 *>(stage + ((size_t)(erow0 + j) * vr + cv_b) * 16)
                                   : make_uint4(0u, 0u, 0u, 0u);
        float old[kOut][NPG];
#pragma unroll
        for (int k = 0; k < kOut; ++k)
#pragma unroll
          for (int q = 0; q < NPG; ++q) {
            const int row = erow0 + obase + k;
            old[k][q] = p.add_inputs && store_lane && q < ng && row < rows
                            ? bf16_bits_to_float(reinterpret_cast<const uint16_t *>(stage + cfg.b_bytes + q * nb * 2)[row])
                            : 0.f;
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta.empty[st]);
        // pair by pair: this thread's 8 t columns (the same in every stage of
        // the item), its 8-column piece of each of its rows, the sums over the
        // vr lanes of each row (ng is the same in every lane), the stores.
        // (Widening each B vector once for all pairs would hold their t
        // columns and sums at once: more registers than a thread has here.)
#pragma unroll
        for (int q = 0; q < NPG; ++q)
          if (q < ng) {
            const ulonglong2 t01 = *reinterpret_cast<const ulonglong2 *>(tf + q * r + cv_b * 8);
            const ulonglong2 t23 = *reinterpret_cast<const ulonglong2 *>(tf + q * r + cv_b * 8 + 4);
            float o[kRowsPerThread];
#pragma unroll
            for (int j = 0; j < kRowsPerThread; ++j) {
              f32x2 bf[4];
              unpack_v(bv[j], bf);
              f32x2 acc = ffma2(bf[0], t01.x, 0ull);
              acc = ffma2(bf[1], t01.y, acc);
              acc = ffma2(bf[2], t23.x, acc);
              acc = ffma2(bf[3], t23.y, acc);
              o[j] = f2_sum(acc);
            }
            rows_reduce<vr, kRowsPerThread>(o, lane);
            if (store_lane) {
              uint16_t *yq = p.y + (size_t)fq[q] * p.ldy + col0 + n0;
#pragma unroll
              for (int k = 0; k < kOut; ++k) {
                const int row = erow0 + obase + k;
                if (row < rows) yq[row] = float_to_bf16_bits(o[k] * wq[q] + old[k][q]);
              }
            }
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&meta.dempty[d]);
    };

    for (uint32_t item = 0;; ++item) {
      const int d = item % kDesc;
      mbar_wait(&meta.dfull[d], (item / kDesc) & 1, abort, p.err);
      const Desc &ds = meta.desc[d];
      const int ng = min(ds.ng, NPG);
      // every consumer thread takes the same decision (no thread may leave
      // the named barriers below to the others)
      const bool more = named_barrier_and(1, kConsumers, ng > 0 && !*abort);
      if (more) {
        const int b = item & 1;
        // this CTA receives C partials of ng x r floats for the item
        if (tid == 0) mbar_arrive_expect_tx(&meta.t_ready[b], (uint32_t)(C * ng * r * 4));

        // ---- shrink: this CTA's partial t over its K columns
        float acc[kVecsPerThread][NPG];
#pragma unroll
        for (int i = 0; i < kVecsPerThread; ++i)
#pragma unroll
          for (int q = 0; q < NPG; ++q) acc[i][q] = 0.f;
        for (int k0 = k_lo; k0 < k_hi; k0 += kc, advance()) {
          const int st = cst;
          mbar_wait(&meta.full[st], cph, abort, p.err);
          const uint8_t *stage = ring + (size_t)st * cfg.stage_bytes;
          // The stage's vectors go to registers and the stage is handed back
          // before any arithmetic, so that its next fill is in flight while
          // this one is reduced.  This thread's column vector is the same in
          // all its rows (va divides the consumer threads): its x pieces are
          // read once per stage.
          const bool live = cv_a < k_hi - k0;
          uint4 xv[NPG], av[kVecsPerThread];
          if (live) {
#pragma unroll
            for (int q = 0; q < NPG; ++q)
              if (q < ng) xv[q] = *reinterpret_cast<const uint4 *>(stage + cfg.a_bytes + (q * kc + cv_a) * 2);
#pragma unroll
            for (int i = 0; i < kVecsPerThread; ++i)
              if (i * kConsumers < r * va) av[i] = *reinterpret_cast<const uint4 *>(stage + (size_t)(i * kConsumers + tid) * 16);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&meta.empty[st]);
          if (live) {
#pragma unroll
            for (int q = 0; q < NPG; ++q)
              if (q < ng) {
#pragma unroll
                for (int i = 0; i < kVecsPerThread; ++i)
                  if (i * kConsumers < r * va) acc[i][q] = dot8_bf16_acc(av[i], xv[q], acc[i][q]);
              }
          }
        }
        // sum each row's partial over the va lanes that share it (va <= 32:
        // consecutive lanes); the first of them keeps it
#pragma unroll
        for (int i = 0; i < kVecsPerThread; ++i)
#pragma unroll
          for (int q = 0; q < NPG; ++q)
            if (q < ng) {
              float v = acc[i][q];
#pragma unroll
              for (int dd = va >> 1; dd > 0; dd >>= 1) v += __shfl_xor_sync(0xffffffffu, v, dd);
              acc[i][q] = v;
            }
        if ((tid & (va - 1)) == 0) {
#pragma unroll
          for (int i = 0; i < kVecsPerThread; ++i) {
            const int row = (i * kConsumers + tid) >> lg_va;
            if (row < r)
#pragma unroll
              for (int q = 0; q < NPG; ++q)
                if (q < ng) stg[q * r + row] = acc[i][q];
          }
        }
        // every CTA is done with its buffer b (two items back) before this
        // item's partials go into it
        if (item >= 2 && tid == 0) mbar_wait_cluster(&meta.t_free[b], ((item >> 1) - 1) & 1, abort, p.err);
        named_barrier(1, kConsumers);
        {
          const int nv4 = ng * r / 4;
          const uint32_t src = smem_addr(rbuf + (size_t)(b * C + c) * NPG * r);
          const uint32_t bar = smem_addr(&meta.t_ready[b]);
          for (int i = tid; i < C * nv4; i += kConsumers) {
            const int dst = i / nv4, v = i - dst * nv4;
            const float4 val = reinterpret_cast<const float4 *>(stg)[v];
            st_async_v4(cluster_map(src + v * 16, dst), val, cluster_map(bar, dst));
          }
        }
      }
      // the previous item's exchange has had this item's shrink to land
      if (have_prev) finish(pv_item);
      if (!more) break;
      have_prev = true;
      pv_item = item;
    }
  }
  // no CTA leaves while a peer may still write into its shared memory or
  // arrive on its barriers
  cluster_arrive_release();
  cluster_wait();
}

int ilog2(int v) {
  int l = 0;
  while ((1 << (l + 1)) <= v) ++l;
  return l;
}

// Geometry and shared-memory layout for C CTAs per cluster and npg pairs per
// work item.
bool layout(const FusedArgs &f, const DeviceInfo &dev, int C, int npg, CsCfg *cfg) {
  const int r = f.rank;
  if (r < 8 || r > 128 || (r & (r - 1)) != 0) return false;   // ranks 8, 16, 32, 64, 128
  cfg->C = C;
  cfg->npg = npg;
  int kc = 256;
  while (r * kc > kStageVecs * 8) kc >>= 1;   // the A box holds at most kStageVecs vectors
  cfg->kc = kc;
  cfg->lg_va = ilog2(kc / 8);   // equals kLgVa<log2(r / 8)> of the kernel
  cfg->nb = std::min(512, kStageVecs * 8 / r);
  cfg->lg_vr = ilog2(r / 8);
  cfg->a_bytes = r * kc * 2;
  cfg->b_bytes = cfg->nb * r * 2;
  const int st_a = cfg->a_bytes + npg * kc * 2, st_b = cfg->b_bytes + npg * cfg->nb * 2;
  cfg->stage_bytes = (std::max(st_a, st_b) + 127) / 128 * 128;   // TMA destinations: 128-byte aligned
  const int k8 = f.K / 8, n8 = f.N / 8;
  for (int i = 0; i < kMaxCluster; ++i) {
    const int cc = i < C ? i : C - 1;
    cfg->k_lo[i] = (cc * k8 / C) * 8;
    cfg->k_hi[i] = ((cc + 1) * k8 / C) * 8;
    cfg->n_lo[i] = (cc * n8 / C) * 8;
    cfg->n_hi[i] = ((cc + 1) * n8 / C) * 8;
  }
  const int rbuf = 2 * C * npg * r * 4, tfull = 2 * npg * r * 4, stg = npg * r * 4;
  const int fixed = rbuf + tfull + stg + ((int)sizeof(CsMeta) + 127) / 128 * 128;
  // kCtasPerSm CTAs share an SM's 228 KB (each CTA also reserves 1 KB)
  const int budget = std::min((int)dev.max_smem_optin, 228 * 1024 / kCtasPerSm - 1024);
  int stages = (budget - fixed) / cfg->stage_bytes;
  stages = std::min(stages, kMaxStages);
  if (stages < 4) return false;
  cfg->stages = stages;
  cfg->off_rbuf = stages * cfg->stage_bytes;
  cfg->off_tfull = cfg->off_rbuf + rbuf;
  cfg->off_stg = cfg->off_tfull + tfull;
  cfg->off_meta = cfg->off_stg + stg;
  cfg->smem_bytes = cfg->off_meta + ((int)sizeof(CsMeta) + 127) / 128 * 128;
  return cfg->smem_bytes <= budget;
}

template <bool NAIVE, int LG_VR, int NPG>
int resident_clusters(const CsCfg &cfg, const DeviceInfo &dev) {
  struct Entry {
    int device, C, smem, clusters;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].device == dev.device && cache[i].C == cfg.C && cache[i].smem == cfg.smem_bytes)
      return cache[i].clusters;
  const void *fn = (const void *)fused_cluster_stream_kernel<NAIVE, LG_VR, NPG>;
  int clusters = 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes) == cudaSuccess) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(cfg.C, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = cfg.smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cfg.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&clusters, fn, &lc) != cudaSuccess) clusters = 0;
  }
  cudaGetLastError();   // a failed query leaves no sticky error
  if (clusters <= 0) clusters = std::max(1, kCtasPerSm * dev.sm_count / cfg.C);
  if (n < 32) cache[n++] = {dev.device, cfg.C, cfg.smem_bytes, clusters};
  return clusters;
}

// Work items the call may have (host bound): pairs x slices (the naive
// assignment, or blocks applied one pair at a time), else blocks x slices.
long long unit_bound(const FusedArgs &f, bool naive, int npg) {
  if (naive || npg == 1) return (long long)f.M * f.topk * f.num_slices;
  return fused_block_bound(f.M, f.topk, f.num_experts, f.num_active_loras, f.block_size) * f.num_slices;
}

// Pairs per work item and cluster size.  Measured on the gpt-oss-shaped w2
// decode (rank 64, K = N = 2880) and the Qwen3-shaped w13 decode.  Pairs of
// the naive assignment: one per item, clusters of one CTA.  Blocks of the
// align output when the pairs are no more than the (LoRA, expert) pairs
// (decode: mostly one pair per block): one pair per item, from a balanced
// list, clusters of one CTA -- a block's second pair re-reads its adapters,
// mostly from L2, rather than doubling the arithmetic of one CTA (gpt-oss
// w2 decode: 31 us against 40 us).  Fuller blocks: up to kNPG pairs per item,
// split over 4 CTAs (K and N halves of 2 CTAs stream too long a share per
// CTA; 8-CTA exchanges cost more than they balance).  Smaller clusters are
// taken when K or N has too few 8-element chunks.  resident(cfg) gives the
// clusters of that shape that fit at once.
template <typename ResidentFn>
int choose(const FusedArgs &f, const DeviceInfo &dev, bool naive, ResidentFn resident, CsCfg *out, long long *grid) {
  const bool single = naive || (long long)f.M * f.topk <= (long long)f.num_experts * f.num_active_loras;
  const int npg = single ? 1 : kNPG;
  int want = single ? 1 : 4;
  while (want > 1 && (f.K / 8 < want || f.N / 8 < want)) want >>= 1;
  for (int C = want; C >= 1; C >>= 1) {
    CsCfg cfg;
    if (!layout(f, dev, C, npg, &cfg)) continue;
    const int clusters = resident(cfg);
    *out = cfg;
    *grid = std::max(1LL, std::min<long long>(unit_bound(f, naive, npg), clusters));
    return 0;
  }
  return MOE_LORA_ERR_UNSUPPORTED;
}

template <bool NAIVE, int LG_VR, int NPG>
int launch_with(const FusedArgs &f, const CsCfg &cfg, long long G, cudaStream_t stream) {
  CsMaps maps;
  const uint64_t LE = (uint64_t)f.max_loras * f.num_experts;
  for (int s = 0; s < kMaxSlices; ++s) {
    const int src = s < f.num_slices ? s : 0;
    if (int st = stream::encode_3d(&maps.a[s], f.lora_a[src], (uint64_t)f.K, (uint64_t)f.rank, LE, (uint32_t)cfg.kc,
                                   (uint32_t)f.rank, CU_TENSOR_MAP_SWIZZLE_NONE))
      return st;
  }
  const void *fn = (const void *)fused_cluster_stream_kernel<NAIVE, LG_VR, NPG>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes) != cudaSuccess)
    return MOE_LORA_ERR_LAUNCH;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)(G * cfg.C), 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = cfg.smem_bytes;
  lc.stream = stream;
  // Single-CTA clusters (one pair per item, at most one item per CTA on
  // decode batches) are launched as programmatic dependents: a CTA may start
  // while the kernel before it finishes and waits for it with
  // griddepcontrol.wait before reading any input (gpt-oss w2 decode step
  // 39.1 -> 37.4 us).  Larger clusters are launched after it completes: the
  // grid is every cluster that fits on an idle GPU, and clusters launched
  // early beside the align's CTAs could not all be placed -- the rest would
  // run as a second wave, each with a full share of the units.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cfg.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = cfg.C == 1 ? 2 : 1;
  return cudaLaunchKernelEx(&lc, fused_cluster_stream_kernel<NAIVE, LG_VR, NPG>, maps, f, cfg) == cudaSuccess
             ? 0
             : MOE_LORA_ERR_LAUNCH;
}

template <bool NAIVE, int LG_VR>
int launch_cs(const FusedArgs &f, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  CsCfg cfg;
  long long G = 0;
  auto resident = [&](const CsCfg &c) {
    if constexpr (NAIVE) return resident_clusters<NAIVE, LG_VR, 1>(c, dev);
    else return c.npg == 1 ? resident_clusters<NAIVE, LG_VR, 1>(c, dev) : resident_clusters<NAIVE, LG_VR, kNPG>(c, dev);
  };
  if (int st = choose(f, dev, NAIVE, resident, &cfg, &G)) return st;
  if (unit_bound(f, NAIVE, cfg.npg) <= 0) return 0;
  if constexpr (NAIVE) return launch_with<NAIVE, LG_VR, 1>(f, cfg, G, stream);
  else return cfg.npg == 1 ? launch_with<NAIVE, LG_VR, 1>(f, cfg, G, stream) : launch_with<NAIVE, LG_VR, kNPG>(f, cfg, G, stream);
}

template <bool NAIVE>
int launch_by_rank(const FusedArgs &f, cudaStream_t stream) {
  if (!cluster_stream_supports(f)) return MOE_LORA_ERR_UNSUPPORTED;
  switch (f.rank) {
    case 8: return launch_cs<NAIVE, 0>(f, stream);
    case 16: return launch_cs<NAIVE, 1>(f, stream);
    case 32: return launch_cs<NAIVE, 2>(f, stream);
    case 64: return launch_cs<NAIVE, 3>(f, stream);
    case 128: return launch_cs<NAIVE, 4>(f, stream);
    default: return MOE_LORA_ERR_UNSUPPORTED;
  }
}

}  // namespace

bool cluster_stream_supports(const FusedArgs &f) {
  return f.rank >= 8 && f.rank <= 128 && (f.rank & (f.rank - 1)) == 0 && f.num_active_loras <= kMaxSlots &&
         f.block_size <= 128;
}

int launch_fused_cluster_stream(const FusedArgs &f, cudaStream_t stream) { return launch_by_rank<false>(f, stream); }

int launch_fused_cluster_stream_naive(const FusedArgs &f, cudaStream_t stream) {
  return launch_by_rank<true>(f, stream);
}

int plan_fused_cluster_stream(const FusedArgs &f, const DeviceInfo &dev, bool naive, FusedPlan *out) {
  if (!cluster_stream_supports(f)) return MOE_LORA_ERR_UNSUPPORTED;
  CsCfg cfg;
  long long G = 0;
  // host-only plan: clusters of C CTAs, kCtasPerSm CTAs per SM
  if (int st = choose(f, dev, naive, [&](const CsCfg &c) { return std::max(1, kCtasPerSm * dev.sm_count / c.C); },
                      &cfg, &G))
    return st;
  out->kernel = MOE_LORA_PATH_CUDA_CORE_STREAM;
  out->grid = (int)(G * cfg.C);
  out->threads = kThreads;
  out->smem_bytes = cfg.smem_bytes;
  out->s_sh = cfg.stages;
  out->lag = 0;
  out->s_ex = cfg.kc;
  out->t_bufs = cfg.nb;   // (fields reused: A box columns, B rows per stage)
  out->tmem_cols = 0;
  out->cluster = cfg.C;
  out->pairs_per_group = cfg.npg;
  return 0;
}

}  // namespace moe_lora
