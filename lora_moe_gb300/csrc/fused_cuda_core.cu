// fused_cuda_core.cu -- the decode-sized fused MoE-LoRA shrink+expand on CUDA
// cores (sm_103a).
//
// Computes, for every block b of every active slot z (l = lora_ids[z],
// e = expert_ids[l][b]), every adapter slice s and every pair f of that block
// (input row x_f: row f / topk, or row f when x holds one row per pair; router
// weight w_f, 1 without weights):
//     t[j]    = sum_k x_f[k] * A_s[l][e][j][k]                (fp32)
//     y[f][off + s*N + n] = bf16((add_inputs ? y_in : 0) + w_f * sum_j B_s[l][e][n][j] * t[j])
// (prhub.com.cn summary of vLLM PR #42290, "Implementation breakdown" step 1:
// one kernel does the shrink by lora_a and the expand by lora_b and keeps the
// rank dimension on chip; its small-batch kernel is the decode specialisation.)
//
// At decode sizes a block holds one or two real pairs, so the work is a skinny
// GEMV bound by reading A[l,e] (r x K) and B[l,e] (N x r) -- and, at a few
// megabytes per call, by latency.  Design:
//   * grid (C, num_slices * num_active_loras, blocks): CTA (c, s * nact + z, b)
//     serves slice s of block b of slot z (vLLM PR #32005: the LoRA grid
//     dimension is the number of active LoRAs), capped at the clusters that
//     can be resident at once (CTAs then walk further blocks); blocks past
//     num_tokens_post_padded exit after one dependent load.  With naive block
//     assignment the grid is (C, num_slices, pairs) and each work item is one
//     pair, its LoRA and expert read from token_lora_mapping and topk_ids.
//   * a thread-block cluster of C CTAs shares a block: CTA c streams the
//     K-slice c of A and of the gathered x rows and the N-slice c of B and y;
//     the C partial t's are summed through distributed shared memory in rank
//     order (deterministic).
//   * operands are requested before the first wait: the A slice (16-byte
//     cp.async) and the contiguous B slice (one bulk copy) as soon as the
//     expert id is known, the x and y_in rows once the block's pairs are
//     compacted.  Dot products read 16-byte shared-memory vectors and reduce
//     with warp shuffles; y is written with coalesced stores.
//   * pairs are processed in groups whose size is a template constant (2 for
//     blocks with at most two real pairs, else 8), so no shuffle sits in
//     divergent code.
#include <cooperative_groups.h>
#include <algorithm>
#include <mutex>
#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace moe_lora {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPG = 8;        // most pairs processed together
constexpr int kMaxBlock = 128;   // largest block_size
constexpr int kMaxCluster = 16;

struct CcCfg {
  int C;               // CTAs per block (cluster size)
  int pg;              // pairs processed together (the kernel's NPG)
  int kslice, nslice;  // per-CTA K / N slice capacity (multiples of 8)
  int a_pitch;         // bytes per staged A row (kslice + 8 bf16: rows skewed by 16 B)
  int off_a, off_x, off_b, off_y, off_tp, off_t;
  int smem_bytes;
  int lpr_log2;        // expand: lanes per B row, log2
  unsigned long long wait_limit_ns;   // limit of the wait for the B slice (kWaitTimeoutNs)
  int withhold_b;      // test of the bounded wait: the B slice's copy is never issued
  // cluster rank c's slices: K columns [k_lo, k_lo + kn), N rows [n_lo, n_lo + nn)
  int k_lo[kMaxCluster], kn[kMaxCluster], n_lo[kMaxCluster], nn[kMaxCluster];
};

struct Meta {
  uint64_t bar;                  // the B slice's bulk copy
  int pf[kMaxBlock];             // the block's real pairs (flat index), in order
  int pm[kMaxBlock];             // their row of x
  float pw[kMaxBlock];           // their router weight
  uint16_t *yp[kMaxPG];          // the group's output rows, at this CTA's first column
  int wcount[kWarps];
  int nv;
  int abort;
};

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void unpack4(const uint2 v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
}

__device__ __forceinline__ float dot8(const float (&a)[8], const uint4 xv) {
  float x[8];
  unpack8(xv, x);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = fmaf(a[i], x[i], s);
  return s;
}

// Request this CTA's slices of A[l][e] (rows j, columns [k_lo, k_lo + 8 kch),
// by cp.async) and of B[l][e] (rows [n_lo, n_lo + nn), one bulk copy) as soon
// as the expert is known; x and y_in rows follow once the pairs are.
// After a wait has given up (*abort) nothing more is requested: the CTA's
// barrier may still be in a phase that never completed, and no copy may be
// left in flight when it exits.
__device__ __forceinline__ void request_adapters(const FusedArgs &p, const CcCfg &cfg, Meta &meta, uint8_t *a_s,
                                                 uint8_t *b_s, int l, int e, int sl, int k_lo, int kch, int n_lo,
                                                 int nn) {
  if (__syncthreads_or(meta.abort)) return;
  const int r = p.rank, K = p.K, N = p.N;
  const size_t le = (size_t)l * p.num_experts + e;
  const uint16_t *A = slice_a(p, sl) + le * r * K;
  const uint16_t *Bm = slice_b(p, sl) + le * N * r;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&meta.bar, (uint32_t)nn * r * 2);
    if (!cfg.withhold_b) bulk_g2s(b_s, Bm + (size_t)n_lo * r, (uint32_t)nn * r * 2, &meta.bar);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < r; j += kWarps)
    for (int ch = lane; ch < kch; ch += 32)
      cp_async_16(a_s + (size_t)j * cfg.a_pitch + ch * 16, A + (size_t)j * K + k_lo + ch * 8, 16u);
}

// Naive block assignment: whether pair f is covered, and its LoRA and
// expert.  Uniform over the CTA (every thread returns the same), and over the
// cluster (every CTA reads the same values).
__device__ __forceinline__ bool naive_pair(const FusedArgs &p, int f, int &l, int &e) {
  const int m = f / p.topk;
  l = __ldg(p.token_lora_mapping + m);
  e = __ldg(p.topk_ids + f);
  const bool slot_ok = l >= 0 && l < p.max_loras && (!p.adapter_enabled || __ldg(p.adapter_enabled + l) != 0);
  int listed = 0;
  if (slot_ok)
    for (int i = threadIdx.x; i < p.num_active_loras; i += blockDim.x) listed |= __ldg(p.lora_ids + i) == l;
  listed = __syncthreads_or(listed);
  if (!listed) return false;
  if (e < 0 || e >= p.num_experts) {
    if (threadIdx.x == 0 && cg::this_cluster().block_rank() == 0 && blockIdx.y == 0)
      flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
    return false;
  }
  return true;
}

// Sum each of the NPG values v[0..NPG) over the 32 lanes of the warp.  The
// first log2(NPG) butterfly steps also halve the values each lane carries
// (a reduce-scatter), the rest are a plain butterfly; every sum is formed in
// the same order as a plain 5-step butterfly of that value would form it.  On
// return lane L holds the total of value q = L >> (5 - log2 NPG) in v[0].
template <int NPG>
__device__ __forceinline__ void warp_sum_scatter(float (&v)[NPG], int lane) {
  int d = 16;
#pragma unroll
  for (int n = NPG; n > 1; n >>= 1, d >>= 1) {
    const bool upper = (lane & d) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = upper ? v[i + n / 2] : v[i];
      const float send = upper ? v[i] : v[i + n / 2];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
    }
  }
#pragma unroll
  for (; d > 0; d >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], d);
}

template <int NPG>
constexpr int log2_pg() {
  return NPG >= 8 ? 3 : (NPG >= 4 ? 2 : (NPG >= 2 ? 1 : 0));
}

// Everything one CTA of the cluster needs to apply a group of pairs.
struct GroupCtx {
  const FusedArgs &p;
  const CcCfg &cfg;
  Meta &meta;
  uint8_t *a_s, *x_s, *b_s, *y_s;
  float *tpart, *t;
  int C, c, tid, lane, warp, sl, k_lo, kch, n_lo, nn, nch;
  uint32_t phase;
  volatile int *abort;
};

// One group of nvg <= NPG pairs (meta.pf[g0 .. g0 + nvg)): gather their x
// and y_in rows, shrink over this CTA's K-slice, sum the cluster's partial
// t's, expand over this CTA's N-slice and store.  The loops over the NPG
// slots run every slot whether or not it holds a pair (stale operands in
// unused slots give values that are never stored), so no shuffle sits in
// divergent code.  Ends with a cluster barrier (peers are done reading this
// CTA's partial t and every thread with the group's shared memory).
template <int RV, int NPG>
__device__ __forceinline__ void run_group(const GroupCtx &g, int g0, int nvg) {
  const FusedArgs &p = g.p;
  const CcCfg &cfg = g.cfg;
  Meta &meta = g.meta;
  uint8_t *x_s = g.x_s, *y_s = g.y_s;
  const uint8_t *a_s = g.a_s, *b_s = g.b_s;
  float *tpart = g.tpart, *t = g.t;
  const int C = g.C, tid = g.tid, lane = g.lane, warp = g.warp, sl = g.sl;
  const int k_lo = g.k_lo, kch = g.kch, n_lo = g.n_lo, nn = g.nn, nch = g.nch;
  const int r = p.rank, K = p.K;
  cg::cluster_group cluster = cg::this_cluster();
  volatile int *abort = g.abort;
  const uint32_t phase = g.phase;
  if (tid < nvg) meta.yp[tid] = p.y + y_base(p, meta.pf[g0 + tid], sl) + n_lo;
  for (int q = warp; q < nvg; q += kWarps) {
    const uint16_t *xr = p.x + (size_t)meta.pm[g0 + q] * K + k_lo;
    for (int ch = lane; ch < kch; ch += 32) cp_async_16(x_s + (size_t)q * cfg.kslice * 2 + ch * 16, xr + ch * 8, 16u);
  }
  if (p.add_inputs)
    for (int q = warp; q < nvg; q += kWarps) {
      const uint16_t *yr = p.y + y_base(p, meta.pf[g0 + q], sl) + n_lo;
      for (int ch = lane; ch < nch; ch += 32) cp_async_16(y_s + (size_t)q * cfg.nslice * 2 + ch * 16, yr + ch * 8, 16u);
    }
  cp_async_commit();
  cp_async_wait_group<0>();
  __syncthreads();

  // ---- shrink: partial t over this CTA's K-slice; warp w owns rows j = w (mod 8)
  {
    float *dst = C == 1 ? t : tpart;
    constexpr int kLg = log2_pg<NPG>();
    const int q_mine = lane >> (5 - kLg);
    const bool writer = (lane & ((1 << (5 - kLg)) - 1)) == 0 && q_mine < nvg;
    for (int j = warp; j < r; j += kWarps) {
      float acc[NPG];
#pragma unroll
      for (int q = 0; q < NPG; ++q) acc[q] = 0.f;
      const uint4 *arow = reinterpret_cast<const uint4 *>(a_s + (size_t)j * cfg.a_pitch);
      for (int ch = lane; ch < kch; ch += 32) {
        float af[8];
        unpack8(arow[ch], af);
#pragma unroll
        for (int q = 0; q < NPG; ++q)
          acc[q] += dot8(af, reinterpret_cast<const uint4 *>(x_s + (size_t)q * cfg.kslice * 2)[ch]);
      }
      warp_sum_scatter<NPG>(acc, lane);
      if (writer) dst[q_mine * r + j] = acc[0];
    }
  }

  // ---- t = sum of the C partials through distributed shared memory, in
  // rank order (deterministic); the C remote loads of an element are
  // issued together.
  if (C > 1) {
    cluster_arrive_release();
    cluster_wait();
    for (int i = tid; i < nvg * r; i += kThreads) {
      float v[kMaxCluster];
#pragma unroll
      for (int q = 0; q < kMaxCluster; ++q) v[q] = q < C ? cluster.map_shared_rank(tpart, q)[i] : 0.f;
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < kMaxCluster; ++q)
        if (q < C) sum += v[q];
      t[i] = sum;
    }
    // this CTA reads no peer's partial t after this; the matching wait is
    // at the end of the group
    cluster_arrive_relaxed();
  }
  __syncthreads();
  if (g0 == 0) mbar_wait_for(&meta.bar, phase, abort, p.err, cfg.wait_limit_ns);

  // ---- expand: y rows of this CTA's N-slice.  A B row is read by lpr
  // lanes (one shared-memory vector each); their partial sums meet by
  // shuffles (lpr comes from a kernel parameter: uniform control flow).
  {
    const int vecs = r / RV;
    const int lg = cfg.lpr_log2, lpr = 1 << lg;
    const int rows_per_warp = 32 >> lg;
    const int ch0 = lane & (lpr - 1);
    for (int row0 = warp * rows_per_warp; row0 < nn; row0 += kWarps * rows_per_warp) {
      const int nl = row0 + (lane >> lg);
      float acc[NPG];
#pragma unroll
      for (int q = 0; q < NPG; ++q) acc[q] = 0.f;
      if (nl < nn) {
        for (int ch = ch0; ch < vecs; ch += lpr) {
          const int j0 = ch * RV;
          if constexpr (RV == 8) {
            float bf[8];
            unpack8(*reinterpret_cast<const uint4 *>(b_s + ((size_t)nl * r + j0) * 2), bf);
#pragma unroll
            for (int q = 0; q < NPG; ++q) {
              const float4 t0 = *reinterpret_cast<const float4 *>(t + q * r + j0);
              const float4 t1 = *reinterpret_cast<const float4 *>(t + q * r + j0 + 4);
              acc[q] += bf[0] * t0.x + bf[1] * t0.y + bf[2] * t0.z + bf[3] * t0.w +
                        bf[4] * t1.x + bf[5] * t1.y + bf[6] * t1.z + bf[7] * t1.w;
            }
          } else {
            float bf[4];
            unpack4(*reinterpret_cast<const uint2 *>(b_s + ((size_t)nl * r + j0) * 2), bf);
#pragma unroll
            for (int q = 0; q < NPG; ++q) {
              const float4 t0 = *reinterpret_cast<const float4 *>(t + q * r + j0);
              acc[q] += bf[0] * t0.x + bf[1] * t0.y + bf[2] * t0.z + bf[3] * t0.w;
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < NPG; ++q) {
        float v = acc[q];
#pragma unroll
        for (int d = 8; d > 0; d >>= 1)
          if (d < lpr) v += __shfl_xor_sync(0xffffffffu, v, d);
        if (ch0 == 0 && nl < nn && q < nvg) {
          const float old = p.add_inputs
                                ? bf16_bits_to_float(reinterpret_cast<const uint16_t *>(
                                      y_s + (size_t)q * cfg.nslice * 2)[nl])
                                : 0.f;
          meta.yp[q][nl] = float_to_bf16_bits(v * meta.pw[g0 + q] + old);
        }
      }
    }
  }
  // Peers are done reading this CTA's partial t (they arrived after their
  // reads) and every thread with this group's shared memory before the next
  // group or block reuses it, or before the CTA exits.
  if (C > 1) cluster_wait();
  __syncthreads();
}

// RV: elements of B per shared-memory vector (8 when rank % 8 == 0, else 4).
// NAIVE: one pair per work item, found from topk_ids and token_lora_mapping
// (naive block assignment, no align); otherwise blocks of the align output.
// NPG: pairs per group the shared-memory layout holds (8, 2 or 1).  A block
// with at most two real pairs runs the two-pair group body, a larger one
// groups of eight (when NPG is 8).
template <int RV, bool NAIVE, int NPG>
__global__ void __launch_bounds__(kThreads, 4) fused_cuda_core_kernel(const FusedArgs p, const CcCfg cfg) {
  extern __shared__ __align__(128) uint8_t smem[];
  Meta &meta = *reinterpret_cast<Meta *>(smem);
  uint8_t *a_s = smem + cfg.off_a;
  uint8_t *x_s = smem + cfg.off_x;
  uint8_t *b_s = smem + cfg.off_b;
  uint8_t *y_s = smem + cfg.off_y;
  float *tpart = reinterpret_cast<float *>(smem + cfg.off_tp);   // [NPG][r] this CTA's partial t
  float *t = reinterpret_cast<float *>(smem + cfg.off_t);         // [NPG][r] the group's t

  cg::cluster_group cluster = cg::this_cluster();
  const int C = cfg.C;
  const int c = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.num_experts, bs = p.block_size;
  const int P = p.M * p.topk;
  // grid.y: slice * num_active_loras + slot (sorted), or the slice (naive)
  const int z = NAIVE ? 0 : (int)(blockIdx.y % p.num_active_loras);
  const int sl = NAIVE ? (int)blockIdx.y : (int)(blockIdx.y / p.num_active_loras);
  // This CTA's K- and N-slices.
  const int k_lo = cfg.k_lo[c], kn = cfg.kn[c], n_lo = cfg.n_lo[c], nn = cfg.nn[c];
  const int kch = kn / 8, nch = nn / 8;

  // The slot's LoRA index and enable flag are inputs the align does not
  // write: they are read before waiting for it.  Everything else is read
  // after griddepcontrol.wait.
  int l = 0, en = 1;
  if (!NAIVE) {
    l = __ldg(p.lora_ids + z);
    if (l >= 0 && l < p.max_loras && p.adapter_enabled) en = __ldg(p.adapter_enabled + l);
  }
  wait_for_prior_grid();   // the align outputs are read from here on
  int nitems = P, e_first = 0, f_first = -1;
  if (!NAIVE) {
    // Uniform over the cluster: every CTA of it reads the same values.
    if (l < 0 || l >= p.max_loras) {
      if (c == 0 && tid == 0 && blockIdx.z == 0 && sl == 0) flag_error(p.err, MOE_LORA_DEVERR_LORA_ID);
      return;
    }
    if (en == 0) return;
    // The first block's expert and pair ids are requested together with the
    // slot's block count (one round trip); they are only used if the block exists.
    const int b_first = blockIdx.z;
    e_first = __ldg(p.expert_ids + (size_t)l * p.max_num_m_blocks + b_first);
    if (tid < bs && b_first * bs + tid < p.max_num_tokens_padded)
      f_first = __ldg(p.sorted_token_ids + (size_t)l * p.max_num_tokens_padded + b_first * bs + tid);
    nitems = min(__ldg(p.num_tokens_post_padded + l) / bs, p.max_num_m_blocks);
    // the first block's ids were requested with the count: keep them there
    // (not sunk below the exit test), so that one round trip brings all three
    asm volatile("" ::"r"(e_first), "r"(f_first));
    if (b_first >= nitems) return;
  } else if (c == 0 && tid == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
    for (int i = 0; i < p.num_active_loras; ++i) {
      const int li = __ldg(p.lora_ids + i);
      if (li < 0 || li >= p.max_loras) flag_error(p.err, MOE_LORA_DEVERR_LORA_ID);
    }
  }

  if (tid == 0) {
    mbar_init(&meta.bar, 1);
    meta.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int *abort = &meta.abort;
  uint32_t phase = 0;

  for (int b = blockIdx.z; b < nitems; b += gridDim.z) {
    int e;
    if (NAIVE) {
      // work item b is pair b
      if (!naive_pair(p, b, l, e)) continue;
      request_adapters(p, cfg, meta, a_s, b_s, l, e, sl, k_lo, kch, n_lo, nn);
      if (tid == 0) {
        meta.pf[0] = b;
        meta.pm[0] = x_row(p, b);
        meta.pw[0] = route_weight(p, b);
        meta.nv = 1;
      }
      __syncthreads();
    } else {
      e = b == (int)blockIdx.z ? e_first : __ldg(p.expert_ids + (size_t)l * p.max_num_m_blocks + b);
      const bool e_ok = e >= 0 && e < E;   // uniform over the cluster
      if (e_ok) request_adapters(p, cfg, meta, a_s, b_s, l, e, sl, k_lo, kch, n_lo, nn);
      // Compact the block's real pairs, keeping their order.
      const int idx = b * bs + tid;
      int f = -1;
      if (tid < bs && idx < p.max_num_tokens_padded) {
        f = b == (int)blockIdx.z ? f_first : __ldg(p.sorted_token_ids + (size_t)l * p.max_num_tokens_padded + idx);
        if (f < 0 || f > P) {
          if (c == 0 && sl == 0) flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);
          f = -1;
        } else if (f == P) {
          f = -1;
        }
      }
      const unsigned bal = __ballot_sync(0xffffffffu, f >= 0);
      if (lane == 0) meta.wcount[warp] = __popc(bal);
      __syncthreads();
      int base = 0, tot = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        base += (w < warp) ? meta.wcount[w] : 0;
        tot += meta.wcount[w];
      }
      if (f >= 0) {
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        meta.pf[pos] = f;
        meta.pm[pos] = x_row(p, f);
        meta.pw[pos] = route_weight(p, f);
      }
      if (tid == 0) meta.nv = tot;
      __syncthreads();
      if (!e_ok) {
        if (tid == 0 && c == 0 && sl == 0) flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
        continue;
      }
    }
    const int nv = meta.nv;
    if (nv == 0) {
      // nothing to apply; the requested slices must land before their buffers
      // are reused or the CTA exits
      cp_async_wait_group<0>();
      mbar_wait_for(&meta.bar, phase, abort, p.err, cfg.wait_limit_ns);
      phase ^= 1;
      __syncthreads();
      continue;
    }

    const GroupCtx gctx{p, cfg, meta, a_s, x_s, b_s, y_s, tpart, t, C, c, tid, lane, warp, sl,
                        k_lo, kch, n_lo, nn, nch, phase, abort};
    if (NPG >= 8 && nv > 2) {
      for (int g0 = 0; g0 < nv; g0 += 8) run_group<RV, (NPG >= 8 ? 8 : 1)>(gctx, g0, min(8, nv - g0));
    } else if (NPG >= 2) {
      for (int g0 = 0; g0 < nv; g0 += 2) run_group<RV, (NPG >= 2 ? 2 : 1)>(gctx, g0, min(2, nv - g0));
    } else {
      for (int g0 = 0; g0 < nv; ++g0) run_group<RV, 1>(gctx, g0, 1);
    }
    phase ^= 1;
  }
}

// Shared-memory layout for cluster size C and pg pairs per group, with the
// per-rank slice tables; returns false if it does not fit.
bool layout(const FusedArgs &f, const DeviceInfo &dev, int C, int pg, CcCfg *cfg) {
  const int r = f.rank;
  cfg->C = C;
  cfg->pg = pg;
  const int k8 = f.K / 8, n8 = f.N / 8;
  cfg->kslice = (k8 + C - 1) / C * 8;
  cfg->nslice = (n8 + C - 1) / C * 8;
  cfg->a_pitch = (cfg->kslice + 8) * 2;
  for (int c = 0; c < kMaxCluster; ++c) {
    const int cc = c < C ? c : C - 1;
    cfg->k_lo[c] = (cc * k8 / C) * 8;
    cfg->kn[c] = ((cc + 1) * k8 / C) * 8 - cfg->k_lo[c];
    cfg->n_lo[c] = (cc * n8 / C) * 8;
    cfg->nn[c] = ((cc + 1) * n8 / C) * 8 - cfg->n_lo[c];
  }
  const int vecs = r / (r % 8 == 0 ? 8 : 4);
  int lg = 0;
  while ((1 << lg) < vecs && lg < 4) ++lg;
  cfg->lpr_log2 = lg;
  cfg->wait_limit_ns = kWaitTimeoutNs;
  cfg->withhold_b = 0;
  size_t off = (sizeof(Meta) + 127) / 128 * 128;
  cfg->off_a = (int)off;
  off += (size_t)r * cfg->a_pitch;
  cfg->off_x = (int)off;
  off += (size_t)pg * cfg->kslice * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_b = (int)off;
  off += (size_t)cfg->nslice * r * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_y = (int)off;
  off += (size_t)pg * cfg->nslice * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_tp = (int)off;
  off += (size_t)pg * r * 4;
  cfg->off_t = (int)off;
  off += (size_t)pg * r * 4;
  cfg->smem_bytes = (int)off;
  return (size_t)cfg->smem_bytes <= dev.max_smem_optin;
}

// Spread a block's adapter bytes over up to 16 CTAs: at least ~12 KB each
// (so that each CTA is worth its launch, up to 8 CTAs) and at most ~48 KB each
// (so that several CTAs share an SM); more CTAs if shared memory demands it.
// Blocks of the align output (one cluster per block, grid capped at the
// resident clusters) whose adapters want more than 8 CTAs take clusters of
// 12 (non-portable): measured on the Qwen3-shaped w13 decode 7.5 against
// 8.2 us with 8 (10: 8.5, 16: 11.4), on the gpt-oss-shaped w2 decode 103
// against 123 us.  The naive assignment (a cluster per pair, several waves)
// keeps 8 (12: 8.5 against 7.6 us on Qwen3).
// pg: the preferred pairs per group; smaller groups are tried if it does not fit.
int pick_cfg(const FusedArgs &f, const DeviceInfo &dev, int pg, bool per_block, CcCfg *cfg) {
  const long long item_bytes = (long long)(f.K + f.N) * f.rank * 2;
  const long long lo = (item_bytes + 48 * 1024 - 1) / (48 * 1024);
  long long hi = (item_bytes + 12 * 1024 - 1) / (12 * 1024);
  if (hi > 8) hi = per_block && f.K / 8 >= 12 && f.N / 8 >= 12 ? 12 : 8;
  long long want = lo > hi ? lo : hi;
  const long long cmax = std::min<long long>(kMaxCluster, std::min(f.K / 8, f.N / 8));
  if (want > cmax) want = cmax;
  if (want < 1) want = 1;
  for (int g = pg; g >= 1; g = g == 8 ? 2 : g - 1)
    for (long long C = want; C <= cmax; ++C)
      if (layout(f, dev, (int)C, g, cfg)) return 0;
  return MOE_LORA_ERR_UNSUPPORTED;
}

template <int RV, bool NAIVE, int NPG>
int launch_one(const FusedArgs &f, const CcCfg &cfg, unsigned gy, unsigned gz, cudaStream_t stream) {
  const void *fn = (const void *)fused_cuda_core_kernel<RV, NAIVE, NPG>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes) != cudaSuccess)
    return MOE_LORA_ERR_LAUNCH;
  if (cfg.C > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return MOE_LORA_ERR_LAUNCH;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(cfg.C, gy, gz);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = cfg.smem_bytes;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cfg.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // May start while the kernel before it (the align) is finishing: it waits
  // for that kernel with griddepcontrol.wait before reading any input.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, fused_cuda_core_kernel<RV, NAIVE, NPG>, f, cfg) == cudaSuccess
             ? 0
             : MOE_LORA_ERR_LAUNCH;
}

template <bool NAIVE, int NPG>
int launch_rv(const FusedArgs &f, const CcCfg &cfg, unsigned gy, unsigned gz, cudaStream_t stream) {
  return f.rank % 8 == 0 ? launch_one<8, NAIVE, NPG>(f, cfg, gy, gz, stream)
                         : launch_one<4, NAIVE, NPG>(f, cfg, gy, gz, stream);
}

// Clusters of this configuration that can be resident at once (cached per
// device, kernel, cluster size and shared-memory size).  Grids no larger than
// this start every CTA at once: CTAs that find no work then never hold a slot
// that a working CTA waits for.
template <int RV, bool NAIVE, int NPG>
int resident_clusters_of(const CcCfg &cfg, const DeviceInfo &dev) {
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
  const void *fn = (const void *)fused_cuda_core_kernel<RV, NAIVE, NPG>;
  int clusters = 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes) == cudaSuccess &&
      (cfg.C <= 8 || cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess)) {
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
  if (clusters <= 0) clusters = dev.sm_count / cfg.C;   // fallback: one CTA per SM
  if (n < 32) cache[n++] = {dev.device, cfg.C, cfg.smem_bytes, clusters};
  return clusters;
}

template <bool NAIVE, int NPG>
int resident_clusters(const FusedArgs &f, const CcCfg &cfg, const DeviceInfo &dev) {
  return f.rank % 8 == 0 ? resident_clusters_of<8, NAIVE, NPG>(cfg, dev)
                         : resident_clusters_of<4, NAIVE, NPG>(cfg, dev);
}

}  // namespace

int launch_fused_cuda_core(const FusedArgs &f, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  if (f.block_size > kMaxBlock) return MOE_LORA_ERR_UNSUPPORTED;
  if ((long long)f.num_active_loras * f.num_slices > 65535) return MOE_LORA_ERR_UNSUPPORTED;
  // Blocks one slot can produce: floor(M*topk / bs) full ones plus one partly
  // filled block per non-empty expert segment.
  const long long pairs = (long long)f.M * f.topk;
  // Room for groups of eight pairs where it fits (blocks with more than two
  // real pairs run eight at a time; the others the two-pair body).
  CcCfg cfg;
  if (int st = pick_cfg(f, dev, 8, true, &cfg)) return st;
  long long per_slot = pairs / f.block_size + (pairs < f.num_experts ? pairs : f.num_experts);
  if (per_slot > f.max_num_m_blocks) per_slot = f.max_num_m_blocks;
  // Blocks a slot really has are usually far fewer than that bound: the grid
  // is capped at what is resident at once (at least one cluster per slot),
  // and CTAs walk further blocks of their slot in turn.
  const long long units = (long long)f.num_active_loras * f.num_slices;
  const int resident = cfg.pg == 8 ? resident_clusters<false, 8>(f, cfg, dev)
                                   : (cfg.pg == 2 ? resident_clusters<false, 2>(f, cfg, dev)
                                                  : resident_clusters<false, 1>(f, cfg, dev));
  const long long cap = std::max<long long>(1, resident / units);
  if (per_slot > cap) per_slot = cap;
  if (per_slot > 65535) per_slot = 65535;
  if (per_slot <= 0) return 0;
  const unsigned gy = (unsigned)units;
  switch (cfg.pg) {
    case 8: return launch_rv<false, 8>(f, cfg, gy, (unsigned)per_slot, stream);
    case 2: return launch_rv<false, 2>(f, cfg, gy, (unsigned)per_slot, stream);
    default: return launch_rv<false, 1>(f, cfg, gy, (unsigned)per_slot, stream);
  }
}

int plan_fused_cuda_core(const FusedArgs &f, const DeviceInfo &dev, FusedPlan *out) {
  if (f.block_size > kMaxBlock) return MOE_LORA_ERR_UNSUPPORTED;
  CcCfg cfg;
  if (int st = pick_cfg(f, dev, 8, true, &cfg)) return st;
  out->kernel = MOE_LORA_PATH_CUDA_CORE_CLUSTER;
  out->grid = 0;   // capped at run time by the clusters that can be resident at once
  out->threads = kThreads;
  out->smem_bytes = cfg.smem_bytes;
  out->s_sh = out->lag = out->s_ex = out->t_bufs = out->tmem_cols = 0;
  out->cluster = cfg.C;
  out->pairs_per_group = cfg.pg;
  return 0;
}

int launch_fused_naive(const FusedArgs &f, cudaStream_t stream, unsigned long long wait_limit_ns, int withhold_b) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  CcCfg cfg;
  if (int st = pick_cfg(f, dev, 1, false, &cfg)) return st;
  if (wait_limit_ns) cfg.wait_limit_ns = wait_limit_ns;
  cfg.withhold_b = withhold_b;
  // grid (C, slices, pairs), as the one-program-per-pair grid of the naive
  // assignment; past a few waves, CTAs walk several pairs.
  // Every pair gets its own cluster (uncovered ones exit at once and free
  // their slot); very large batches walk pairs in turn.
  long long items = (long long)f.M * f.topk;
  const long long cap = std::max<long long>(64, 16LL * dev.sm_count / ((long long)cfg.C * f.num_slices));
  if (items > cap) items = cap;
  if (items > 65535) items = 65535;
  if (items <= 0) return 0;
  return launch_rv<true, 1>(f, cfg, (unsigned)f.num_slices, (unsigned)items, stream);
}

}  // namespace moe_lora
