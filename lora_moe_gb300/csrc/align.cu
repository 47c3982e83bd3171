// align.cu -- moe_lora_align kernels for sm_103a.
//
// For each active LoRA slot the pairs f = m*topk + k of its tokens are counted
// per expert, each count is padded to a multiple of block_size, the padded
// counts are prefix-summed into segment offsets, and every pair is written to
// its expert's segment in ascending f, padding slots holding the sentinel
// M*topk (vLLM PR #29257 "Lora MoE Align Improvements", section Purpose: a
// shared-memory variant, and a global-memory variant for large num_experts).
//
// Determinism without sorting: the pairs are split into contiguous per-warp
// ranges.  A warp walks its range 32 pairs at a time; __match_any_sync groups
// the lanes that hold the same expert, so a lane's rank among equal experts is
// the popcount of the lower lanes in its group, and the group's size is added
// to that warp's private counter for the expert.  A column scan over the warp
// ranges (in range order) turns the counters into each warp's starting
// position inside every segment, so the second walk scatters every pair to a
// position that only depends on f -- the same result as a stable sort.
//
//   shared-memory variant : one CTA (32 warps) per active slot; the per-warp
//                           counters live in shared memory.
//   global-memory variant : many CTAs per slot; per-warp counters go to the
//                           caller's workspace and three launches (count, scan,
//                           scatter) replace the CTA-wide barriers.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_utils.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace moe_lora {

namespace {

constexpr int kSmemWarps = 32;                  // shared-memory variant: warps per CTA
constexpr int kSmemThreads = kSmemWarps * 32;
constexpr int kGlobalWarpsPerCta = 8;           // global variant, count / scatter kernels
constexpr int kGlobalThreads = kGlobalWarpsPerCta * 32;
constexpr int kScanThreads = 1024;              // one thread per expert (E <= 1024)
constexpr int kMaxGlobalWarpRanges = 128;       // global variant: target warp ranges per slot

// Expert of pair f for slot l, or -1 when the pair is not this slot's or its
// expert is out of range (flagged once, in the counting pass).  Without a
// token_lora_mapping every token belongs to the one slot (plain MoE align).
__device__ __forceinline__ int pair_expert(const AlignArgs &a, int f, int l, bool flag) {
  const int m = f / a.topk;
  if (a.token_lora_mapping && __ldg(a.token_lora_mapping + m) != l) return -1;
  const int e = __ldg(a.topk_ids + f);
  if (e < 0 || e >= a.num_experts) {
    if (flag) flag_error(a.err, MOE_LORA_DEVERR_EXPERT_ID);
    return -1;
  }
  return e;
}

// Slot z's LoRA index, or -1 when the slot is skipped (bad id: flagged;
// disabled adapter: its num_tokens_post_padded is set to 0 by `writer`).
// Without lora_ids, slot z is row z (plain MoE align: one slot, row 0).
__device__ __forceinline__ int slot_lora(const AlignArgs &a, int z, bool writer) {
  const int l = a.lora_ids ? __ldg(a.lora_ids + z) : z;
  if (l < 0 || l >= a.max_loras) {
    if (writer) flag_error(a.err, MOE_LORA_DEVERR_LORA_ID);
    return -1;
  }
  if (a.adapter_enabled && __ldg(a.adapter_enabled + l) == 0) {
    if (writer) a.num_tokens_post_padded[l] = 0;
    return -1;
  }
  return l;
}

// Walk [lo, hi) one warp-width at a time, adding group sizes to tab[e].
__device__ __forceinline__ void warp_count(const AlignArgs &a, int l, int lo, int hi, int *tab,
                                           int lane) {
  for (int base = lo; base < hi; base += 32) {
    const int f = base + lane;
    const int e = (f < hi) ? pair_expert(a, f, l, true) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) tab[e] += __popc(peers);
  }
}

// Second walk: tab[e] + seg[e] (seg may be null) is this warp's next position
// in segment e.
__device__ __forceinline__ void warp_scatter(const AlignArgs &a, int l, int lo, int hi, int *tab,
                                             const int *seg, int32_t *sorted, int lane) {
  const unsigned lower = (1u << lane) - 1u;
  for (int base = lo; base < hi; base += 32) {
    const int f = base + lane;
    const int e = (f < hi) ? pair_expert(a, f, l, false) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int pos = (e >= 0) ? tab[e] + (seg ? seg[e] : 0) + __popc(peers & lower) : 0;
    __syncwarp();
    if (e >= 0) {
      sorted[pos] = f;
      if (lane == __ffs(peers) - 1) tab[e] += __popc(peers);
    }
    __syncwarp();
  }
}

// Exclusive scan of one int per thread across the CTA (blockDim.x a multiple
// of 32, at most 1024); returns the thread's exclusive prefix and writes the
// total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, s, d);
      if (lane >= d) s += t;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[nwarps - 1];
  return excl;
}

// n ints from p (16-byte aligned) set to zero by the whole CTA.
__device__ __forceinline__ void zero_ints(int *p, int n) {
  const int n4 = n / 4;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) reinterpret_cast<int4 *>(p)[i] = make_int4(0, 0, 0, 0);
  for (int i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) p[i] = 0;
}

// Column scan of a W x E table of per-warp counts (row w = warp w): every
// entry becomes the count of the rows above it in its column, and cnt[e]
// the column total.  One thread per column (consecutive columns: no bank
// conflicts), its rows read eight at a time so that the loads of a batch are
// in flight together.  Called by every thread of the CTA, with a barrier
// before (the table complete) and after (the scan visible).
__device__ __forceinline__ void column_scan(int *tab, int W, int E, int *cnt) {
  const int e = threadIdx.x;
  if (e >= E) return;
  int run = 0, w = 0;
  for (; w + 8 <= W; w += 8) {
    int v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = tab[(w + i) * E + e];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      tab[(w + i) * E + e] = run;
      run += v[i];
    }
  }
  for (; w < W; ++w) {
    const int v = tab[w * E + e];
    tab[w * E + e] = run;
    run += v;
  }
  cnt[e] = run;
}

// Padding sentinels and block labels of the segment of expert e (n real
// pairs from offset o, padded to a block multiple), by one thread.
__device__ __forceinline__ void write_padding(const AlignArgs &a, int l, int e, int n, int o) {
  const int bs = a.block_size;
  const int padded = (n + bs - 1) / bs * bs;
  int32_t *sorted = a.sorted_token_ids + (size_t)l * a.max_num_tokens_padded;
  int32_t *experts = a.expert_ids + (size_t)l * a.max_num_m_blocks;
  const int sentinel = a.M * a.topk;
  for (int i = o + n; i < o + padded; ++i) sorted[i] = sentinel;
  for (int b = o / bs; b < (o + padded) / bs; ++b) experts[b] = e;
}

// The same for experts e = e0, e0 + step, ... (counts n[e], offsets off[e]),
// a warp per expert, its lanes one slot or block each: for CTAs with many
// warps and few experts each.
__device__ __forceinline__ void write_padding_warps(const AlignArgs &a, int l, const int *n, const int *off, int e0,
                                                    int step) {
  const int E = a.num_experts, bs = a.block_size;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int32_t *sorted = a.sorted_token_ids + (size_t)l * a.max_num_tokens_padded;
  int32_t *experts = a.expert_ids + (size_t)l * a.max_num_m_blocks;
  const int sentinel = a.M * a.topk;
  for (int e = e0 + warp * step; e < E; e += nwarps * step) {
    const int c = n[e], o = off[e];
    const int padded = (c + bs - 1) / bs * bs;
    for (int i = c + lane; i < padded; i += 32) sorted[o + i] = sentinel;
    for (int b = lane; b < padded / bs; b += 32) experts[o / bs + b] = e;
  }
}

// Given per-expert counts cnt[e] (e < E, one per thread), compute segment
// offsets off[0..E], write num_tokens_post_padded[l], the padding sentinels and
// expert_ids.  Returns false (uniformly) when the result exceeds the caller's
// capacity.  Called by every thread of a CTA of at least E threads.
__device__ bool write_segments(const AlignArgs &a, int l, const int *cnt, int *off, int *warp_sums) {
  const int E = a.num_experts, bs = a.block_size, tid = threadIdx.x;
  const int c = (tid < E) ? cnt[tid] : 0;
  const int padded = (c + bs - 1) / bs * bs;
  int total;
  const int excl = block_exclusive_scan(padded, warp_sums, &total);
  if (tid < E) off[tid] = excl;
  if (tid == 0) off[E] = total;
  __syncthreads();
  if (total > a.max_num_tokens_padded || total / bs > a.max_num_m_blocks) {
    if (tid == 0) {
      flag_error(a.err, MOE_LORA_DEVERR_CAPACITY);
      a.num_tokens_post_padded[l] = 0;
    }
    return false;
  }
  if (tid == 0) a.num_tokens_post_padded[l] = total;
  if (tid < E) write_padding(a, l, tid, c, excl);
  return true;
}

// ----------------------------------------------------- shared-memory variant

constexpr int kCache = 8;   // warp-widths of expert ids a lane keeps between the two walks

// The routing of a warp's pairs [lo, hi) (hi - lo <= kCache * 32), loaded
// into registers in one round trip, before the slot's LoRA index is known:
// rm[it] the LoRA of pair lo + 32 it + lane's token (kNoSlot past hi; the
// slot itself, 0, without a mapping), re[it] its expert id.
constexpr int kNoSlot = -2;
__device__ __forceinline__ void warp_load_routing(const AlignArgs &a, int lo, int hi, int lane, int (&rm)[kCache],
                                                  int (&re)[kCache]) {
#pragma unroll
  for (int it = 0; it < kCache; ++it) {
    const int f = lo + it * 32 + lane;
    rm[it] = kNoSlot;
    re[it] = -1;
    if (f < hi) {
      rm[it] = a.token_lora_mapping ? __ldg(a.token_lora_mapping + f / a.topk) : 0;
      re[it] = __ldg(a.topk_ids + f);
    }
  }
}

// The first of the two walks of one warp over [lo, hi), from the routing in
// registers; the pairs' experts (-1: not this slot's, or out of range) stay
// in ec for the second walk.  `tab` is this warp's counter row; `l` the
// slot's LoRA index (0 without a mapping).
__device__ __forceinline__ void warp_count_cached(const AlignArgs &a, int l, int lo, int hi, int *tab, int lane,
                                                  const int (&rm)[kCache], const int (&re)[kCache],
                                                  int (&ec)[kCache]) {
#pragma unroll
  for (int it = 0; it < kCache; ++it) {
    const int base = lo + it * 32;
    ec[it] = -1;
    if (base < hi) {
      int e = -1;
      if (rm[it] == l) {
        e = re[it];
        if (e < 0 || e >= a.num_experts) {
          flag_error(a.err, MOE_LORA_DEVERR_EXPERT_ID);
          e = -1;
        }
      }
      ec[it] = e;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) tab[e] += __popc(peers);
    }
  }
}

__device__ __forceinline__ void warp_scatter_cached(int lo, int hi, int *tab, const int *seg, int32_t *sorted,
                                                    int lane, const int (&ec)[kCache]) {
  const unsigned lower = (1u << lane) - 1u;
#pragma unroll
  for (int it = 0; it < kCache; ++it) {
    const int base = lo + it * 32;
    if (base < hi) {
      const int e = ec[it];
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int pos = (e >= 0) ? tab[e] + seg[e] + __popc(peers & lower) : 0;
      __syncwarp();
      if (e >= 0) {
        sorted[pos] = base + lane;
        if (lane == __ffs(peers) - 1) tab[e] += __popc(peers);
      }
      __syncwarp();
    }
  }
}

// One CTA per active slot, of max(32 W, E) threads rounded up to a warp: the
// pairs are split over the first W warps (W = min(32, ceil(P / 32))), each a
// contiguous range, and the per-warp counters form a W x E table in shared
// memory; one thread per expert does the column scan.
__global__ void __launch_bounds__(kSmemThreads, 1) align_smem_kernel(const AlignArgs a) {
  extern __shared__ int smem[];
  const int E = a.num_experts;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = a.M * a.topk;
  const int W = max(1, min(kSmemWarps, (P + 31) / 32));
  int *tab = smem;                          // [W][E] per-warp counters, then cursors
  int *cnt = tab + W * E;                   // [E]
  int *off = cnt + E;                       // [E + 1]
  int *warp_sums = off + E + 1;             // [32]

  // The fused kernel may be launched as this grid's programmatic dependent; it
  // waits for this grid's completion before it reads any output.
  asm volatile("griddepcontrol.launch_dependents;");

  const int per_warp = ((P + W - 1) / W + 31) / 32 * 32;
  const int lo = min(P, warp * per_warp), hi = warp < W ? min(P, lo + per_warp) : lo;
  const bool cached = per_warp <= kCache * 32;
  // the routing goes out together with the slot's LoRA index (one round trip)
  int rm[kCache], re[kCache];
  if (cached) warp_load_routing(a, lo, hi, lane, rm, re);

  const int l = slot_lora(a, blockIdx.x, tid == 0);
  if (l < 0) return;

  zero_ints(tab, W * E);
  __syncthreads();

  int *mine = tab + (warp < W ? warp : 0) * E;
  int ec[kCache];
  if (warp < W) {
    if (cached) warp_count_cached(a, a.token_lora_mapping ? l : 0, lo, hi, mine, lane, rm, re, ec);
    else warp_count(a, l, lo, hi, mine, lane);
  }
  __syncthreads();

  // Column scan: each warp's starting position relative to its segment.
  column_scan(tab, W, E, cnt);
  __syncthreads();
  if (!write_segments(a, l, cnt, off, warp_sums)) return;

  // a warp's position in segment e: its column-scan entry + the segment's offset
  if (warp < W) {
    int32_t *sorted = a.sorted_token_ids + (size_t)l * a.max_num_tokens_padded;
    if (cached) warp_scatter_cached(lo, hi, mine, off, sorted, lane, ec);
    else warp_scatter(a, l, lo, hi, mine, off, sorted, lane);
  }
}

// ----------------------------------------------------- global-memory variant
// Workspace per slot z: hist[z] = int [W][E] (W warp ranges), then off[z] = int [E].

struct GlobalLayout {
  int pairs_per_warp;
  int warps;  // W
};

__host__ __device__ inline size_t slot_stride_ints(int W, int E) { return (size_t)W * E + E; }

__global__ void __launch_bounds__(kGlobalThreads) align_global_count_kernel(const AlignArgs a, int *ws,
                                                                            GlobalLayout g) {
  extern __shared__ int smem[];
  const int E = a.num_experts;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int z = blockIdx.y;
  const int l = slot_lora(a, z, false);
  if (l < 0) return;
  const int gw = blockIdx.x * kGlobalWarpsPerCta + warp;
  if (blockIdx.x * kGlobalWarpsPerCta >= g.warps) return;
  int *mine = smem + warp * E;
  for (int i = lane; i < E; i += 32) mine[i] = 0;
  __syncwarp();
  const int P = a.M * a.topk;
  if (gw < g.warps) {
    const int lo = min(P, gw * g.pairs_per_warp), hi = min(P, lo + g.pairs_per_warp);
    warp_count(a, l, lo, hi, mine, lane);
    __syncwarp();
    int *hist = ws + (size_t)z * slot_stride_ints(g.warps, E) + (size_t)gw * E;
    for (int i = lane; i < E; i += 32) hist[i] = mine[i];
  }
}

__global__ void __launch_bounds__(kScanThreads, 1) align_global_scan_kernel(const AlignArgs a, int *ws,
                                                                            GlobalLayout g) {
  extern __shared__ int smem[];
  const int E = a.num_experts, tid = threadIdx.x;
  int *cnt = smem;            // [E]
  int *off = cnt + E;         // [E + 1]
  int *warp_sums = off + E + 1;
  const int z = blockIdx.x;
  const int l = slot_lora(a, z, tid == 0);
  if (l < 0) return;
  int *hist = ws + (size_t)z * slot_stride_ints(g.warps, E);
  if (tid < E) {
    int run = 0;
    int w = 0;
    // four independent loads in flight per step
    for (; w + 4 <= g.warps; w += 4) {
      const int t0 = hist[(size_t)(w + 0) * E + tid];
      const int t1 = hist[(size_t)(w + 1) * E + tid];
      const int t2 = hist[(size_t)(w + 2) * E + tid];
      const int t3 = hist[(size_t)(w + 3) * E + tid];
      hist[(size_t)(w + 0) * E + tid] = run; run += t0;
      hist[(size_t)(w + 1) * E + tid] = run; run += t1;
      hist[(size_t)(w + 2) * E + tid] = run; run += t2;
      hist[(size_t)(w + 3) * E + tid] = run; run += t3;
    }
    for (; w < g.warps; ++w) {
      const int t = hist[(size_t)w * E + tid];
      hist[(size_t)w * E + tid] = run;
      run += t;
    }
    cnt[tid] = run;
  }
  __syncthreads();
  if (!write_segments(a, l, cnt, off, warp_sums)) {
    // mark the slot as failed for the scatter kernel
    if (tid == 0) hist[(size_t)g.warps * E] = -1;
    return;
  }
  if (tid < E) hist[(size_t)g.warps * E + tid] = off[tid];
}

__global__ void __launch_bounds__(kGlobalThreads) align_global_scatter_kernel(const AlignArgs a, int *ws,
                                                                              GlobalLayout g) {
  extern __shared__ int smem[];
  asm volatile("griddepcontrol.launch_dependents;");
  const int E = a.num_experts;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int z = blockIdx.y;
  const int l = slot_lora(a, z, false);
  if (l < 0) return;
  const int gw = blockIdx.x * kGlobalWarpsPerCta + warp;
  if (gw >= g.warps) return;
  const int *slot = ws + (size_t)z * slot_stride_ints(g.warps, E);
  const int *seg_off = slot + (size_t)g.warps * E;
  if (__ldg(seg_off) < 0) return;  // capacity failure reported by the scan kernel
  int *mine = smem + warp * E;
  const int *base = slot + (size_t)gw * E;
  for (int i = lane; i < E; i += 32) mine[i] = base[i] + seg_off[i];
  __syncwarp();
  const int P = a.M * a.topk;
  const int lo = min(P, gw * g.pairs_per_warp), hi = min(P, lo + g.pairs_per_warp);
  warp_scatter(a, l, lo, hi, mine, nullptr, a.sorted_token_ids + (size_t)l * a.max_num_tokens_padded, lane);
}

// ----------------------------------------------------- cluster variant
// One thread-block cluster of CA CTAs per active slot (one launch).  CTA c
// takes the pair range [P c / CA, P (c + 1) / CA), counts it per warp (the
// warp histograms of the shared-memory variant), and column-scans its warps.
// The CA CTAs' per-expert counts are then read through distributed shared
// memory: every CTA forms the slot's totals and its own starting position in
// each segment by summing the lower ranks in rank order, so the result is
// the same stable order as the other variants.  Expert e's sentinels and
// block labels are written by CTA e mod CA; every CTA scatters its pairs.

constexpr int kClusterAlignWarps = 32;
constexpr int kClusterAlignThreads = kClusterAlignWarps * 32;
constexpr int kMaxAlignCluster = 8;

__global__ void __launch_bounds__(kClusterAlignThreads, 1) align_cluster_kernel(const AlignArgs a, int CA) {
  extern __shared__ int smem[];
  const int E = a.num_experts;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = a.M * a.topk;
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int z = blockIdx.x / CA;
  int *tab = smem;                                    // [W][E] per-warp counters, then column-scanned
  int *cnt = tab + kClusterAlignWarps * E;            // [E] this CTA's counts (read by peers)
  int *before = cnt + E;                              // [E] pairs of lower-ranked CTAs, then scatter bases
  int *tot = before + E;                              // [E] the slot's counts
  int *off = tot + E;                                 // [E + 1]
  int *warp_sums = off + E + 1;                       // [32]

  asm volatile("griddepcontrol.launch_dependents;");

  const int lo_c = (int)((long long)P * c / CA), hi_c = (int)((long long)P * (c + 1) / CA);
  const int per_warp = ((hi_c - lo_c + kClusterAlignWarps - 1) / kClusterAlignWarps + 31) / 32 * 32;
  const int lo = min(hi_c, lo_c + warp * per_warp), hi = min(hi_c, lo + per_warp);
  const bool cached = per_warp <= kCache * 32;
  // the routing goes out together with the slot's LoRA index (one round trip)
  int rm[kCache], re[kCache];
  if (cached) warp_load_routing(a, lo, hi, lane, rm, re);

  const int l = slot_lora(a, z, tid == 0 && c == 0);   // the same for every CTA of the cluster
  if (l < 0) return;                                    // (the whole cluster returns)

  zero_ints(tab, kClusterAlignWarps * E);
  __syncthreads();
  int *mine = tab + warp * E;
  int ec[kCache];
  if (cached) warp_count_cached(a, a.token_lora_mapping ? l : 0, lo, hi, mine, lane, rm, re, ec);
  else warp_count(a, l, lo, hi, mine, lane);
  __syncthreads();
  // column scan over this CTA's warps
  column_scan(tab, kClusterAlignWarps, E, cnt);
  // every CTA's counts are complete before any CTA reads them
  cluster_arrive_release();
  cluster_wait();
  if (tid < E) {
    int total = 0, below = 0;
    for (int q = 0; q < CA; ++q) {
      const int v = cluster.map_shared_rank(cnt, q)[tid];
      total += v;
      if (q < c) below += v;
    }
    before[tid] = below;
    tot[tid] = total;
  }
  // This CTA reads no peer's counts after this.  The matching wait is at the
  // end: no CTA exits while a peer may still read its counts.
  cluster_arrive_relaxed();
  __syncthreads();
  bool ok;
  {
    const int n_e = tid < E ? tot[tid] : 0;
    const int padded = (n_e + a.block_size - 1) / a.block_size * a.block_size;
    int total;
    const int excl = block_exclusive_scan(padded, warp_sums, &total);
    if (tid < E) {
      off[tid] = excl;
      before[tid] += excl;   // this CTA's first position in segment tid
    }
    if (tid == 0) off[E] = total;
    __syncthreads();
    ok = total <= a.max_num_tokens_padded && total / a.block_size <= a.max_num_m_blocks;
    if (!ok) {
      if (tid == 0 && c == 0) {
        flag_error(a.err, MOE_LORA_DEVERR_CAPACITY);
        a.num_tokens_post_padded[l] = 0;
      }
    } else {
      if (tid == 0 && c == 0) a.num_tokens_post_padded[l] = total;
      // experts e = c, c + CA, ...: sentinels and block labels by this CTA
      write_padding_warps(a, l, tot, off, c, CA);
    }
  }
  if (ok) {
    // a warp's position in segment e: its column-scan entry + this CTA's base
    int32_t *sorted = a.sorted_token_ids + (size_t)l * a.max_num_tokens_padded;
    if (cached) warp_scatter_cached(lo, hi, mine, before, sorted, lane, ec);
    else warp_scatter(a, l, lo, hi, mine, before, sorted, lane);
  }
  cluster_wait();
}

int set_smem_limit(const void *fn, size_t bytes) {
  if (bytes <= 48 * 1024) return 0;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
                 cudaSuccess
             ? 0
             : MOE_LORA_ERR_LAUNCH;
}

}  // namespace

bool align_smem_fits(int E) {
  const size_t bytes = ((size_t)kSmemWarps * E + 2 * (size_t)E + 1 + 32) * sizeof(int);
  return bytes <= 200 * 1024;
}

int align_global_pairs_per_warp(int M, int topk) {
  const long long P = (long long)M * topk;
  long long per = (P + kMaxGlobalWarpRanges - 1) / kMaxGlobalWarpRanges;
  per = (per + 31) / 32 * 32;
  return (int)(per < 32 ? 32 : per);
}

size_t align_global_workspace_bytes(int M, int topk, int E, int nact) {
  const long long P = (long long)M * topk;
  const int per = align_global_pairs_per_warp(M, topk);
  const long long W = P > 0 ? (P + per - 1) / per : 1;
  return (size_t)nact * slot_stride_ints((int)W, E) * sizeof(int);
}

int launch_align_smem(const AlignArgs &a, cudaStream_t stream) {
  const long long P = (long long)a.M * a.topk;
  const int W = (int)std::max(1LL, std::min<long long>(kSmemWarps, (P + 31) / 32));
  const size_t bytes = ((size_t)W * a.num_experts + 2 * (size_t)a.num_experts + 1 + 32) * sizeof(int);
  const int threads = std::min(kSmemThreads, (std::max(32 * W, a.num_experts) + 31) / 32 * 32);
  if (int st = set_smem_limit((const void *)align_smem_kernel, bytes)) return st;
  align_smem_kernel<<<a.num_active_loras, threads, bytes, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

int align_cluster_size(int M, int topk) {
  // about 2048 pairs (64 per warp, kept in registers between the walks) per
  // CTA, at most 8 CTAs (larger clusters could not all be placed at once:
  // 16-CTA clusters took 12.3 us on the large-E routing against 7.6)
  const long long P = (long long)M * topk;
  long long ca = (P + 2047) / 2048;
  if (ca < 1) ca = 1;
  if (ca > kMaxAlignCluster) ca = kMaxAlignCluster;
  int c = 1;
  while (c < ca) c <<= 1;
  return c;
}

bool align_cluster_fits(int E) {
  const size_t bytes = ((size_t)kClusterAlignWarps * E + 4 * (size_t)E + 1 + 32) * sizeof(int);
  return bytes <= 200 * 1024;
}

int launch_align_cluster(const AlignArgs &a, cudaStream_t stream) {
  const int CA = align_cluster_size(a.M, a.topk);
  const size_t bytes = ((size_t)kClusterAlignWarps * a.num_experts + 4 * (size_t)a.num_experts + 1 + 32) * sizeof(int);
  if (cudaFuncSetAttribute((const void *)align_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes) != cudaSuccess)
    return MOE_LORA_ERR_LAUNCH;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)(a.num_active_loras * CA), 1, 1);
  lc.blockDim = dim3(kClusterAlignThreads, 1, 1);
  lc.dynamicSmemBytes = bytes;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CA;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, align_cluster_kernel, a, CA) == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

int launch_align_global(const AlignArgs &a, void *workspace, cudaStream_t stream) {
  const long long P = (long long)a.M * a.topk;
  GlobalLayout g;
  g.pairs_per_warp = align_global_pairs_per_warp(a.M, a.topk);
  g.warps = P > 0 ? (int)((P + g.pairs_per_warp - 1) / g.pairs_per_warp) : 1;
  int *ws = static_cast<int *>(workspace);
  const int E = a.num_experts;
  const size_t warp_tab = (size_t)kGlobalWarpsPerCta * E * sizeof(int);
  const size_t scan_bytes = (2 * (size_t)E + 1 + 32) * sizeof(int);
  if (int st = set_smem_limit((const void *)align_global_count_kernel, warp_tab)) return st;
  if (int st = set_smem_limit((const void *)align_global_scatter_kernel, warp_tab)) return st;
  const dim3 grid((g.warps + kGlobalWarpsPerCta - 1) / kGlobalWarpsPerCta, a.num_active_loras);
  align_global_count_kernel<<<grid, kGlobalThreads, warp_tab, stream>>>(a, ws, g);
  align_global_scan_kernel<<<a.num_active_loras, kScanThreads, scan_bytes, stream>>>(a, ws, g);
  align_global_scatter_kernel<<<grid, kGlobalThreads, warp_tab, stream>>>(a, ws, g);
  return cudaGetLastError() == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

}  // namespace moe_lora
