// stream_pipeline.cuh -- the streaming skeleton shared by the two fused
// kernels that walk balanced (block, output tile) ranges: the tensor-core
// kernel (fused_tcgen05.cu) and the CUDA-core streaming kernel
// (fused_stream_cc.cu).
//
// The work of a call is the list of (block, slice, 128-column tile) triples
// over all blocks of all listed slots (vLLM PR #32005: the grid is sized by the
// active LoRAs) and all adapter slices.  A (block, slice) pair is a "unit";
// units are numbered block-major (unit = block * num_slices + slice) so that
// the slices of one block, which gather the same x rows, run back to back.
// Each persistent CTA takes a share of that list (cta_range: equal shares of
// (unit, tile) pairs, or whole units strided over the grid).  For every unit
// it touches it needs that unit's rank-r intermediate (the shrink over all of
// K), then it produces its tiles of the unit.
//
// Two producers feed the consumers through shared-memory rings guarded by
// mbarriers:
//   * shrink producers (two warps, alternating k-tiles): the A tile of each
//     64-wide K step by TMA (3-D tensor map, rows past the rank zero-filled)
//     and the block's x rows by 16-byte cp.async, both into 128-byte-swizzled
//     K-major tiles;
//   * expand producer (one warp): the B tile of each 128-column output tile by
//     TMA (swizzle width matched to the rank) and the y_in rows of the tile by
//     16-byte cp.async.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_utils.cuh"
#include "internal.h"

namespace moe_lora {
namespace stream {

constexpr int kMaxSlots = 128;
constexpr int kTileK = 64;        // shrink K per stage (one 128-byte swizzle row)
constexpr int kTileN = 128;       // expand output columns per tile
constexpr int kMaxStages = 12;
constexpr int kMaxLag = 4;

struct Cfg {
  int r_pad;          // rank rounded up to 16, 32, 64 or 128
  int ka;             // expand K atom width in elements: 16, 32 or 64 (32/64/128-byte swizzle)
  int natoms;         // r_pad / ka
  int s_sh, lag, s_ex;
  int t_bufs;         // (tensor-core kernel) T buffers
  int nacc;           // (tensor-core kernel) expand accumulators in TMEM
  int tmem_cols;
  int off_sh, sh_stage, at_off;   // shrink stage: x tile (block_size rows), A tile at +at_off
  int off_ex, ex_stage, yt_off;   // expand stage: B tile, y tile at +yt_off
  int off_t, t_part;              // consumer-private region (T tiles or fp32 t)
  int off_meta;
  int smem_bytes;
  int kt_total, nt_total;
  long long unit_sh_bytes;   // bytes one unit's shrink streams (x rows + A, all k-tiles)
  long long tile_bytes;      // bytes one expand tile streams (B tile + y_in rows)
};

// The A and B tensor maps of every slice (kernel parameter).
struct TmapSet {
  CUtensorMap a[kMaxSlices];
  CUtensorMap b[kMaxSlices];
};

struct Meta {
  uint64_t full_sh[kMaxStages], empty_sh[kMaxStages];
  uint64_t full_ex[kMaxStages], empty_ex[kMaxStages];
  uint64_t tfull[2], tempty[2];   // (tensor-core kernel) the two expand accumulators
  uint64_t shrink_done, shrink_free;
  uint64_t t_full[2], t_empty[2];
  uint32_t tmem_base;
  int abort;
  int nv;
  int prefix[kMaxSlots + 1];
  int prod_f[128];    // expand producer's copy of the current block's pair ids (-1 = padding)
  int epi_f[128];     // consumers' copy
  float epi_w[128];   // consumers: router weight of each row's pair
  int cpx[128];       // consumers: rows (positions in the block) of the real pairs, in order
  int wcount[8];      // (CUDA-core kernel) real pairs per compute warp
};

// Shared-memory descriptor of a K-major operand tile whose rows are
// `row_bytes` (32, 64 or 128) long and swizzled at that width (16-byte chunk c
// of row r stored at chunk position c ^ ((r * row_bytes / 128) mod (row_bytes / 16))).
// 8-row groups are 8 * row_bytes apart; the tile base is aligned to that.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, int row_bytes) {
  const uint64_t layout = row_bytes == 128 ? 2 : (row_bytes == 64 ? 4 : 6);
  return (uint64_t((saddr & 0x3FFFFu) >> 4)) | (uint64_t(1) << 16) | (uint64_t((8 * row_bytes) >> 4) << 32) |
         (uint64_t(1) << 46) | (layout << 61);
}

// Byte offset of 16-byte chunk `c` of row `r` in such a tile.
__device__ __forceinline__ uint32_t swz(int r, int c, int row_bytes) {
  const int mask = row_bytes / 16 - 1;
  return (uint32_t)(r * row_bytes + ((c ^ ((r * row_bytes >> 7) & mask)) << 4));
}

__device__ __forceinline__ int find_slot(const int *prefix, int nact, int item) {
  int lo = 0, hi = nact;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid;
  }
  return lo;
}

struct BlockRef {
  int l, e, s;          // LoRA, expert and adapter slice of the unit
  const int32_t *ids;   // the block's pair ids
};

template <int BS>
__device__ __forceinline__ BlockRef block_ref(const FusedArgs &p, const Meta &meta, int unit) {
  BlockRef br;
  const int gb = unit / p.num_slices;
  br.s = unit - gb * p.num_slices;
  const int z = find_slot(meta.prefix, p.num_active_loras, gb);
  br.l = __ldg(p.lora_ids + z);
  const int b = gb - meta.prefix[z];
  br.e = __ldg(p.expert_ids + (size_t)br.l * p.max_num_m_blocks + b);
  br.ids = p.sorted_token_ids + (size_t)br.l * p.max_num_tokens_padded + (size_t)b * BS;
  return br;
}

// Blocks per listed slot and their prefix sum, into meta.prefix (all threads).
template <int BS>
__device__ __forceinline__ void slot_prefix(const FusedArgs &p, Meta &meta) {
  for (int z = threadIdx.x; z < p.num_active_loras; z += blockDim.x) {
    const int l = __ldg(p.lora_ids + z);
    int nb = 0;
    if (l < 0 || l >= p.max_loras) {
      if (blockIdx.x == 0) flag_error(p.err, MOE_LORA_DEVERR_LORA_ID);
    } else if (!p.adapter_enabled || __ldg(p.adapter_enabled + l) != 0) {
      nb = __ldg(p.num_tokens_post_padded + l) / BS;
      nb = max(0, min(nb, p.max_num_m_blocks));
    }
    meta.prefix[z + 1] = nb;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    meta.prefix[0] = 0;
    for (int z = 0; z < p.num_active_loras; ++z) meta.prefix[z + 1] += meta.prefix[z];
  }
}

// This CTA's share [t0, t1) of the (unit, tile) list and the units it touches
// (gb0..gb1 number units).
struct Range {
  long long t0, t1;
  int gb0, gb1, step;   // units gb0, gb0 + step, ..., gb1
  int nt_total;
  __device__ int tile_lo(int gb) const { return (int)max(t0 - (long long)gb * nt_total, 0LL); }
  __device__ int tile_hi(int gb) const { return (int)min(t1 - (long long)gb * nt_total, (long long)nt_total); }
};

// Two ways to split the list: equal shares of (unit, tile) pairs, where a
// unit cut by a share boundary has its shrink streamed by both CTAs, or whole
// units, at most ceil(units / CTAs) each.  Every CTA takes the one whose
// busiest CTA streams fewer bytes (the same choice everywhere: it depends on
// the unit count, the grid and the configuration only).  Whole units are
// strided over the grid, so units of one segment share their adapter reads
// through L2, which the byte count leaves out: they are taken within 3%.
__device__ __forceinline__ Range cta_range(const Meta &meta, int nact, int num_slices, const Cfg &cfg) {
  Range rg;
  const int nt_total = cfg.nt_total;
  const long long units = (long long)meta.prefix[nact] * num_slices;
  const long long total = units * nt_total;
  const double per = (double)units / gridDim.x;
  const double shared_cost = (per + 1.0) * (double)cfg.unit_sh_bytes + per * nt_total * (double)cfg.tile_bytes;
  const double whole_cost = ceil(per) * ((double)cfg.unit_sh_bytes + nt_total * (double)cfg.tile_bytes);
  if (whole_cost < 1.03 * shared_cost) {
    // Whole units, strided over the grid: units u = blockIdx.x + i * gridDim.x.
    // Consecutive units (the blocks of one segment share its A and B) run on
    // neighbouring CTAs at the same time, so the later reads come from L2.
    rg.t0 = 0;
    rg.t1 = total;
    rg.nt_total = nt_total;
    rg.step = gridDim.x;
    rg.gb0 = blockIdx.x;
    rg.gb1 = units > blockIdx.x ? (int)(blockIdx.x + (units - 1 - blockIdx.x) / gridDim.x * gridDim.x)
                                : rg.gb0 - rg.step;
    return rg;
  }
  rg.t0 = total * blockIdx.x / gridDim.x;
  rg.t1 = total * (blockIdx.x + 1) / gridDim.x;
  rg.step = 1;
  rg.nt_total = nt_total;
  rg.gb0 = (int)(rg.t0 / nt_total);
  rg.gb1 = rg.t1 > rg.t0 ? (int)((rg.t1 - 1) / nt_total) : rg.gb0 - 1;
  return rg;
}

// Shrink producer `me` (0 or 1) of two: k-tiles alternate between them.  Each
// k-tile: the A tile by TMA into the stage, the block's x rows (16-byte chunk
// lane % 8 of rows lane/8 + 4i) by cp.async; a stage is released `lag` owned
// k-tiles later, once its copies are complete and fenced for async-proxy
// readers.
template <int BS>
__device__ void shrink_producer(const FusedArgs &p, const Cfg &cfg, Meta &meta, const TmapSet *maps,
                                uint8_t *sh_base, const Range &rg, int me) {
  const int lane = threadIdx.x & 31;
  const int K = p.K, E = p.num_experts, P = p.M * p.topk;
  volatile int *abort = &meta.abort;
  constexpr int kRowsPerLane = BS / 4;
  const int ch = lane & 7;
  uint32_t sh_iter = 0;
  int owned = 0;
  for (int gb = rg.gb0; gb <= rg.gb1; gb += rg.step) {
    const BlockRef br = block_ref<BS>(p, meta, gb);
    const bool e_ok = br.e >= 0 && br.e < E;
    if (!e_ok && lane == 0 && me == 0) flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
    const int le = br.l * E + (e_ok ? br.e : 0);
    const CUtensorMap *tmap_a = &maps->a[br.s];
    int xrow[kRowsPerLane];
#pragma unroll
    for (int i = 0; i < kRowsPerLane; ++i) {
      const int f = __ldg(br.ids + (lane >> 3) + 4 * i);
      xrow[i] = (f >= 0 && f < P && e_ok) ? x_row(p, f) : -1;
    }
    for (int kt = 0; kt < cfg.kt_total; ++kt, ++sh_iter) {
      if ((int)(sh_iter & 1) != me) continue;
      const int s = sh_iter % cfg.s_sh;
      const uint32_t n = sh_iter / cfg.s_sh;
      if (sh_iter >= (uint32_t)cfg.s_sh) mbar_wait(&meta.empty_sh[s], (n - 1) & 1, abort, p.err);
      uint8_t *xt = sh_base + (size_t)s * cfg.sh_stage;
      if (lane == 0) {
        mbar_arrive_expect_tx(&meta.full_sh[s], (uint32_t)cfg.r_pad * 128);
        tma_load_3d(xt + cfg.at_off, tmap_a, kt * kTileK, 0, le, &meta.full_sh[s]);
      }
      const int k = kt * kTileK + ch * 8;
#pragma unroll
      for (int i = 0; i < kRowsPerLane; ++i) {
        const int pr = (lane >> 3) + 4 * i;
        const bool ok = xrow[i] >= 0 && k < K;
        cp_async_16(xt + pr * 128 + ((ch ^ (pr & 7)) << 4), ok ? p.x + (size_t)xrow[i] * K + k : p.x,
                    ok ? 16u : 0u);
      }
      cp_async_commit();
      if (owned >= cfg.lag) {
        switch (cfg.lag) {
          case 0: cp_async_wait_group<0>(); break;
          case 1: cp_async_wait_group<1>(); break;
          case 2: cp_async_wait_group<2>(); break;
          case 3: cp_async_wait_group<3>(); break;
          default: cp_async_wait_group<4>(); break;
        }
        fence_proxy_async_cta();
        mbar_arrive(&meta.full_sh[(sh_iter - 2 * cfg.lag) % cfg.s_sh]);
      }
      ++owned;
    }
  }
  cp_async_wait_group<0>();
  fence_proxy_async_cta();
  const int tail = min(owned, cfg.lag);
  uint32_t k_last = sh_iter - 1;          // the last k-tile this warp owned
  if ((int)(k_last & 1) != me) --k_last;
  for (int i = tail - 1; i >= 0; --i) mbar_arrive(&meta.full_sh[(k_last - 2 * i) % cfg.s_sh]);
}

// Expand producer: per tile, the B tile by TMA and the y_in rows (16-byte chunk
// lane % 16 of rows lane/16 + 2i, real pairs only) by cp.async.  The row ids
// are read before any copy is issued so that the copies go out back to back.
template <int BS>
__device__ void expand_producer(const FusedArgs &p, const Cfg &cfg, Meta &meta, const TmapSet *maps,
                                uint8_t *ex_base, const Range &rg) {
  const int lane = threadIdx.x & 31;
  const int E = p.num_experts, N = p.N, P = p.M * p.topk;
  const int kb = cfg.ka * 2;
  volatile int *abort = &meta.abort;
  uint32_t ex_iter = 0;
  for (int gb = rg.gb0; gb <= rg.gb1; gb += rg.step) {
    const BlockRef br = block_ref<BS>(p, meta, gb);
    const int le = br.l * E + ((br.e >= 0 && br.e < E) ? br.e : 0);
    const CUtensorMap *tmap_b = &maps->b[br.s];
    const int s_col = p.y_offset + br.s * N;   // this slice's first output column
    __syncwarp();
    for (int pr = lane; pr < BS; pr += 32) {
      const int f = __ldg(br.ids + pr);
      meta.prod_f[pr] = (f >= 0 && f < P) ? f : -1;
    }
    __syncwarp();
    for (int nt = rg.tile_lo(gb); nt < rg.tile_hi(gb); ++nt, ++ex_iter) {
      const int s = ex_iter % cfg.s_ex;
      const uint32_t n = ex_iter / cfg.s_ex;
      if (ex_iter >= (uint32_t)cfg.s_ex) mbar_wait(&meta.empty_ex[s], (n - 1) & 1, abort, p.err);
      uint8_t *bt = ex_base + (size_t)s * cfg.ex_stage;
      uint8_t *yt = bt + cfg.yt_off;
      const int n0 = nt * kTileN;
      if (lane == 0) {
        mbar_arrive_expect_tx(&meta.full_ex[s], (uint32_t)cfg.natoms * kTileN * kb);
        for (int a = 0; a < cfg.natoms; ++a)
          tma_load_3d(bt + a * (kTileN * kb), tmap_b, a * cfg.ka, n0, le, &meta.full_ex[s]);
      }
      if (p.add_inputs) {
        const int c16 = lane & 15;
        const int nn = n0 + c16 * 8;
        if (nn < N) {
          constexpr int kRows = BS / 2;
          int fr[kRows];
#pragma unroll
          for (int i = 0; i < kRows; ++i) fr[i] = meta.prod_f[(lane >> 4) + 2 * i];
#pragma unroll
          for (int i = 0; i < kRows; ++i)
            if (fr[i] >= 0)
              cp_async_16(yt + ((lane >> 4) + 2 * i) * (kTileN * 2) + c16 * 16,
                          p.y + (size_t)fr[i] * p.ldy + s_col + nn, 16u);
        }
      }
      cp_async_mbar_arrive_noinc(&meta.full_ex[s]);
    }
  }
}

// ------------------------------------------------------------------ host side

int encode_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
              CUtensorMapSwizzle swizzle);

// Tensor maps of every slice's A ([L*E, r, K], 64 x r_pad boxes, 128-byte
// swizzle) and B ([L*E, N, r], ka x 128 boxes, swizzle matched to ka).
int make_tensor_maps(const FusedArgs &f, const Cfg &cfg, TmapSet *maps);

// Fill the geometry of cfg (r_pad, ka, stage sizes, tile counts) and choose
// ring depths for a consumer region of `consumer_bytes` (per T buffer, up to
// t_bufs_max buffers) that fit the shared memory of one CTA.
int plan(const FusedArgs &f, const DeviceInfo &dev, int consumer_bytes, int t_bufs_max, Cfg *cfg);

}  // namespace stream
}  // namespace moe_lora
