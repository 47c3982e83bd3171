// fused_tcgen05.cu -- the prefill-sized fused MoE-LoRA shrink+expand on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// Same definition as the CUDA-core path (prhub.com.cn summary of vLLM PR
// #42290, "Implementation breakdown" step 1: shrink by lora_a, expand by
// lora_b, rank dimension kept on chip, add_inputs accumulate/overwrite):
//     T[p][j]   = sum_k x[m_p][k] * A[l][e][j][k]        p < block_size, j < r
//     y[f_p][n] = bf16((add ? y[f_p][n] : 0) + sum_j B[l][e][n][j] * T[p][j])
//
// Work split.  The work of a call is the list of (block, 128-column tile)
// pairs over all blocks of all listed slots (vLLM PR #32005: the grid is sized
// by the active LoRAs).  Each persistent CTA takes one contiguous, equal share
// of that list, so every SM streams the same number of output tiles; a block
// whose tiles straddle two CTAs has its shrink computed by both.  T lives only
// in shared and tensor memory.
//
// Warp roles (416 threads):
//   warps 10, 11  shrink producers: alternate k-tiles; gather the block's x rows
//                 with 16-byte cp.async into 128-byte-swizzled K-major tiles and
//                 TMA-load the A tile (3-D tensor map, out-of-bounds rows zero).
//   warp 12       shrink MMA: D[128 x r_pad] = X[128 x 64] * A[r_pad x 64]^T
//                 over the K tiles, into its own TMEM columns.
//   warps 2..9    epilogue: (i) read the shrink accumulator and write T as two
//                 bf16 tiles, T_hi = bf16(T) and T_lo = bf16(T - T_hi), so the
//                 expand keeps fp32-level accuracy; (ii) per output tile, read the
//                 expand accumulator, add y_in, round to bf16, store 16-byte rows.
//   warp 0        expand producer: TMA-loads B tiles (swizzle width matched to
//                 the rank) and cp.async-loads the y_in rows of each tile.
//   warp 1        expand MMA (and TMEM owner): D[128 cols x bs] = B * T^T over
//                 T_hi and T_lo, double-buffered in TMEM; output columns sit on
//                 the 128 TMEM lanes so every lane quarter carries data.
// The next block's shrink runs while the current block's tiles are expanded
// (separate producers, separate MMA issuers, T double-buffered when it fits).
// Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_utils.cuh"
#include "internal.h"

namespace moe_lora {

namespace {

constexpr int kWarps = 13;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kMaxSlots = 128;
constexpr int kTileK = 64;        // shrink K per stage (one 128-byte swizzle row)
constexpr int kTileN = 128;       // expand output columns per tile (TMEM lanes)
constexpr int kMmaRows = 128;     // M of every tcgen05.mma here
constexpr int kMaxStages = 12;
constexpr int kMaxLag = 4;

struct TcCfg {
  int r_pad;          // rank rounded up to 16, 32, 64 or 128
  int ka;             // expand K atom width in elements: 16, 32 or 64 (32/64/128-byte swizzle)
  int natoms;         // r_pad / ka
  int s_sh, lag, s_ex, t_bufs;
  int tmem_cols;
  int off_sh, sh_stage, at_off;   // shrink stage: x tile (block_size rows), A tile at +at_off
  int off_ex, ex_stage, yt_off;   // expand stage: B tile, y tile at +yt_off
  int off_t, t_part;              // T buffers: [t_bufs][hi, lo] of t_part bytes each
  int off_meta;
  int smem_bytes;
  int kt_total, nt_total;
};

struct TcMeta {
  uint64_t full_sh[kMaxStages], empty_sh[kMaxStages];
  uint64_t full_ex[kMaxStages], empty_ex[kMaxStages];
  uint64_t tfull[2], tempty[2];
  uint64_t shrink_done, shrink_free;
  uint64_t t_full[2], t_empty[2];
  uint32_t tmem_base;
  int abort;
  int prefix[kMaxSlots + 1];
  int prod_f[128];    // expand producer's copy of the current block's pair ids (-1 = padding)
  int epi_f[128];     // epilogue's copy
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
  int l, e;
  const int32_t *ids;
};

template <int BS>
__device__ __forceinline__ BlockRef block_ref(const FusedArgs &p, const TcMeta &meta, int gb) {
  BlockRef br;
  const int z = find_slot(meta.prefix, p.num_active_loras, gb);
  br.l = __ldg(p.lora_ids + z);
  const int b = gb - meta.prefix[z];
  br.e = __ldg(p.expert_ids + (size_t)br.l * p.max_num_m_blocks + b);
  br.ids = p.sorted_token_ids + (size_t)br.l * p.max_num_tokens_padded + (size_t)b * BS;
  return br;
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
    fused_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const FusedArgs p, const TcCfg cfg) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  TcMeta &meta = *reinterpret_cast<TcMeta *>(smem + cfg.off_meta);
  uint8_t *sh_base = smem + cfg.off_sh;
  uint8_t *ex_base = smem + cfg.off_ex;
  uint8_t *t_base = smem + cfg.off_t;
  const int K = p.K, N = p.N, E = p.num_experts, r = p.rank, r_pad = cfg.r_pad;
  const int P = p.M * p.topk;
  const int kt_total = cfg.kt_total, nt_total = cfg.nt_total;
  const int kb = cfg.ka * 2;     // bytes per expand-operand row per atom
  volatile int *abort = &meta.abort;

  if (tid == 0) {
    for (int s = 0; s < cfg.s_sh; ++s) {
      mbar_init(&meta.full_sh[s], 1 + 32);
      mbar_init(&meta.empty_sh[s], 1);
    }
    for (int s = 0; s < cfg.s_ex; ++s) {
      mbar_init(&meta.full_ex[s], 1 + 32);
      mbar_init(&meta.empty_ex[s], 1 + kEpiWarps / 2);   // MMA commit + the 4 warps of one group
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&meta.tfull[a], 1);
      mbar_init(&meta.tempty[a], kEpiWarps / 2);       // accumulator a is drained by group a
      mbar_init(&meta.t_full[a], kEpiWarps);
      mbar_init(&meta.t_empty[a], 1);
    }
    mbar_init(&meta.shrink_done, 1);
    mbar_init(&meta.shrink_free, kEpiWarps);
    meta.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensor_map(&tmap_a);
    prefetch_tensor_map(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(&meta.tmem_base, cfg.tmem_cols);
    tmem_relinquish();
  }
  wait_for_prior_grid();   // align outputs are read from here on
  for (int z = tid; z < p.num_active_loras; z += kThreads) {
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
  if (tid == 0) {
    meta.prefix[0] = 0;
    for (int z = 0; z < p.num_active_loras; ++z) meta.prefix[z + 1] += meta.prefix[z];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = meta.tmem_base;
  const uint32_t tmem_sh = tmem + 2 * BS;   // shrink accumulator columns

  // This CTA's share of the (block, tile) list.
  const long long total = (long long)meta.prefix[p.num_active_loras] * nt_total;
  const long long t0 = total * blockIdx.x / gridDim.x, t1 = total * (blockIdx.x + 1) / gridDim.x;
  const int gb0 = (int)(t0 / nt_total), gb1 = t1 > t0 ? (int)((t1 - 1) / nt_total) : gb0 - 1;
  auto tile_lo = [&](int gb) { return (int)std::max<long long>(t0 - (long long)gb * nt_total, 0); };
  auto tile_hi = [&](int gb) { return (int)std::min<long long>(t1 - (long long)gb * nt_total, nt_total); };

  if (warp == 10 || warp == 11) {
    // ======================= shrink producers (k-tiles alternate between the two warps)
    const int me = warp - 10;
    constexpr int kRowsPerLane = BS / 4;   // lane gathers chunk (lane % 8) of rows lane/8 + 4i
    const int ch = lane & 7;
    uint32_t sh_iter = 0;
    int owned = 0;
    for (int gb = gb0; gb <= gb1; ++gb) {
      const BlockRef br = block_ref<BS>(p, meta, gb);
      const bool e_ok = br.e >= 0 && br.e < E;
      if (!e_ok && lane == 0 && me == 0) flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
      const int le = br.l * E + (e_ok ? br.e : 0);
      int xrow[kRowsPerLane];
#pragma unroll
      for (int i = 0; i < kRowsPerLane; ++i) {
        const int f = __ldg(br.ids + (lane >> 3) + 4 * i);
        xrow[i] = (f >= 0 && f < P && e_ok) ? f / p.topk : -1;
      }
      for (int kt = 0; kt < kt_total; ++kt, ++sh_iter) {
        if ((int)(sh_iter & 1) != me) continue;
        const int s = sh_iter % cfg.s_sh;
        const uint32_t n = sh_iter / cfg.s_sh;
        if (sh_iter >= (uint32_t)cfg.s_sh) mbar_wait(&meta.empty_sh[s], (n - 1) & 1, abort, p.err);
        uint8_t *xt = sh_base + (size_t)s * cfg.sh_stage;
        if (lane == 0) {
          mbar_arrive_expect_tx(&meta.full_sh[s], (uint32_t)r_pad * 128);
          tma_load_3d(xt + cfg.at_off, &tmap_a, kt * kTileK, 0, le, &meta.full_sh[s]);
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
        // Release this warp's stage issued `lag` owned k-tiles ago (owned
        // k-tiles are every other one): its copies are complete, and the fence
        // makes them visible to the tensor core's (async-proxy) reads.
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
    {
      const int tail = std::min(owned, cfg.lag);
      uint32_t k_last = sh_iter - 1;          // the last k-tile this warp owned
      if ((int)(k_last & 1) != me) --k_last;
      for (int i = tail - 1; i >= 0; --i) mbar_arrive(&meta.full_sh[(k_last - 2 * i) % cfg.s_sh]);
    }
  } else if (warp == 12) {
    // ======================= shrink MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_bf16(kMmaRows, r_pad);
      uint32_t sh_iter = 0;
      int kk = 0;
      for (int gb = gb0; gb <= gb1; ++gb, ++kk) {
        if (kk > 0) mbar_wait(&meta.shrink_free, (kk - 1) & 1, abort, p.err);
        tc_fence_after();
        for (int kt = 0; kt < kt_total; ++kt, ++sh_iter) {
          const int s = sh_iter % cfg.s_sh;
          mbar_wait(&meta.full_sh[s], (sh_iter / cfg.s_sh) & 1, abort, p.err);
          tc_fence_after();
          const uint32_t xa = smem_addr(sh_base + (size_t)s * cfg.sh_stage);
          const uint32_t aa = xa + cfg.at_off;
#pragma unroll
          for (int k16 = 0; k16 < kTileK / 16; ++k16)
            tc_mma_bf16(tmem_sh, make_sdesc(xa + k16 * 32, 128), make_sdesc(aa + k16 * 32, 128), idesc,
                        (kt | k16) ? 1u : 0u);
          tc_commit(&meta.empty_sh[s]);
        }
        tc_commit(&meta.shrink_done);
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // ======================= expand producer
    uint32_t ex_iter = 0;
    for (int gb = gb0; gb <= gb1; ++gb) {
      const BlockRef br = block_ref<BS>(p, meta, gb);
      const int le = br.l * E + ((br.e >= 0 && br.e < E) ? br.e : 0);
      __syncwarp();
      for (int pr = lane; pr < BS; pr += 32) {
        const int f = __ldg(br.ids + pr);
        meta.prod_f[pr] = (f >= 0 && f < P) ? f : -1;
      }
      __syncwarp();
      for (int nt = tile_lo(gb); nt < tile_hi(gb); ++nt, ++ex_iter) {
        const int s = ex_iter % cfg.s_ex;
        const uint32_t n = ex_iter / cfg.s_ex;
        if (ex_iter >= (uint32_t)cfg.s_ex) mbar_wait(&meta.empty_ex[s], (n - 1) & 1, abort, p.err);
        uint8_t *bt = ex_base + (size_t)s * cfg.ex_stage;
        uint8_t *yt = bt + cfg.yt_off;
        const int n0 = nt * kTileN;
        if (lane == 0) {
          mbar_arrive_expect_tx(&meta.full_ex[s], (uint32_t)cfg.natoms * kTileN * kb);
          for (int a = 0; a < cfg.natoms; ++a)
            tma_load_3d(bt + a * (kTileN * kb), &tmap_b, a * cfg.ka, n0, le, &meta.full_ex[s]);
        }
        if (p.add_inputs) {
          // y_in rows through the load/store unit: lane takes 16-byte chunk
          // (lane % 16) of rows lane/16 + 2i; the row ids are read before any
          // copy is issued so that the copies go out back to back.
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
                cp_async_16(yt + ((lane >> 4) + 2 * i) * (kTileN * 2) + c16 * 16, p.y + (size_t)fr[i] * N + nn, 16u);
          }
        }
        cp_async_mbar_arrive_noinc(&meta.full_ex[s]);
      }
    }
  } else if (warp == 1) {
    // ======================= expand MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_bf16(kMmaRows, BS);
      uint32_t ex_iter = 0, acc_iter = 0;
      int kk = 0;
      for (int gb = gb0; gb <= gb1; ++gb, ++kk) {
        const int tb = kk % cfg.t_bufs;
        mbar_wait(&meta.t_full[tb], (kk / cfg.t_bufs) & 1, abort, p.err);
        tc_fence_after();
        const uint32_t ta = smem_addr(t_base + (size_t)tb * 2 * cfg.t_part);
        for (int nt = tile_lo(gb); nt < tile_hi(gb); ++nt, ++ex_iter, ++acc_iter) {
          const int s = ex_iter % cfg.s_ex;
          mbar_wait(&meta.full_ex[s], (ex_iter / cfg.s_ex) & 1, abort, p.err);
          const int a = acc_iter & 1;
          if (acc_iter >= 2) mbar_wait(&meta.tempty[a], ((acc_iter >> 1) - 1) & 1, abort, p.err);
          tc_fence_after();
          const uint32_t ba = smem_addr(ex_base + (size_t)s * cfg.ex_stage);
          for (int part = 0; part < 2; ++part) {       // T_hi, then T_lo
            const uint32_t tp = ta + part * cfg.t_part;
            for (int ks = 0; ks < r_pad / 16; ++ks) {
              const int atom = ks * 16 / cfg.ka, within = (ks * 16 % cfg.ka) * 2;
              tc_mma_bf16(tmem + a * BS, make_sdesc(ba + atom * (kTileN * kb) + within, kb),
                          make_sdesc(tp + atom * (BS * kb) + within, kb), idesc, (part | ks) ? 1u : 0u);
            }
          }
          tc_commit(&meta.tfull[a]);
          tc_commit(&meta.empty_ex[s]);
        }
        tc_commit(&meta.t_empty[tb]);
      }
    }
    __syncwarp();
  } else {
    // ======================= epilogue warps 2..9
    // Two groups of four warps (h = 0: warps 2..5, h = 1: warps 6..9), one warp
    // per TMEM lane quarter each.  Both read the shrink accumulator; for the
    // expand, group h takes the tiles that land in accumulator h (every other
    // tile), so one group's TMEM loads overlap the other group's stores.
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int etid = tid - 64;
    const int gtid = etid & 127;             // thread index inside the group
    constexpr int kCR = BS < 32 ? BS : 32;   // rows per piece of a tile
    constexpr int kChunks = BS / kCR;
    constexpr int kStoreRows = BS / 8;       // rows a thread stores per tile
    uint32_t ex_iter = 0, acc_iter = 0;
    int kk = 0;
    for (int gb = gb0; gb <= gb1; ++gb, ++kk) {
      const BlockRef br = block_ref<BS>(p, meta, gb);
      const bool e_ok = br.e >= 0 && br.e < E;
      named_barrier(1, kEpiThreads);   // every epilogue thread is done with the previous block's epi_f
      if (etid < BS) {
        const int f = __ldg(br.ids + etid);
        int v = -1;
        if (f >= 0 && f < P && e_ok) v = f;
        else if (f < 0 || f > P) flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);
        meta.epi_f[etid] = v;
      }
      named_barrier(1, kEpiThreads);
      uint32_t valid[kChunks];   // bit i of valid[c]: row kCR*c + i is a real pair
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        valid[c] = 0;
#pragma unroll
        for (int i = 0; i < kCR; ++i) valid[c] |= (uint32_t)(meta.epi_f[kCR * c + i] >= 0) << i;
      }
      int st_f[kStoreRows];
#pragma unroll
      for (int i = 0; i < kStoreRows; ++i) st_f[i] = meta.epi_f[(gtid >> 4) + 8 * i];

      // -- shrink readout: T (fp32 in TMEM) -> T_hi, T_lo (bf16, swizzled) in buffer tb
      const int tb = kk % cfg.t_bufs;
      mbar_wait(&meta.shrink_done, kk & 1, abort, p.err);
      if (kk >= cfg.t_bufs) mbar_wait(&meta.t_empty[tb], ((kk / cfg.t_bufs) - 1) & 1, abort, p.err);
      tc_fence_after();
      uint8_t *thi = t_base + (size_t)tb * 2 * cfg.t_part;
      uint8_t *tlo = thi + cfg.t_part;
      if (32 * q < BS) {
        const int prow = 32 * q + lane;
        const bool rv = prow < BS && meta.epi_f[min(prow, BS - 1)] >= 0;
        const int half_groups = r_pad / 16;    // 8-column groups per warp of this quarter
        for (int g = h * half_groups; g < (h + 1) * half_groups; ++g) {
          float v[8];
          tmem_ld8(tmem_sh + ((uint32_t)(32 * q) << 16) + g * 8, v);
          tc_wait_ld();
          if (prow < BS) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float a0 = v[2 * i], a1 = v[2 * i + 1];
              const int j0 = g * 8 + 2 * i;
              if (!rv || j0 >= r) a0 = 0.f;
              if (!rv || j0 + 1 >= r) a1 = 0.f;
              const uint16_t h0 = float_to_bf16_bits(a0), h1 = float_to_bf16_bits(a1);
              const uint16_t l0 = float_to_bf16_bits(a0 - bf16_bits_to_float(h0));
              const uint16_t l1 = float_to_bf16_bits(a1 - bf16_bits_to_float(h1));
              hw[i] = (uint32_t)h0 | ((uint32_t)h1 << 16);
              lw[i] = (uint32_t)l0 | ((uint32_t)l1 << 16);
            }
            const int atom = g * 8 / cfg.ka, c = (g * 8 % cfg.ka) / 8;
            const uint32_t off = (uint32_t)atom * (BS * kb) + swz(prow, c, kb);
            *reinterpret_cast<uint4 *>(thi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(tlo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_cta();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&meta.t_full[tb]);
        mbar_arrive(&meta.shrink_free);
      }

      // -- expand epilogue: this group's tiles of the block
      for (int nt = tile_lo(gb); nt < tile_hi(gb); ++nt, ++ex_iter, ++acc_iter) {
        if ((int)(acc_iter & 1) != h) continue;
        const int s = ex_iter % cfg.s_ex;
        const int a = h;
        mbar_wait(&meta.tfull[a], (acc_iter >> 1) & 1, abort, p.err);
        tc_fence_after();
        mbar_wait(&meta.full_ex[s], (ex_iter / cfg.s_ex) & 1, abort, p.err);
        uint8_t *yt = ex_base + (size_t)s * cfg.ex_stage + cfg.yt_off;
        const int n0 = nt * kTileN;
        const int nl = 32 * q + lane;
        const bool col_ok = n0 + nl < N;
        uint16_t *col = reinterpret_cast<uint16_t *>(yt) + nl;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          float v[kCR];
#pragma unroll
          for (int c0 = 0; c0 < kCR; c0 += 8) {
            float w8[8];
            tmem_ld8(tmem + a * BS + ((uint32_t)(32 * q) << 16) + kCR * c + c0, w8);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[c0 + i] = w8[i];
          }
          tc_wait_ld();
          if (col_ok) {
            if (p.add_inputs) {
              uint16_t old[kCR];   // all loads first, then all stores
#pragma unroll
              for (int i = 0; i < kCR; ++i) old[i] = col[(kCR * c + i) * kTileN];
#pragma unroll
              for (int i = 0; i < kCR; ++i) v[i] += bf16_bits_to_float(old[i]);
            }
#pragma unroll
            for (int i = 0; i < kCR; ++i)
              if ((valid[c] >> i) & 1) col[(kCR * c + i) * kTileN] = float_to_bf16_bits(v[i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta.tempty[a]);
        named_barrier(2 + h, kEpiThreads / 2);
        {
          // write the finished rows back: thread takes 16-byte chunk (gtid % 16)
          // of rows gtid/16 + 8i
          const int c16 = gtid & 15;
          const int nn = n0 + c16 * 8;
          if (nn < N) {
            uint4 vals[kStoreRows];
#pragma unroll
            for (int i = 0; i < kStoreRows; ++i)
              vals[i] = *reinterpret_cast<const uint4 *>(yt + ((gtid >> 4) + 8 * i) * (kTileN * 2) + c16 * 16);
#pragma unroll
            for (int i = 0; i < kStoreRows; ++i)
              if (st_f[i] >= 0) *reinterpret_cast<uint4 *>(p.y + (size_t)st_f[i] * N + nn) = vals[i];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta.empty_ex[s]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, cfg.tmem_cols);
  }
}

// cuTensorMapEncodeTiled, fetched through the runtime so that the library
// does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

int encode_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
              CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return MOE_LORA_ERR_LAUNCH;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? 0 : MOE_LORA_ERR_LAUNCH;
}

int round_up(int v, int a) { return (v + a - 1) / a * a; }

int pick_cfg(const FusedArgs &f, const DeviceInfo &dev, TcCfg *cfg) {
  const int BS = f.block_size;
  const int r16 = round_up(f.rank, 16);
  cfg->r_pad = r16 <= 16 ? 16 : (r16 <= 32 ? 32 : (r16 <= 64 ? 64 : 128));
  cfg->ka = cfg->r_pad >= 64 ? 64 : cfg->r_pad;
  cfg->natoms = cfg->r_pad / cfg->ka;
  const int kb = cfg->ka * 2;
  cfg->kt_total = (f.K + kTileK - 1) / kTileK;
  cfg->nt_total = (f.N + kTileN - 1) / kTileN;
  // shrink stage: x tile (BS rows x 128 B), then the A tile (r_pad rows x 128 B)
  cfg->at_off = BS * 128;
  cfg->sh_stage = round_up(BS * 128 + cfg->r_pad * 128, 1024);
  // expand stage: B tile (natoms x 128 rows x kb), then the y tile (BS rows x 256 B)
  cfg->yt_off = round_up(cfg->natoms * kTileN * kb, 1024);
  cfg->ex_stage = round_up(cfg->yt_off + BS * kTileN * 2, 1024);
  cfg->t_part = round_up(cfg->natoms * BS * kb, 1024);
  const int meta_bytes = round_up((int)sizeof(TcMeta), 1024);
  const int budget = (int)dev.max_smem_optin;
  // Pick the plan with the most bytes in flight (shrink stages in flight are
  // 2 * (lag + 1): two producer warps, each up to `lag` stages ahead).
  int best = -1 << 30;
  TcCfg pick = *cfg;
  for (int s_sh = kMaxStages; s_sh >= 2; --s_sh) {
    const int lag = std::min(kMaxLag, (s_sh - 1) / 2);
    for (int s_ex = kMaxStages; s_ex >= 1; --s_ex) {
      for (int t_bufs = 2; t_bufs >= 1; --t_bufs) {
        const int after_sh = s_ex * cfg->ex_stage + t_bufs * 2 * cfg->t_part + meta_bytes;
        const int total = s_sh * cfg->sh_stage + after_sh;
        if (total > budget) continue;
        // the M=128 shrink MMA reads 128 x-tile rows: the rows past block_size
        // (never used) must still lie inside the allocation
        if (cfg->sh_stage + after_sh < 128 * 128) continue;
        const int sh_fly = std::min(s_sh, 2 * (lag + 1)) * cfg->sh_stage;
        const int score = std::min(sh_fly, 128 * 1024) + std::min(s_ex * cfg->ex_stage, 128 * 1024) +
                          (t_bufs == 2 ? 8 * 1024 : 0) - total / 64;
        if (score > best) {
          best = score;
          pick = *cfg;
          pick.s_sh = s_sh;
          pick.lag = lag;
          pick.s_ex = s_ex;
          pick.t_bufs = t_bufs;
          pick.off_sh = 0;
          pick.off_ex = s_sh * cfg->sh_stage;
          pick.off_t = pick.off_ex + s_ex * cfg->ex_stage;
          pick.off_meta = pick.off_t + t_bufs * 2 * cfg->t_part;
          pick.smem_bytes = total;
        }
      }
    }
  }
  if (best == (-1 << 30)) return MOE_LORA_ERR_UNSUPPORTED;
  *cfg = pick;
  int cols = 32;
  while (cols < 2 * BS + cfg->r_pad) cols <<= 1;
  cfg->tmem_cols = cols;
  // CTAs that share an SM share its 512 TMEM columns: ask for enough shared
  // memory that they never need more than that.
  const int per_sm = 228 * 1024;
  while ((per_sm / (cfg->smem_bytes + 1024)) * cols > 512) cfg->smem_bytes += 4096;
  if (cfg->smem_bytes > budget) return MOE_LORA_ERR_UNSUPPORTED;
  return 0;
}

template <int BS>
int launch_bs(const FusedArgs &f, const TcCfg &cfg, const CUtensorMap &ta, const CUtensorMap &tb, int G,
              cudaStream_t stream) {
  const void *fn = (const void *)fused_tcgen05_kernel<BS>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes) != cudaSuccess)
    return MOE_LORA_ERR_LAUNCH;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(G, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = cfg.smem_bytes;
  lc.stream = stream;
  // May start while the align kernel before it is finishing (it waits for it
  // with griddepcontrol.wait before touching the align outputs).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&lc, fused_tcgen05_kernel<BS>, ta, tb, f, cfg);
  return err == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

}  // namespace

bool tcgen05_path_supports(const FusedArgs &f) { return f.rank % 8 == 0 && f.num_active_loras <= kMaxSlots; }

int launch_fused_tcgen05(const FusedArgs &f, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  if (!tcgen05_path_supports(f)) return MOE_LORA_ERR_UNSUPPORTED;
  TcCfg cfg;
  if (int st = pick_cfg(f, dev, &cfg)) return st;
  CUtensorMap ta, tb;
  const uint64_t LE = (uint64_t)f.max_loras * f.num_experts;
  if (int st = encode_3d(&ta, f.lora_a, (uint64_t)f.K, (uint64_t)f.rank, LE, kTileK, (uint32_t)cfg.r_pad,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return st;
  const CUtensorMapSwizzle bsw = cfg.ka == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                              : (cfg.ka == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  if (int st = encode_3d(&tb, f.lora_b, (uint64_t)f.rank, (uint64_t)f.N, LE, (uint32_t)cfg.ka, kTileN, bsw))
    return st;
  const long long bound = fused_block_bound(f.M, f.topk, f.num_experts, f.num_active_loras, f.block_size);
  if (bound <= 0) return 0;
  const int per_sm = std::max(1, (228 * 1024) / (cfg.smem_bytes + 1024));
  long long G = (long long)dev.sm_count * per_sm;
  if (G > bound * cfg.nt_total) G = bound * cfg.nt_total;
  if (G < 1) G = 1;
  switch (f.block_size) {
    case 16: return launch_bs<16>(f, cfg, ta, tb, (int)G, stream);
    case 32: return launch_bs<32>(f, cfg, ta, tb, (int)G, stream);
    case 64: return launch_bs<64>(f, cfg, ta, tb, (int)G, stream);
    case 128: return launch_bs<128>(f, cfg, ta, tb, (int)G, stream);
    default: return MOE_LORA_ERR_UNSUPPORTED;
  }
}

}  // namespace moe_lora
