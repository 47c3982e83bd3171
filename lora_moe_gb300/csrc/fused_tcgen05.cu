// fused_tcgen05.cu -- the prefill-sized fused MoE-LoRA shrink+expand on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// Same definition as the CUDA-core path (prhub.com.cn summary of vLLM PR
// #42290, "Implementation breakdown" step 1: shrink by lora_a, expand by
// lora_b, rank dimension kept on chip, add_inputs accumulate/overwrite), per
// adapter slice s, with the pair's input row x_p (row m or row f) and router
// weight w_p (1 without weights):
//     T[p][j]   = sum_k x_p[k] * A_s[l][e][j][k]           p < block_size, j < r
//     y[f_p][off + s*N + n] = bf16((add ? y_in : 0) + w_p * sum_j B_s[l][e][n][j] * T[p][j])
//
// Work split.  The work of a call is the list of (unit, 128-column tile)
// pairs, a unit being one adapter slice of one block of a listed slot (vLLM
// PR #32005: the grid is sized by the active LoRAs).  The persistent CTAs split
// it either into equal shares of (unit, tile) pairs (a unit whose tiles
// straddle two CTAs has its shrink computed by both) or into whole units
// strided over the grid, whichever streams fewer bytes on the busiest CTA
// (stream_pipeline.cuh, cta_range).  T lives only in shared and tensor memory.
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
#include "stream_pipeline.cuh"

namespace moe_lora {

namespace {

constexpr int kWarps = 13;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kMmaRows = 128;     // M of every tcgen05.mma here

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
    fused_tcgen05_kernel(const __grid_constant__ stream::TmapSet maps, const FusedArgs p, const stream::Cfg cfg) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  stream::Meta &meta = *reinterpret_cast<stream::Meta *>(smem + cfg.off_meta);
  uint8_t *sh_base = smem + cfg.off_sh;
  uint8_t *ex_base = smem + cfg.off_ex;
  uint8_t *t_base = smem + cfg.off_t;
  const int N = p.N, E = p.num_experts, r = p.rank, r_pad = cfg.r_pad;
  const int P = p.M * p.topk;
  const int kt_total = cfg.kt_total;
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
      mbar_init(&meta.tempty[a], kEpiWarps / 2);       // accumulator a is drained by group a % 2
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&meta.t_full[a], kEpiWarps);
      mbar_init(&meta.t_empty[a], 1);
    }
    mbar_init(&meta.shrink_done, 1);
    mbar_init(&meta.shrink_free, kEpiWarps);
    meta.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < p.num_slices) {
    prefetch_tensor_map(&maps.a[lane]);
    prefetch_tensor_map(&maps.b[lane]);
  }
  if (warp == 1) {
    tmem_alloc(&meta.tmem_base, cfg.tmem_cols);
    tmem_relinquish();
  }
  wait_for_prior_grid();   // align outputs are read from here on
  stream::slot_prefix<BS>(p, meta);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = meta.tmem_base;
  const uint32_t tmem_sh = tmem + cfg.nacc * BS;   // shrink accumulator columns

  const stream::Range rg = stream::cta_range(meta, p.num_active_loras, p.num_slices, cfg);
  const int gb0 = rg.gb0, gb1 = rg.gb1;
  auto tile_lo = [&](int gb) { return rg.tile_lo(gb); };
  auto tile_hi = [&](int gb) { return rg.tile_hi(gb); };

  if (warp == 10 || warp == 11) {
    stream::shrink_producer<BS>(p, cfg, meta, &maps, sh_base, rg, warp - 10);
  } else if (warp == 12) {
    // ======================= shrink MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_bf16(kMmaRows, r_pad);
      uint32_t sh_iter = 0;
      int kk = 0;
      for (int gb = gb0; gb <= gb1; gb += rg.step, ++kk) {
        if (kk > 0) mbar_wait(&meta.shrink_free, (kk - 1) & 1, abort, p.err);
        tc_fence_after();
        for (int kt = 0; kt < kt_total; ++kt, ++sh_iter) {
          const int s = sh_iter % cfg.s_sh;
          mbar_wait(&meta.full_sh[s], (sh_iter / cfg.s_sh) & 1, abort, p.err);
          tc_fence_after();
          const uint32_t xa = smem_addr(sh_base + (size_t)s * cfg.sh_stage);
          const uint32_t aa = xa + cfg.at_off;
#pragma unroll
          for (int k16 = 0; k16 < stream::kTileK / 16; ++k16)
            tc_mma_bf16(tmem_sh, stream::make_sdesc(xa + k16 * 32, 128), stream::make_sdesc(aa + k16 * 32, 128), idesc,
                        (kt | k16) ? 1u : 0u);
          tc_commit(&meta.empty_sh[s]);
        }
        tc_commit(&meta.shrink_done);
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    stream::expand_producer<BS>(p, cfg, meta, &maps, ex_base, rg);
  } else if (warp == 1) {
    // ======================= expand MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_bf16(kMmaRows, BS);
      uint32_t ex_iter = 0, acc_iter = 0;
      int kk = 0;
      for (int gb = gb0; gb <= gb1; gb += rg.step, ++kk) {
        const int tb = kk % cfg.t_bufs;
        mbar_wait(&meta.t_full[tb], (kk / cfg.t_bufs) & 1, abort, p.err);
        tc_fence_after();
        const uint32_t ta = smem_addr(t_base + (size_t)tb * 2 * cfg.t_part);
        for (int nt = tile_lo(gb); nt < tile_hi(gb); ++nt, ++ex_iter, ++acc_iter) {
          const int s = ex_iter % cfg.s_ex;
          mbar_wait(&meta.full_ex[s], (ex_iter / cfg.s_ex) & 1, abort, p.err);
          const int a = acc_iter % cfg.nacc;
          if (acc_iter >= (uint32_t)cfg.nacc) mbar_wait(&meta.tempty[a], ((acc_iter / cfg.nacc) - 1) & 1, abort, p.err);
          tc_fence_after();
          const uint32_t ba = smem_addr(ex_base + (size_t)s * cfg.ex_stage);
          for (int part = 0; part < 2; ++part) {       // T_hi, then T_lo
            const uint32_t tp = ta + part * cfg.t_part;
            for (int ks = 0; ks < r_pad / 16; ++ks) {
              const int atom = ks * 16 / cfg.ka, within = (ks * 16 % cfg.ka) * 2;
              tc_mma_bf16(tmem + a * BS, stream::make_sdesc(ba + atom * (stream::kTileN * kb) + within, kb),
                          stream::make_sdesc(tp + atom * (BS * kb) + within, kb), idesc, (part | ks) ? 1u : 0u);
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
    // rows per piece of a tile: 16 keeps the live values per thread low
    // enough that the epilogue's schedule does not depend on small changes
    // elsewhere in the kernel (32-row pieces ran 10-15% slower after an
    // unrelated change to the argument block)
    constexpr int kCR = BS < 16 ? BS : 16;
    constexpr int kChunks = BS / kCR;
    constexpr int kStoreRows = BS / 8;       // rows a thread stores per tile
    uint32_t ex_iter = 0, acc_iter = 0;
    int kk = 0;
    for (int gb = gb0; gb <= gb1; gb += rg.step, ++kk) {
      const stream::BlockRef br = stream::block_ref<BS>(p, meta, gb);
      const bool e_ok = br.e >= 0 && br.e < E;
      named_barrier(1, kEpiThreads);   // every epilogue thread is done with the previous block's epi_f
      if (etid < BS) {
        const int f = __ldg(br.ids + etid);
        int v = -1;
        if (f >= 0 && f < P && e_ok) v = f;
        else if ((f < 0 || f > P) && br.s == 0) flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);
        meta.epi_f[etid] = v;
        meta.epi_w[etid] = v >= 0 ? route_weight(p, v) : 0.f;
      }
      named_barrier(1, kEpiThreads);
      uint32_t valid[kChunks];   // bit i of valid[c]: row kCR*c + i is a real pair
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        valid[c] = 0;
#pragma unroll
        for (int i = 0; i < kCR; ++i) valid[c] |= (uint32_t)(meta.epi_f[kCR * c + i] >= 0) << i;
      }
      const bool weighted = p.topk_weights != nullptr;
      const size_t s_col = (size_t)p.y_offset + (size_t)br.s * N;   // the slice's first output column
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
            const uint32_t off = (uint32_t)atom * (BS * kb) + stream::swz(prow, c, kb);
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
        const int a = acc_iter % cfg.nacc;
        mbar_wait(&meta.tfull[a], (acc_iter / cfg.nacc) & 1, abort, p.err);
        tc_fence_after();
        mbar_wait(&meta.full_ex[s], (ex_iter / cfg.s_ex) & 1, abort, p.err);
        uint8_t *yt = ex_base + (size_t)s * cfg.ex_stage + cfg.yt_off;
        const int n0 = nt * stream::kTileN;
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
            if (weighted) {
#pragma unroll
              for (int i = 0; i < kCR; ++i) v[i] *= meta.epi_w[kCR * c + i];
            }
            if (p.add_inputs) {
              uint16_t old[kCR];   // all loads first, then all stores
#pragma unroll
              for (int i = 0; i < kCR; ++i) old[i] = col[(kCR * c + i) * stream::kTileN];
#pragma unroll
              for (int i = 0; i < kCR; ++i) v[i] += bf16_bits_to_float(old[i]);
            }
#pragma unroll
            for (int i = 0; i < kCR; ++i)
              if ((valid[c] >> i) & 1) col[(kCR * c + i) * stream::kTileN] = float_to_bf16_bits(v[i]);
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
              vals[i] = *reinterpret_cast<const uint4 *>(yt + ((gtid >> 4) + 8 * i) * (stream::kTileN * 2) + c16 * 16);
#pragma unroll
            for (int i = 0; i < kStoreRows; ++i)
              if (st_f[i] >= 0) *reinterpret_cast<uint4 *>(p.y + (size_t)st_f[i] * p.ldy + s_col + nn) = vals[i];
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

template <int BS>
int launch_bs(const FusedArgs &f, const stream::Cfg &cfg, const stream::TmapSet &maps, int G,
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
  const cudaError_t err = cudaLaunchKernelEx(&lc, fused_tcgen05_kernel<BS>, maps, f, cfg);
  return err == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

}  // namespace

bool tcgen05_path_supports(const FusedArgs &f) { return f.rank % 8 == 0 && f.num_active_loras <= stream::kMaxSlots; }

namespace {

// Ring depths, TMEM columns, shared memory and grid of one call.
int configure(const FusedArgs &f, const DeviceInfo &dev, stream::Cfg *out, long long *grid) {
  if (!tcgen05_path_supports(f)) return MOE_LORA_ERR_UNSUPPORTED;
  stream::Cfg cfg;
  // consumer region per T buffer: T_hi and T_lo tiles (bf16, swizzled)
  {
    const int r16 = (f.rank + 15) / 16 * 16;
    const int r_pad = r16 <= 16 ? 16 : (r16 <= 32 ? 32 : (r16 <= 64 ? 64 : 128));
    const int ka = r_pad >= 64 ? 64 : r_pad;
    const int part = ((r_pad / ka) * f.block_size * ka * 2 + 1023) / 1024 * 1024;
    if (int st = stream::plan(f, dev, 2 * part, 2, &cfg)) return st;
    cfg.t_part = part;   // the kernel addresses T buffers as [t_bufs][hi, lo] of one part each
  }
  cfg.nacc = 2;   // Meta holds barriers for two expand accumulators
  int cols = 32;
  while (cols < cfg.nacc * f.block_size + cfg.r_pad) cols <<= 1;
  cfg.tmem_cols = cols;
  // CTAs that share an SM share its 512 TMEM columns: ask for enough shared
  // memory that they never need more than that.
  while (((228 * 1024) / (cfg.smem_bytes + 1024)) * cols > 512) cfg.smem_bytes += 4096;
  if (cfg.smem_bytes > (int)dev.max_smem_optin) return MOE_LORA_ERR_UNSUPPORTED;
  const long long bound = fused_block_bound(f.M, f.topk, f.num_experts, f.num_active_loras, f.block_size);
  const int per_sm = std::max(1, (228 * 1024) / (cfg.smem_bytes + 1024));
  long long G = (long long)dev.sm_count * per_sm;
  if (G > bound * f.num_slices * cfg.nt_total) G = bound * f.num_slices * cfg.nt_total;
  *out = cfg;
  *grid = bound <= 0 ? 0 : std::max(1LL, G);
  return 0;
}

}  // namespace

int plan_fused_tcgen05(const FusedArgs &f, const DeviceInfo &dev, FusedPlan *out) {
  stream::Cfg cfg;
  long long G = 0;
  if (int st = configure(f, dev, &cfg, &G)) return st;
  out->kernel = MOE_LORA_PATH_TCGEN05;
  out->grid = (int)G;
  out->threads = kThreads;
  out->smem_bytes = cfg.smem_bytes;
  out->s_sh = cfg.s_sh;
  out->lag = cfg.lag;
  out->s_ex = cfg.s_ex;
  out->t_bufs = cfg.t_bufs;
  out->tmem_cols = cfg.tmem_cols;
  out->cluster = 1;
  out->pairs_per_group = f.block_size;
  return 0;
}

int launch_fused_tcgen05(const FusedArgs &f, cudaStream_t stream_) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  stream::Cfg cfg;
  long long G = 0;
  if (int st = configure(f, dev, &cfg, &G)) return st;
  if (G <= 0) return 0;
  stream::TmapSet maps;
  if (int st = stream::make_tensor_maps(f, cfg, &maps)) return st;
  switch (f.block_size) {
    case 16: return launch_bs<16>(f, cfg, maps, (int)G, stream_);
    case 32: return launch_bs<32>(f, cfg, maps, (int)G, stream_);
    case 64: return launch_bs<64>(f, cfg, maps, (int)G, stream_);
    case 128: return launch_bs<128>(f, cfg, maps, (int)G, stream_);
    default: return MOE_LORA_ERR_UNSUPPORTED;
  }
}

}  // namespace moe_lora
