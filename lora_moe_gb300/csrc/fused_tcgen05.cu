// fused_tcgen05.cu -- the prefill-sized fused MoE-LoRA shrink+expand on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// Same definition as the CUDA-core path (prhub.com.cn summary of vLLM PR
// #42290, "Implementation breakdown" step 1: shrink by lora_a, expand by
// lora_b, rank dimension kept on chip, add_inputs accumulate/overwrite):
//     T[p][j] = sum_k x[m_p][k] * A[l][e][j][k]       p < block_size, j < r
//     y[f_p][n] = bf16((add ? y[f_p][n] : 0) + sum_j B[l][e][n][j] * T[p][j])
//
// One work item is one (slot, block) of the align output.  A thread-block
// cluster of C CTAs shares it: CTA c runs the shrink over K-slice c, the C
// partial T's (fp32, block_size x r) are reduce-scattered through distributed
// shared memory (summed in rank order, so the result is deterministic), every
// CTA receives the full T, and CTA c then produces the N-slice c of the block's
// y rows.  T never reaches global memory.  The expand MMA takes bf16 operands,
// so T is passed as two bf16 tiles, T_hi = bf16(T) and T_lo = bf16(T - T_hi),
// and the expand runs over both (the B tile is read twice): the product then
// carries T to about 16 significant bits instead of 8, which keeps the
// result within the fp32 path's error.
//
// Warp roles (320 threads):
//   warp 0      producer: gathers the block's x rows with 16-byte cp.async into
//               128-byte-swizzled K-major tiles, TMA-loads A / B tiles
//               (cp.async.bulk.tensor, 3-D tensor maps, OOB zero fill) and
//               bulk-copies the y rows of each N tile.
//   warp 1      owns tensor memory and issues tcgen05.mma (one thread):
//               shrink  D[128 x r_pad]  = Xtile[128 x 64]  * Atile[r_pad x 64]^T   (K loop)
//               expand  D[128 x bs]     = Btile[128 x r_pad] * T[bs x r_pad]^T    per 128 output columns
//               (the expand puts output columns on the 128 TMEM lanes so that all
//               four lane quarters carry data whatever the block size).
//   warps 2..9  epilogue: read accumulators with tcgen05.ld, reduce T across the
//               cluster, add y_in, round to bf16, bulk-store y rows.
// Stages are tracked with mbarriers; every wait is bounded.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace moe_lora {

namespace {

constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kMaxSlots = 512;
constexpr int kTileK = 64;        // shrink K per stage (one 128-byte swizzle row)
constexpr int kTileN = 128;       // expand output columns per tile (TMEM lanes)
constexpr int kMmaRows = 128;     // M of every tcgen05.mma here

struct TcCfg {
  int C;
  int r_pad;          // rank rounded up to 16
  int natoms;         // ceil(r_pad / 64): 128-byte K atoms of the B tile and of T
  int s_sh, s_ex;     // pipeline depth of shrink / expand stages
  int tmem_cols;
  // byte offsets from the 1024-aligned smem base
  int off_sh, sh_stage_bytes, at_offset;   // shrink stage: x tile (block_size rows), then A tile
  int lag;            // x-gather stages in flight before a stage is released (< s_sh)
  int off_ex, ex_stage_bytes, yt_offset;   // expand stage: B tile, then y tile at +yt_offset
  int off_t;          // T_hi then T_lo tiles (bf16, swizzled, natoms x bs rows x 128 B each)
  int t_bytes;        // bytes of one T tile
  int tp_pitch;       // floats per row of the fp32 partial T (aliases the shrink stages)
  int off_meta;
  int smem_bytes;     // including alignment slack
};

struct TcMeta {
  uint64_t full_sh[4], empty_sh[4];
  uint64_t full_ex[4], empty_ex[4];
  uint64_t tfull[2], tempty[2];
  uint64_t shrink_done;
  uint32_t tmem_base;
  int abort;
  int slot_l[kMaxSlots];
  int prefix[kMaxSlots + 1];
  int epi_f[128];     // the current block's pair ids for the epilogue warps (-1 = padding)
  int prod_f[128];    // the same for the producer warp (it may run one block ahead)
};

__device__ __forceinline__ int find_slot(const int *prefix, int nact, int item) {
  int lo = 0, hi = nact;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid;
  }
  return lo;
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
    fused_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const FusedArgs p, const TcCfg cfg) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcMeta &meta = *reinterpret_cast<TcMeta *>(smem + cfg.off_meta);
  uint8_t *sh_base = smem + cfg.off_sh;
  uint8_t *ex_base = smem + cfg.off_ex;
  uint8_t *t_tile = smem + cfg.off_t;
  float *tpart = reinterpret_cast<float *>(sh_base);

  cg::cluster_group cluster = cg::this_cluster();
  const int C = cfg.C;
  const int c = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K, N = p.N, E = p.num_experts, r = p.rank, r_pad = cfg.r_pad;
  const int P = p.M * p.topk;
  volatile int *abort = &meta.abort;

  if (tid == 0) {
    for (int s = 0; s < cfg.s_sh; ++s) {
      mbar_init(&meta.full_sh[s], 1 + 32);
      mbar_init(&meta.empty_sh[s], 1);
    }
    for (int s = 0; s < cfg.s_ex; ++s) {
      mbar_init(&meta.full_ex[s], 1 + 32);              // B tile (tx) + 32 lanes' y_in copies
      mbar_init(&meta.empty_ex[s], 1 + kEpiThreads / 32); // MMA commit + epilogue warps
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&meta.tfull[a], 1);
      mbar_init(&meta.tempty[a], kEpiThreads / 32);
    }
    mbar_init(&meta.shrink_done, 1);
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
      if (c == 0 && blockIdx.y == 0) flag_error(p.err, MOE_LORA_DEVERR_LORA_ID);
    } else if (!p.adapter_enabled || __ldg(p.adapter_enabled + l) != 0) {
      nb = __ldg(p.num_tokens_post_padded + l) / BS;
      nb = max(0, min(nb, p.max_num_m_blocks));
    }
    meta.slot_l[z] = l;
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
  const int total_blocks = meta.prefix[p.num_active_loras];

  const int kt_total = (K + kTileK - 1) / kTileK;
  const int kt0 = c * kt_total / C, kt1 = (c + 1) * kt_total / C;
  const int nt_total = (N + kTileN - 1) / kTileN;
  const int nt0 = c * nt_total / C, nt1 = (c + 1) * nt_total / C;

  uint32_t sh_iter = 0, ex_iter = 0, acc_iter = 0, item_iter = 0;

  for (int item = blockIdx.y; item < total_blocks; item += gridDim.y, ++item_iter) {
    const int z = find_slot(meta.prefix, p.num_active_loras, item);
    const int l = meta.slot_l[z];
    const int b = item - meta.prefix[z];
    const int e = __ldg(p.expert_ids + (size_t)l * p.max_num_m_blocks + b);
    if (e < 0 || e >= E) {   // the same for every CTA of the cluster
      if (tid == 0 && c == 0) flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
      --item_iter;
      continue;
    }
    const int32_t *ids = p.sorted_token_ids + (size_t)l * p.max_num_tokens_padded + (size_t)b * BS;
    const int le = l * E + e;

    // ======================= shrink: partial T over this CTA's K-slice
    if (warp == 0) {
      for (int pr = lane; pr < BS; pr += 32) {
        const int f = __ldg(ids + pr);
        meta.prod_f[pr] = (f >= 0 && f < P) ? f : -1;
      }
      __syncwarp();
      // This lane gathers 16-byte chunk (lane % 8) of rows lane/8 + 4i.
      constexpr int kRowsPerLane = BS / 4;
      const int ch = lane & 7;
      int xrow[kRowsPerLane];
#pragma unroll
      for (int i = 0; i < kRowsPerLane; ++i) {
        const int pr = (lane >> 3) + 4 * i;
        const int f = __ldg(ids + pr);
        xrow[i] = (f >= 0 && f < P) ? f / p.topk : -1;
      }
      int issued = 0;
      for (int kt = kt0; kt < kt1; ++kt, ++sh_iter, ++issued) {
        const int s = sh_iter % cfg.s_sh;
        const uint32_t n = sh_iter / cfg.s_sh;
        if (sh_iter >= (uint32_t)cfg.s_sh) mbar_wait(&meta.empty_sh[s], (n - 1) & 1, abort, p.err);
        uint8_t *xt = sh_base + (size_t)s * cfg.sh_stage_bytes;
        uint8_t *at = xt + cfg.at_offset;
        if (lane == 0) {
          mbar_arrive_expect_tx(&meta.full_sh[s], (uint32_t)r_pad * 128);
          tma_load_3d(at, &tmap_a, kt * kTileK, 0, le, &meta.full_sh[s]);
        }
        const int k = kt * kTileK + ch * 8;
#pragma unroll
        for (int i = 0; i < kRowsPerLane; ++i) {
          const int pr = (lane >> 3) + 4 * i;
          const bool ok = xrow[i] >= 0 && k < K;
          const uint16_t *src = ok ? p.x + (size_t)xrow[i] * K + k : p.x;
          cp_async_16(xt + pr * 128 + ((ch ^ (pr & 7)) << 4), src, ok ? 16u : 0u);
        }
        cp_async_commit();
        if (issued >= cfg.lag) {
          if (cfg.lag == 1) cp_async_wait_group<1>(); else cp_async_wait_group<2>();
          fence_proxy_async_cta();
          mbar_arrive(&meta.full_sh[(sh_iter - cfg.lag) % cfg.s_sh]);
        }
      }
      cp_async_wait_group<0>();
      fence_proxy_async_cta();
      const int tail = issued < cfg.lag ? issued : cfg.lag;
      for (int i = tail; i > 0; --i) mbar_arrive(&meta.full_sh[(sh_iter - i) % cfg.s_sh]);
    } else if (warp == 1) {
      if (lane == 0) {
        const uint32_t idesc = make_idesc_bf16(kMmaRows, r_pad);
        uint32_t first = 1;
        for (int kt = kt0; kt < kt1; ++kt) {
          const int s = sh_iter % cfg.s_sh;
          mbar_wait(&meta.full_sh[s], (sh_iter / cfg.s_sh) & 1, abort, p.err);
          tc_fence_after();
          const uint32_t xa = smem_addr(sh_base + (size_t)s * cfg.sh_stage_bytes);
          const uint32_t aa = xa + cfg.at_offset;
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk) {
            tc_mma_bf16(tmem_sh, make_sdesc_sw128(xa + kk * 32), make_sdesc_sw128(aa + kk * 32), idesc,
                        first ? 0u : 1u);
            first = 0;
          }
          tc_commit(&meta.empty_sh[s]);
          ++sh_iter;
        }
        tc_commit(&meta.shrink_done);
      } else {
        sh_iter += kt1 - kt0;
      }
      __syncwarp();
    } else {
      // epilogue warps: remember this block's pairs, read the partial T.
      const int etid = tid - 64;
      if (etid < BS) {
        const int f = __ldg(ids + etid);
        int v = -1;
        if (f >= 0 && f < P) v = f;
        else if (f != P && c == 0) flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);
        meta.epi_f[etid] = v;
      }
      mbar_wait(&meta.shrink_done, item_iter & 1, abort, p.err);
      tc_fence_after();
      const int q = warp & 3, h = (warp - 2) >> 2;
      if (32 * q < BS) {
        const int prow = 32 * q + lane;
        const int half = r_pad / 2;
        for (int c0 = h * half; c0 < (h + 1) * half; c0 += 8) {
          float v[8];
          tmem_ld8(tmem_sh + ((uint32_t)(32 * q) << 16) + c0, v);
          tc_wait_ld();
          if (prow < BS) {
            float4 *dst = reinterpret_cast<float4 *>(tpart + (size_t)prow * cfg.tp_pitch + c0);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
          }
        }
      }
      tc_fence_before();
    }

    // ======================= reduce-scatter T across the cluster
    cluster.sync();
    if (warp >= 2) {
      const int etid = tid - 64;
      const int p0 = c * BS / C, p1 = (c + 1) * BS / C;
      const int halfr = r_pad / 2;
      for (int idx = etid; idx < (p1 - p0) * halfr; idx += kEpiThreads) {
        const int pr = p0 + idx / halfr;
        const int j = 2 * (idx % halfr);
        float s0 = 0.f, s1 = 0.f;
        for (int q = 0; q < C; ++q) {
          const float2 v = *reinterpret_cast<const float2 *>(
              cluster.map_shared_rank(tpart + (size_t)pr * cfg.tp_pitch + j, q));
          s0 += v.x;
          s1 += v.y;
        }
        const bool valid = meta.epi_f[pr] >= 0;
        if (!valid || j >= r) s0 = 0.f;
        if (!valid || j + 1 >= r) s1 = 0.f;
        const uint16_t h0 = float_to_bf16_bits(s0), h1 = float_to_bf16_bits(s1);
        const uint16_t l0 = float_to_bf16_bits(s0 - bf16_bits_to_float(h0));
        const uint16_t l1 = float_to_bf16_bits(s1 - bf16_bits_to_float(h1));
        const uint32_t hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
        const uint32_t lo = (uint32_t)l0 | ((uint32_t)l1 << 16);
        const int jj = j & 63;
        const size_t off = (size_t)(j >> 6) * (BS * 128) + (size_t)pr * 128 +
                           ((((jj >> 3) ^ (pr & 7)) << 4)) + (jj & 7) * 2;
        for (int q = 0; q < C; ++q) {
          *reinterpret_cast<uint32_t *>(cluster.map_shared_rank(t_tile + off, q)) = hi;
          *reinterpret_cast<uint32_t *>(cluster.map_shared_rank(t_tile + cfg.t_bytes + off, q)) = lo;
        }
      }
      fence_proxy_async_cluster();
    }
    cluster.sync();

    // ======================= expand: y rows of this CTA's N-slice
    if (warp == 0) {
      for (int nt = nt0; nt < nt1; ++nt, ++ex_iter) {
        const int s = ex_iter % cfg.s_ex;
        const uint32_t n = ex_iter / cfg.s_ex;
        if (ex_iter >= (uint32_t)cfg.s_ex) mbar_wait(&meta.empty_ex[s], (n - 1) & 1, abort, p.err);
        uint8_t *bt = ex_base + (size_t)s * cfg.ex_stage_bytes;
        uint8_t *yt = bt + cfg.yt_offset;
        const int n0 = nt * kTileN;
        if (lane == 0) {
          mbar_arrive_expect_tx(&meta.full_ex[s], (uint32_t)cfg.natoms * kTileN * 128);
          for (int a = 0; a < cfg.natoms; ++a)
            tma_load_3d(bt + a * (kTileN * 128), &tmap_b, a * 64, n0, le, &meta.full_ex[s]);
        }
        // y_in rows: 16-byte chunks through the load/store unit (row pieces are
        // too small for TMA to pay off); lane handles chunk (lane % 16) of rows
        // lane/16 + 2i.
        if (p.add_inputs) {
          const int ch = lane & 15;
          const int n = n0 + ch * 8;
          if (n < N)
            for (int pr = lane >> 4; pr < BS; pr += 2) {
              const int f = meta.prod_f[pr];
              if (f >= 0) cp_async_16(yt + pr * (kTileN * 2) + ch * 16, p.y + (size_t)f * N + n, 16u);
            }
        }
        cp_async_mbar_arrive_noinc(&meta.full_ex[s]);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        const uint32_t idesc = make_idesc_bf16(kMmaRows, BS);
        const uint32_t ta = smem_addr(t_tile);
        fence_proxy_async_cta();
        for (int nt = nt0; nt < nt1; ++nt) {
          const int s = ex_iter % cfg.s_ex;
          mbar_wait(&meta.full_ex[s], (ex_iter / cfg.s_ex) & 1, abort, p.err);
          const int a = acc_iter & 1;
          if (acc_iter >= 2) mbar_wait(&meta.tempty[a], ((acc_iter >> 1) - 1) & 1, abort, p.err);
          tc_fence_after();
          const uint32_t ba = smem_addr(ex_base + (size_t)s * cfg.ex_stage_bytes);
          for (int part = 0; part < 2; ++part) {          // T_hi, then T_lo
            const uint32_t tp = ta + part * cfg.t_bytes;
            for (int ks = 0; ks < r_pad / 16; ++ks) {
              const uint32_t atom = ks >> 2, within = (ks & 3) * 32;
              tc_mma_bf16(tmem + a * BS, make_sdesc_sw128(ba + atom * (kTileN * 128) + within),
                          make_sdesc_sw128(tp + atom * (BS * 128) + within), idesc,
                          (part | ks) ? 1u : 0u);
            }
          }
          tc_commit(&meta.tfull[a]);
          tc_commit(&meta.empty_ex[s]);
          ++ex_iter;
          ++acc_iter;
        }
      } else {
        ex_iter += nt1 - nt0;
        acc_iter += nt1 - nt0;
      }
      __syncwarp();
    } else {
      const int q = warp & 3, h = (warp - 2) >> 2;
      const int nl = 32 * q + lane;            // column inside the tile
      constexpr int kHalf = BS / 2;
      for (int nt = nt0; nt < nt1; ++nt, ++ex_iter, ++acc_iter) {
        const int s = ex_iter % cfg.s_ex;
        const int a = acc_iter & 1;
        mbar_wait(&meta.tfull[a], (acc_iter >> 1) & 1, abort, p.err);
        tc_fence_after();
        float v[kHalf];
#pragma unroll
        for (int c0 = 0; c0 < kHalf; c0 += 8) {
          float w[8];
          tmem_ld8(tmem + a * BS + ((uint32_t)(32 * q) << 16) + h * kHalf + c0, w);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[c0 + i] = w[i];
        }
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta.tempty[a]);
        mbar_wait(&meta.full_ex[s], (ex_iter / cfg.s_ex) & 1, abort, p.err);
        uint8_t *yt = ex_base + (size_t)s * cfg.ex_stage_bytes + cfg.yt_offset;
        const int n0 = nt * kTileN;
        if (n0 + nl < N) {
#pragma unroll
          for (int i = 0; i < kHalf; ++i) {
            const int pr = h * kHalf + i;
            if (meta.epi_f[pr] >= 0) {
              uint16_t *dst = reinterpret_cast<uint16_t *>(yt + pr * (kTileN * 2)) + nl;
              const float old = p.add_inputs ? bf16_bits_to_float(*dst) : 0.f;
              *dst = float_to_bf16_bits(v[i] + old);
            }
          }
        }
        named_barrier(1, kEpiThreads);
        // Write the finished rows back with 16-byte stores: thread handles chunk
        // (etid % 16) of rows etid/16 + 16i.
        {
          const int etid = tid - 64;
          const int ch = etid & 15;
          const int n = n0 + ch * 8;
          if (n < N)
            for (int pr = etid >> 4; pr < BS; pr += kEpiThreads / 16) {
              const int f = meta.epi_f[pr];
              if (f >= 0)
                *reinterpret_cast<uint4 *>(p.y + (size_t)f * N + n) =
                    *reinterpret_cast<const uint4 *>(yt + pr * (kTileN * 2) + ch * 16);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta.empty_ex[s]);
      }
      // the next item rewrites epi_f only after every epilogue warp is done with it
      named_barrier(1, kEpiThreads);
    }
  }

  // Release tensor memory.
  tc_fence_before();
  __syncthreads();
  if (C > 1) cluster.sync();
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

int encode_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return MOE_LORA_ERR_LAUNCH;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? 0 : MOE_LORA_ERR_LAUNCH;
}

int pick_cfg(const FusedArgs &f, const DeviceInfo &dev, TcCfg *cfg) {
  const int BS = f.block_size;
  cfg->r_pad = (f.rank + 15) / 16 * 16;
  cfg->natoms = (cfg->r_pad + 63) / 64;
  const int kt_total = (f.K + kTileK - 1) / kTileK;
  const int nt_total = (f.N + kTileN - 1) / kTileN;
  int C = 8;
  if (C > kt_total) C = kt_total;
  if (C > nt_total) C = nt_total;
  if (C > BS) C = BS;
  if (C < 1) C = 1;
  cfg->C = C;
  // Shrink stage: the x tile holds block_size rows; the M=128 MMA also reads
  // the 128 - block_size rows after them (the A tile, or the next region),
  // whose products land in accumulator rows nobody reads.
  const int at_bytes = cfg->r_pad * 128;
  cfg->at_offset = BS * 128;
  cfg->sh_stage_bytes = (BS * 128 + at_bytes + 1023) / 1024 * 1024;
  cfg->yt_offset = cfg->natoms * kTileN * 128;
  cfg->ex_stage_bytes = (cfg->yt_offset + BS * kTileN * 2 + 1023) / 1024 * 1024;
  cfg->t_bytes = cfg->natoms * BS * 128;
  const int meta_bytes = (int)((sizeof(TcMeta) + 1023) / 1024 * 1024);
  const int budget = (int)dev.max_smem_optin - 1024;  // alignment slack
  static const int plans[][2] = {{4, 4}, {3, 4}, {3, 3}, {4, 2}, {3, 2}, {2, 2}, {3, 1}, {2, 1}};
  for (int pitch_pad = 4; pitch_pad >= 0; pitch_pad -= 4) {
    cfg->tp_pitch = cfg->r_pad + pitch_pad;   // +4 floats staggers rows across banks
    const int tpart_bytes = BS * cfg->tp_pitch * 4;
    for (const auto &pl : plans) {
      const int s_sh = pl[0], s_ex = pl[1];
      int sh_region = s_sh * cfg->sh_stage_bytes;
      if (sh_region < tpart_bytes) sh_region = (tpart_bytes + 1023) / 1024 * 1024;
      // (the last x tile's over-read, at most (128 - block_size) rows, stays
      // inside the expand stages that follow the shrink region)
      const int total = sh_region + s_ex * cfg->ex_stage_bytes + 2 * cfg->t_bytes + meta_bytes;
      if (total > budget) continue;
      cfg->s_sh = s_sh;
      cfg->s_ex = s_ex;
      cfg->lag = s_sh - 1 < 2 ? s_sh - 1 : 2;
      cfg->off_sh = 0;
      cfg->off_ex = sh_region;
      cfg->off_t = sh_region + s_ex * cfg->ex_stage_bytes;
      cfg->off_meta = cfg->off_t + 2 * cfg->t_bytes;
      cfg->smem_bytes = total + 1024;
      int cols = 32;
      while (cols < 2 * BS + cfg->r_pad) cols <<= 1;
      cfg->tmem_cols = cols;
      // CTAs that share an SM share its 512 TMEM columns: ask for enough shared
      // memory that they never need more (an allocation that cannot be met
      // would wait for a CTA that may itself wait on this one's cluster).
      const int per_sm = 228 * 1024;
      while ((per_sm / (cfg->smem_bytes + 1024)) * cols > 512) cfg->smem_bytes += 4096;
      if (cfg->smem_bytes > (int)dev.max_smem_optin) return MOE_LORA_ERR_UNSUPPORTED;
      return 0;
    }
  }
  return MOE_LORA_ERR_UNSUPPORTED;
}

template <int BS>
int launch_bs(const FusedArgs &f, const TcCfg &cfg, const CUtensorMap &ta, const CUtensorMap &tb, int G,
              cudaStream_t stream) {
  const void *fn = (const void *)fused_tcgen05_kernel<BS>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes) != cudaSuccess)
    return MOE_LORA_ERR_LAUNCH;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(cfg.C, G, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = cfg.smem_bytes;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cfg.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // May start while the align kernel before it is finishing (it waits for it
  // with griddepcontrol.wait before touching the align outputs).
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  const cudaError_t err = cudaLaunchKernelEx(&lc, fused_tcgen05_kernel<BS>, ta, tb, f, cfg);
  return err == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

}  // namespace

int launch_fused_tcgen05(const FusedArgs &f, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  if (f.num_active_loras > kMaxSlots) return MOE_LORA_ERR_UNSUPPORTED;
  if (f.rank % 8 != 0) return MOE_LORA_ERR_UNSUPPORTED;
  TcCfg cfg;
  if (int st = pick_cfg(f, dev, &cfg)) return st;
  CUtensorMap ta, tb;
  const uint64_t LE = (uint64_t)f.max_loras * f.num_experts;
  if (int st = encode_3d(&ta, f.lora_a, (uint64_t)f.K, (uint64_t)f.rank, LE, kTileK, (uint32_t)cfg.r_pad)) return st;
  if (int st = encode_3d(&tb, f.lora_b, (uint64_t)f.rank, (uint64_t)f.N, LE, 64, kTileN)) return st;
  const long long bound = fused_block_bound(f.M, f.topk, f.num_experts, f.num_active_loras, f.block_size);
  if (bound <= 0) return 0;
  long long G = dev.sm_count / cfg.C;   // one CTA per SM (shared memory use keeps it so)
  if (G < 1) G = 1;
  if (G > bound) G = bound;
  switch (f.block_size) {
    case 16: return launch_bs<16>(f, cfg, ta, tb, (int)G, stream);
    case 32: return launch_bs<32>(f, cfg, ta, tb, (int)G, stream);
    case 64: return launch_bs<64>(f, cfg, ta, tb, (int)G, stream);
    case 128: return launch_bs<128>(f, cfg, ta, tb, (int)G, stream);
    default: return MOE_LORA_ERR_UNSUPPORTED;
  }
}

}  // namespace moe_lora
