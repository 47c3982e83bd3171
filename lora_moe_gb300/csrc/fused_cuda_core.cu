// fused_cuda_core.cu -- the decode-sized fused MoE-LoRA shrink+expand on CUDA
// cores (sm_103a).
//
// Computes, for every block b of every active slot z (l = lora_ids[z],
// e = expert_ids[l][b]) and every pair f of that block (m = f / topk):
//     t[j]    = sum_k x[m][k] * A[l][e][j][k]                 (fp32)
//     y[f][n] = bf16((add_inputs ? y[f][n] : 0) + sum_j B[l][e][n][j] * t[j])
// (prhub.com.cn summary of vLLM PR #42290, "Implementation breakdown" step 1:
// one kernel does the shrink by lora_a and the expand by lora_b and keeps the
// rank dimension on chip; its small-batch kernel is the decode specialisation.)
//
// At decode sizes a block holds one or two real pairs, so the work is a skinny
// GEMV bound by reading A[l,e] (r x K) and B[l,e] (N x r).  To spread those
// bytes over many SMs, each block is processed by a thread-block cluster of C
// CTAs: CTA c reads the K-slice c of A and of the gathered x rows and forms a
// partial t; the C partials are summed through distributed shared memory (in
// rank order, so the result is deterministic); then CTA c produces the N-slice
// c of y from its slice of B.  Every operand moves global -> shared with 1-D
// bulk (TMA) copies completing on an mbarrier, all issued before the first
// wait; the first B slice is fetched while the shrink runs.  Dot products use
// 16-byte shared-memory vectors and warp-shuffle reductions.  The y rows are
// written back with bulk stores.  The grid covers only active slots: clusters
// walk the blocks of all listed slots (vLLM PR #32005, grid sized by
// num_active_loras rather than max_loras).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace moe_lora {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPG = 16;          // pairs processed together
constexpr int kMaxBlock = 128;   // largest block_size
constexpr int kMaxSlots = 512;   // largest num_active_loras

struct CcCfg {
  int C;          // CTAs per block (cluster size)
  int kc, nc;     // K columns / N rows per chunk (multiples of 8)
  int a_pitch;    // bytes per staged A row (kc + 8 bf16, a 16-byte skew between rows)
  int off_a, off_x, off_b, off_y, off_tp, off_tf;
  int smem_bytes;
};

struct Meta {
  uint64_t bar[2];               // 0: A + x loads, 1: B + y loads
  int slot_l[kMaxSlots];
  int prefix[kMaxSlots + 1];
  int pf[kMaxBlock];             // the block's real pairs (flat index), compacted in order
  int pm[kMaxBlock];             // their token index
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

template <int RV>
__global__ void __launch_bounds__(kThreads) fused_cuda_core_kernel(const FusedArgs p, const CcCfg cfg) {
  extern __shared__ __align__(128) uint8_t smem[];
  Meta &meta = *reinterpret_cast<Meta *>(smem);
  uint8_t *a_s = smem + cfg.off_a;
  uint8_t *x_s = smem + cfg.off_x;
  uint8_t *b_s = smem + cfg.off_b;
  uint8_t *y_s = smem + cfg.off_y;
  float *tpart = reinterpret_cast<float *>(smem + cfg.off_tp);
  float *tfull = reinterpret_cast<float *>(smem + cfg.off_tf);

  cg::cluster_group cluster = cg::this_cluster();
  const int C = cfg.C;
  const int c = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = p.rank, K = p.K, N = p.N, E = p.num_experts, bs = p.block_size;
  const int P = p.M * p.topk;

  if (tid == 0) {
    mbar_init(&meta.bar[0], 1);
    mbar_init(&meta.bar[1], 1);
    meta.abort = 0;
    fence_barrier_init();
  }
  // Blocks per listed slot, and their prefix sum: the work list of the grid.
  for (int z = tid; z < p.num_active_loras; z += kThreads) {
    const int l = __ldg(p.lora_ids + z);
    int nb = 0;
    if (l < 0 || l >= p.max_loras) {
      if (c == 0 && blockIdx.y == 0) flag_error(p.err, MOE_LORA_DEVERR_LORA_ID);
    } else if (!p.adapter_enabled || __ldg(p.adapter_enabled + l) != 0) {
      nb = __ldg(p.num_tokens_post_padded + l) / bs;
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
  __syncthreads();
  const int total_blocks = meta.prefix[p.num_active_loras];

  // This CTA's K- and N-slices, in units of 8 elements.
  const int k8 = K / 8, n8 = N / 8;
  const int k_lo = (c * k8 / C) * 8, k_hi = ((c + 1) * k8 / C) * 8;
  const int n_lo = (c * n8 / C) * 8, n_hi = ((c + 1) * n8 / C) * 8;
  const int nk_chunks = (k_hi - k_lo + cfg.kc - 1) / cfg.kc;
  const int nn_chunks = (n_hi - n_lo + cfg.nc - 1) / cfg.nc;
  uint32_t ph0 = 0, ph1 = 0;
  volatile int *abort = &meta.abort;

  for (int item = blockIdx.y; item < total_blocks; item += gridDim.y) {
    // Locate (slot, block) of this work item.
    int z = 0;
    {
      int lo = 0, hi = p.num_active_loras;  // prefix[lo] <= item < prefix[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (meta.prefix[mid] <= item) lo = mid; else hi = mid;
      }
      z = lo;
    }
    const int l = meta.slot_l[z];
    const int b = item - meta.prefix[z];
    const int e = __ldg(p.expert_ids + (size_t)l * p.max_num_m_blocks + b);
    if (e < 0 || e >= E) {  // uniform over the cluster: every CTA reads the same entry
      if (tid == 0 && c == 0) flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
      continue;
    }
    // Compact the block's real pairs, keeping their order.
    {
      const int32_t *ids = p.sorted_token_ids + (size_t)l * p.max_num_tokens_padded + (size_t)b * bs;
      int f = -1;
      if (tid < bs) {
        f = __ldg(ids + tid);
        if (f != P && (f < 0 || f > P)) {
          if (c == 0) flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);
          f = -1;
        } else if (f == P) {
          f = -1;
        }
      }
      const unsigned bal = __ballot_sync(0xffffffffu, f >= 0);
      if (lane == 0) meta.wcount[warp] = __popc(bal);
      __syncthreads();
      int base = 0, tot = 0;
      for (int w = 0; w < kWarps; ++w) {
        if (w < warp) base += meta.wcount[w];
        tot += meta.wcount[w];
      }
      if (f >= 0) {
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        meta.pf[pos] = f;
        meta.pm[pos] = f / p.topk;
      }
      if (tid == 0) meta.nv = tot;
      __syncthreads();
    }
    const int nv = meta.nv;
    const size_t le = (size_t)l * E + e;
    const uint16_t *A = p.lora_a + le * r * K;
    const uint16_t *B = p.lora_b + le * N * r;

    for (int g0 = 0; g0 < nv; g0 += kPG) {
      const int nvg = min(kPG, nv - g0);
      // Issue the first B slice (and y rows) now so that they arrive during the shrink.
      auto issue_expand = [&](int nc0) {
        const int ncn = min(cfg.nc, n_hi - nc0);
        if (warp == 0) {
          const uint32_t bytes = (uint32_t)ncn * r * 2 + (p.add_inputs ? (uint32_t)nvg * ncn * 2 : 0u);
          if (lane == 0) {
            mbar_arrive_expect_tx(&meta.bar[1], bytes);
            bulk_g2s(b_s, B + (size_t)nc0 * r, (uint32_t)ncn * r * 2, &meta.bar[1]);
          }
          __syncwarp();
          if (p.add_inputs)
            for (int q = lane; q < nvg; q += 32)
              bulk_g2s(y_s + (size_t)q * cfg.nc * 2, p.y + (size_t)meta.pf[g0 + q] * N + nc0,
                       (uint32_t)ncn * 2, &meta.bar[1]);
        }
      };
      issue_expand(n_lo);

      // ---- shrink: partial t over this CTA's K-slice
      for (int i = tid; i < nvg * r; i += kThreads) tpart[i] = 0.f;
      __syncthreads();
      for (int kci = 0; kci < nk_chunks; ++kci) {
        const int kc0 = k_lo + kci * cfg.kc;
        const int kcn = min(cfg.kc, k_hi - kc0);
        if (warp == 0) {
          if (lane == 0) mbar_arrive_expect_tx(&meta.bar[0], (uint32_t)(r + nvg) * kcn * 2);
          __syncwarp();
          for (int j = lane; j < r; j += 32)
            bulk_g2s(a_s + (size_t)j * cfg.a_pitch, A + (size_t)j * K + kc0, (uint32_t)kcn * 2, &meta.bar[0]);
          for (int q = lane; q < nvg; q += 32)
            bulk_g2s(x_s + (size_t)q * cfg.kc * 2, p.x + (size_t)meta.pm[g0 + q] * K + kc0,
                     (uint32_t)kcn * 2, &meta.bar[0]);
        }
        mbar_wait(&meta.bar[0], ph0, abort, p.err);
        ph0 ^= 1;
        const int nch = kcn / 8;
        for (int j = warp; j < r; j += kWarps) {
          float acc[kPG];
#pragma unroll
          for (int q = 0; q < kPG; ++q) acc[q] = 0.f;
          const uint4 *arow = reinterpret_cast<const uint4 *>(a_s + (size_t)j * cfg.a_pitch);
          for (int ch = lane; ch < nch; ch += 32) {
            float af[8];
            unpack8(arow[ch], af);
#pragma unroll
            for (int q = 0; q < kPG; ++q)
              if (q < nvg) acc[q] += dot8(af, reinterpret_cast<const uint4 *>(x_s + (size_t)q * cfg.kc * 2)[ch]);
          }
#pragma unroll
          for (int q = 0; q < kPG; ++q) {
            if (q < nvg) {
              float v = acc[q];
#pragma unroll
              for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
              if (lane == 0) tpart[q * r + j] += v;
            }
          }
        }
        __syncthreads();
      }

      // ---- sum the C partial t's through distributed shared memory
      const float *t = tpart;
      if (C > 1) {
        cluster.sync();
        for (int i = tid; i < nvg * r; i += kThreads) {
          float s = 0.f;
          for (int q = 0; q < C; ++q) s += cluster.map_shared_rank(tpart, q)[i];
          tfull[i] = s;
        }
        cluster.sync();
        t = tfull;
      }

      // ---- expand: y rows of this CTA's N-slice
      constexpr int kLanesMax = 16;
      const int vecs = r / RV;                 // vectors per B row
      int lpr = 1;                             // lanes per B row (power of two)
      while (lpr < vecs && lpr < kLanesMax) lpr <<= 1;
      const int rows_per_warp = 32 / lpr;
      for (int nci = 0; nci < nn_chunks; ++nci) {
        const int nc0 = n_lo + nci * cfg.nc;
        const int ncn = min(cfg.nc, n_hi - nc0);
        if (nci > 0) issue_expand(nc0);
        mbar_wait(&meta.bar[1], ph1, abort, p.err);
        ph1 ^= 1;
        for (int row0 = warp * rows_per_warp; row0 < ncn; row0 += kWarps * rows_per_warp) {
          const int nl = row0 + lane / lpr;
          const int ch0 = lane % lpr;
          float acc[kPG];
#pragma unroll
          for (int q = 0; q < kPG; ++q) acc[q] = 0.f;
          if (nl < ncn) {
            for (int ch = ch0; ch < vecs; ch += lpr) {
              const int j0 = ch * RV;
              if constexpr (RV == 8) {
                float bf[8];
                unpack8(reinterpret_cast<const uint4 *>(b_s + ((size_t)nl * r + j0) * 2)[0], bf);
#pragma unroll
                for (int q = 0; q < kPG; ++q) {
                  if (q < nvg) {
                    const float4 t0 = *reinterpret_cast<const float4 *>(t + q * r + j0);
                    const float4 t1 = *reinterpret_cast<const float4 *>(t + q * r + j0 + 4);
                    acc[q] += bf[0] * t0.x + bf[1] * t0.y + bf[2] * t0.z + bf[3] * t0.w +
                              bf[4] * t1.x + bf[5] * t1.y + bf[6] * t1.z + bf[7] * t1.w;
                  }
                }
              } else {
                float bf[4];
                unpack4(reinterpret_cast<const uint2 *>(b_s + ((size_t)nl * r + j0) * 2)[0], bf);
#pragma unroll
                for (int q = 0; q < kPG; ++q) {
                  if (q < nvg) {
                    const float4 t0 = *reinterpret_cast<const float4 *>(t + q * r + j0);
                    acc[q] += bf[0] * t0.x + bf[1] * t0.y + bf[2] * t0.z + bf[3] * t0.w;
                  }
                }
              }
            }
          }
#pragma unroll
          for (int q = 0; q < kPG; ++q) {
            if (q < nvg) {
              float v = acc[q];
              for (int d = lpr >> 1; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
              if (ch0 == 0 && nl < ncn) {
                uint16_t *dst = reinterpret_cast<uint16_t *>(y_s + (size_t)q * cfg.nc * 2) + nl;
                const float old = p.add_inputs ? bf16_bits_to_float(*dst) : 0.f;
                *dst = float_to_bf16_bits(v + old);
              }
            }
          }
        }
        fence_proxy_async_cta();
        __syncthreads();
        if (warp == 0) {
          for (int q = lane; q < nvg; q += 32)
            bulk_s2g(p.y + (size_t)meta.pf[g0 + q] * N + nc0, y_s + (size_t)q * cfg.nc * 2, (uint32_t)ncn * 2);
          bulk_commit();
          bulk_wait_read_all();
        }
        __syncthreads();
      }
    }
  }
  if (warp == 0) bulk_wait_all();
  // Keep every CTA of the cluster resident until its peers are done reading
  // this CTA's shared memory.
  if (C > 1) cluster.sync();
}

int pick_cfg(const FusedArgs &f, const DeviceInfo &dev, CcCfg *cfg) {
  const int r = f.rank;
  const long long item_bytes = (long long)(f.K + f.N) * r * 2;
  int C = (int)((item_bytes + 24 * 1024 - 1) / (24 * 1024));
  C = C < 1 ? 1 : (C > 8 ? 8 : C);
  C = C > f.K / 8 ? f.K / 8 : C;
  C = C > f.N / 8 ? f.N / 8 : C;
  if (C < 1) C = 1;
  const int kslice = (f.K / 8 + C - 1) / C * 8;
  const int nslice = (f.N / 8 + C - 1) / C * 8;
  int kc_max = ((64 * 1024) / (2 * r) - 8) / 8 * 8;
  int nc_max = ((48 * 1024) / (2 * r)) / 8 * 8;
  if (kc_max < 8) kc_max = 8;
  if (nc_max < 8) nc_max = 8;
  cfg->C = C;
  cfg->kc = kslice < kc_max ? kslice : kc_max;
  cfg->nc = nslice < nc_max ? nslice : nc_max;
  cfg->a_pitch = (cfg->kc + 8) * 2;
  size_t off = (sizeof(Meta) + 127) / 128 * 128;
  cfg->off_a = (int)off;
  off += (size_t)r * cfg->a_pitch;
  cfg->off_x = (int)off;
  off += (size_t)kPG * cfg->kc * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_b = (int)off;
  off += (size_t)cfg->nc * r * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_y = (int)off;
  off += (size_t)kPG * cfg->nc * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_tp = (int)off;
  off += (size_t)kPG * r * 4;
  cfg->off_tf = (int)off;
  off += (size_t)kPG * r * 4;
  cfg->smem_bytes = (int)off;
  if ((size_t)cfg->smem_bytes > dev.max_smem_optin) return MOE_LORA_ERR_UNSUPPORTED;
  return 0;
}

}  // namespace

int launch_fused_cuda_core(const FusedArgs &f, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  if (f.num_active_loras > kMaxSlots || f.block_size > kMaxBlock) return MOE_LORA_ERR_UNSUPPORTED;
  CcCfg cfg;
  if (int st = pick_cfg(f, dev, &cfg)) return st;
  const long long bound = fused_block_bound(f.M, f.topk, f.num_experts, f.num_active_loras, f.block_size);
  if (bound <= 0) return 0;
  const int G = (int)(bound < 65535 ? bound : 65535);
  const void *fn = (f.rank % 8 == 0) ? (const void *)fused_cuda_core_kernel<8>
                                     : (const void *)fused_cuda_core_kernel<4>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes) != cudaSuccess)
    return MOE_LORA_ERR_LAUNCH;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(cfg.C, G, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = cfg.smem_bytes;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cfg.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaError_t err;
  if (f.rank % 8 == 0)
    err = cudaLaunchKernelEx(&lc, fused_cuda_core_kernel<8>, f, cfg);
  else
    err = cudaLaunchKernelEx(&lc, fused_cuda_core_kernel<4>, f, cfg);
  return err == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

}  // namespace moe_lora
