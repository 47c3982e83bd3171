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
//     dimension is the number of active LoRAs); blocks past
//     num_tokens_post_padded exit after one dependent load.
//   * a thread-block cluster of C CTAs shares a block: CTA c streams the
//     K-slice c of A and of the gathered x rows and the N-slice c of B and y;
//     the C partial t's are summed through distributed shared memory in rank
//     order (deterministic).
//   * every operand is requested at once, before the first wait: A, x and y_in
//     rows with 16-byte cp.async (load/store unit), the contiguous B slice with
//     one bulk copy.  Dot products read 16-byte shared-memory vectors and reduce
//     with warp shuffles; y is written with coalesced stores.
#include <cooperative_groups.h>
#include <algorithm>
#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace moe_lora {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPG = 8;           // pairs processed together
constexpr int kMaxBlock = 128;   // largest block_size
constexpr int kMaxCluster = 16;

struct CcCfg {
  int C;               // CTAs per block (cluster size)
  int kslice, nslice;  // per-CTA K / N slice capacity (multiples of 8)
  int a_pitch;         // bytes per staged A row (kslice + 8 bf16: rows skewed by 16 B)
  int off_a, off_x, off_b, off_y, off_tp, off_tf;
  int smem_bytes;
};

struct Meta {
  uint64_t bar;                  // the B slice's bulk copy
  int pf[kMaxBlock];             // the block's real pairs (flat index), in order
  int pm[kMaxBlock];             // their row of x
  float pw[kMaxBlock];           // their router weight
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

// RV: elements of B per shared-memory vector (8 when rank % 8 == 0, else 4).
// NAIVE: one pair per work item, found from topk_ids and token_lora_mapping
// (naive block assignment, no align); otherwise blocks of the align output.
template <int RV, bool NAIVE>
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
  // grid.y: slice * num_active_loras + slot (sorted), or the slice (naive)
  const int z = NAIVE ? 0 : (int)(blockIdx.y % p.num_active_loras);
  const int sl = NAIVE ? (int)blockIdx.y : (int)(blockIdx.y / p.num_active_loras);

  wait_for_prior_grid();   // every input is read from here on
  int l = 0, nitems = P, e_first = 0, f_first = -1;
  if (!NAIVE) {
    // Uniform over the cluster: every CTA of it reads the same values.
    l = __ldg(p.lora_ids + z);
    if (l < 0 || l >= p.max_loras) {
      if (c == 0 && tid == 0 && blockIdx.z == 0 && sl == 0) flag_error(p.err, MOE_LORA_DEVERR_LORA_ID);
      return;
    }
    if (p.adapter_enabled && __ldg(p.adapter_enabled + l) == 0) return;
    // The first block's expert and pair ids are requested together with the
    // slot's block count (one round trip); they are only used if the block exists.
    const int b_first = blockIdx.z;
    e_first = __ldg(p.expert_ids + (size_t)l * p.max_num_m_blocks + b_first);
    if (tid < bs && b_first * bs + tid < p.max_num_tokens_padded)
      f_first = __ldg(p.sorted_token_ids + (size_t)l * p.max_num_tokens_padded + b_first * bs + tid);
    nitems = min(__ldg(p.num_tokens_post_padded + l) / bs, p.max_num_m_blocks);
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

  // This CTA's K- and N-slices, in units of 8 elements.
  const int k8 = K / 8, n8 = N / 8;
  const int k_lo = (c * k8 / C) * 8, k_hi = ((c + 1) * k8 / C) * 8;
  const int n_lo = (c * n8 / C) * 8, n_hi = ((c + 1) * n8 / C) * 8;
  const int kn = k_hi - k_lo, nn = n_hi - n_lo;

  for (int b = blockIdx.z; b < nitems; b += gridDim.z) {
    int e;
    if (NAIVE) {
      // work item b is pair b
      if (!naive_pair(p, b, l, e)) continue;
      if (tid == 0) {
        meta.pf[0] = b;
        meta.pm[0] = x_row(p, b);
        meta.pw[0] = route_weight(p, b);
        meta.nv = 1;
      }
      __syncthreads();
    } else {
      e = b == (int)blockIdx.z ? e_first : __ldg(p.expert_ids + (size_t)l * p.max_num_m_blocks + b);
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
      if (e < 0 || e >= E) {  // uniform over the cluster
        if (tid == 0 && c == 0 && sl == 0) flag_error(p.err, MOE_LORA_DEVERR_EXPERT_ID);
        continue;
      }
    }
    const int nv = meta.nv;
    const size_t le = (size_t)l * E + e;
    const uint16_t *A = slice_a(p, sl) + le * r * K;
    const uint16_t *Bm = slice_b(p, sl) + le * N * r;

    for (int g0 = 0; g0 < nv; g0 += kPG) {
      const int nvg = min(kPG, nv - g0);
      // ---- request every operand of this group at once
      if (g0 == 0 && tid == 0) {
        mbar_arrive_expect_tx(&meta.bar, (uint32_t)nn * r * 2);
        bulk_g2s(b_s, Bm + (size_t)n_lo * r, (uint32_t)nn * r * 2, &meta.bar);
      }
      {
        const int kch = kn / 8, nch = nn / 8;
        if (g0 == 0)
          for (int i = tid; i < r * kch; i += kThreads) {
            const int j = i / kch, ch = i - j * kch;
            cp_async_16(a_s + (size_t)j * cfg.a_pitch + ch * 16, A + (size_t)j * K + k_lo + ch * 8, 16u);
          }
        for (int i = tid; i < nvg * kch; i += kThreads) {
          const int q = i / kch, ch = i - q * kch;
          cp_async_16(x_s + (size_t)q * cfg.kslice * 2 + ch * 16,
                      p.x + (size_t)meta.pm[g0 + q] * K + k_lo + ch * 8, 16u);
        }
        if (p.add_inputs)
          for (int i = tid; i < nvg * nch; i += kThreads) {
            const int q = i / nch, ch = i - q * nch;
            cp_async_16(y_s + (size_t)q * cfg.nslice * 2 + ch * 16,
                        p.y + y_base(p, meta.pf[g0 + q], sl) + n_lo + ch * 8, 16u);
          }
        cp_async_commit();
      }
      cp_async_wait_group<0>();
      __syncthreads();

      // ---- shrink: partial t over this CTA's K-slice; warp w owns rows j = w (mod 8)
      {
        const int nch = kn / 8;
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
              if (q < nvg)
                acc[q] += dot8(af, reinterpret_cast<const uint4 *>(x_s + (size_t)q * cfg.kslice * 2)[ch]);
          }
#pragma unroll
          for (int q = 0; q < kPG; ++q) {
            if (q < nvg) {
              float v = acc[q];
#pragma unroll
              for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
              if (lane == 0) tpart[q * r + j] = v;
            }
          }
        }
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
        t = tfull;
      }
      __syncthreads();
      if (g0 == 0) mbar_wait(&meta.bar, phase, abort, p.err);

      // ---- expand: y rows of this CTA's N-slice.  A B row is read by lpr lanes
      // (one shared-memory vector each); their partial sums meet by shuffles.
      {
        const int vecs = r / RV;
        int lpr = 1;
        while (lpr < vecs && lpr < 16) lpr <<= 1;
        const int rows_per_warp = 32 / lpr;
        for (int row0 = warp * rows_per_warp; row0 < nn; row0 += kWarps * rows_per_warp) {
          const int nl = row0 + lane / lpr;
          const int ch0 = lane % lpr;
          float acc[kPG];
#pragma unroll
          for (int q = 0; q < kPG; ++q) acc[q] = 0.f;
          if (nl < nn) {
            for (int ch = ch0; ch < vecs; ch += lpr) {
              const int j0 = ch * RV;
              if constexpr (RV == 8) {
                float bf[8];
                unpack8(*reinterpret_cast<const uint4 *>(b_s + ((size_t)nl * r + j0) * 2), bf);
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
                unpack4(*reinterpret_cast<const uint2 *>(b_s + ((size_t)nl * r + j0) * 2), bf);
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
              if (ch0 == 0 && nl < nn) {
                const float old = p.add_inputs
                                      ? bf16_bits_to_float(reinterpret_cast<const uint16_t *>(
                                            y_s + (size_t)q * cfg.nslice * 2)[nl])
                                      : 0.f;
                p.y[y_base(p, meta.pf[g0 + q], sl) + n_lo + nl] = float_to_bf16_bits(v * meta.pw[g0 + q] + old);
              }
            }
          }
        }
      }
      // Peers are done reading this CTA's partial t (and every thread with this
      // group's shared memory) before the next group or block reuses it.
      if (C > 1) cluster.sync(); else __syncthreads();
    }
    if (nv > 0) phase ^= 1;
  }
}

// Shared-memory layout for cluster size C; returns false if it does not fit.
bool layout(const FusedArgs &f, const DeviceInfo &dev, int C, CcCfg *cfg) {
  const int r = f.rank;
  cfg->C = C;
  cfg->kslice = (f.K / 8 + C - 1) / C * 8;
  cfg->nslice = (f.N / 8 + C - 1) / C * 8;
  cfg->a_pitch = (cfg->kslice + 8) * 2;
  size_t off = (sizeof(Meta) + 127) / 128 * 128;
  cfg->off_a = (int)off;
  off += (size_t)r * cfg->a_pitch;
  cfg->off_x = (int)off;
  off += (size_t)kPG * cfg->kslice * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_b = (int)off;
  off += (size_t)cfg->nslice * r * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_y = (int)off;
  off += (size_t)kPG * cfg->nslice * 2;
  off = (off + 127) / 128 * 128;
  cfg->off_tp = (int)off;
  off += (size_t)kPG * r * 4;
  cfg->off_tf = (int)off;
  off += (size_t)kPG * r * 4;
  cfg->smem_bytes = (int)off;
  return (size_t)cfg->smem_bytes <= dev.max_smem_optin;
}

// Spread a block's adapter bytes over up to 16 CTAs: at least ~12 KB each
// (so that each CTA is worth its launch, up to 8 CTAs) and at most ~48 KB each
// (so that several CTAs share an SM); more CTAs if shared memory demands it.
int pick_cfg(const FusedArgs &f, const DeviceInfo &dev, CcCfg *cfg) {
  const long long item_bytes = (long long)(f.K + f.N) * f.rank * 2;
  const long long lo = (item_bytes + 48 * 1024 - 1) / (48 * 1024);
  long long hi = (item_bytes + 12 * 1024 - 1) / (12 * 1024);
  if (hi > 8) hi = 8;
  long long want = lo > hi ? lo : hi;
  const long long cmax = std::min<long long>(kMaxCluster, std::min(f.K / 8, f.N / 8));
  if (want > cmax) want = cmax;
  if (want < 1) want = 1;
  for (long long C = want; C <= cmax; ++C)
    if (layout(f, dev, (int)C, cfg)) return 0;
  return MOE_LORA_ERR_UNSUPPORTED;
}

}  // namespace

namespace {

template <bool NAIVE>
int launch_mode(const FusedArgs &f, const CcCfg &cfg, unsigned gy, unsigned gz, cudaStream_t stream) {
  const void *fn = (f.rank % 8 == 0) ? (const void *)fused_cuda_core_kernel<8, NAIVE>
                                     : (const void *)fused_cuda_core_kernel<4, NAIVE>;
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
  cudaError_t err;
  if (f.rank % 8 == 0)
    err = cudaLaunchKernelEx(&lc, fused_cuda_core_kernel<8, NAIVE>, f, cfg);
  else
    err = cudaLaunchKernelEx(&lc, fused_cuda_core_kernel<4, NAIVE>, f, cfg);
  return err == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

}  // namespace

int launch_fused_cuda_core(const FusedArgs &f, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  if (f.block_size > kMaxBlock) return MOE_LORA_ERR_UNSUPPORTED;
  if ((long long)f.num_active_loras * f.num_slices > 65535) return MOE_LORA_ERR_UNSUPPORTED;
  CcCfg cfg;
  if (int st = pick_cfg(f, dev, &cfg)) return st;
  // Blocks one slot can produce: floor(M*topk / bs) full ones plus one partly
  // filled block per non-empty expert segment.
  const long long pairs = (long long)f.M * f.topk;
  long long per_slot = pairs / f.block_size + (pairs < f.num_experts ? pairs : f.num_experts);
  if (per_slot > f.max_num_m_blocks) per_slot = f.max_num_m_blocks;
  // Blocks a slot really has are usually far fewer than that bound; past a few
  // waves of clusters, CTAs walk several blocks instead of launching empty.
  const long long cap =
      std::max<long long>(48, 4LL * dev.sm_count / ((long long)cfg.C * f.num_active_loras * f.num_slices));
  if (per_slot > cap) per_slot = cap;
  if (per_slot > 65535) per_slot = 65535;
  if (per_slot <= 0) return 0;
  return launch_mode<false>(f, cfg, (unsigned)(f.num_active_loras * f.num_slices), (unsigned)per_slot, stream);
}

int launch_fused_naive(const FusedArgs &f, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  CcCfg cfg;
  if (int st = pick_cfg(f, dev, &cfg)) return st;
  // grid (C, slices, pairs), as the one-program-per-pair grid of the naive
  // assignment; past a few waves, CTAs walk several pairs.
  long long items = (long long)f.M * f.topk;
  const long long cap = std::max<long long>(64, 16LL * dev.sm_count / ((long long)cfg.C * f.num_slices));
  if (items > cap) items = cap;
  if (items > 65535) items = 65535;
  if (items <= 0) return 0;
  return launch_mode<true>(f, cfg, (unsigned)f.num_slices, (unsigned)items, stream);
}

}  // namespace moe_lora
