// fused_stream_cc.cu -- the fused MoE-LoRA shrink+expand on CUDA cores for
// decode-sized blocks with large adapters (sm_103a).
//
// Computes, for each block of each listed slot (l, e), each adapter slice s
// and each real pair f of the block (input row x_f: row f / topk, or row f
// when x holds one row per pair; router weight w_f, 1 without weights):
//     t[j]    = sum_k x_f[k] * A_s[l][e][j][k]                (fp32)
//     y[f][off + s*N + n] = bf16((add_inputs ? y_in : 0) + w_f * sum_j B_s[l][e][n][j] * t[j])
// (prhub.com.cn summary of vLLM PR #42290, "Implementation breakdown" step 1;
// its small-batch kernel is the decode specialisation of the one-shot kernel.)
//
// At decode sizes a block holds one or two real pairs: the work is a skinny
// GEMV bound by streaming A[l,e] and B[l,e].  This kernel streams them through
// the shared rings of stream_pipeline.cuh (balanced (block, tile) ranges per
// persistent CTA, TMA for the adapter tiles, cp.async for x and y rows) and
// does the arithmetic on CUDA cores, reading 16-byte shared-memory vectors
// straight out of the swizzled tiles:
//   warp 0      expand producer     warps 9, 10  shrink producers
//   warps 1..8  compute: per k-tile, each thread accumulates the dot products
//               of its (pair, rank row) items over the tile's 64 columns; at the
//               end of the block t goes to shared memory (fp32); per output
//               tile, each thread forms (column, pair) outputs from a B row and
//               t, adds y_in, rounds to bf16; rows leave with 16-byte stores.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_utils.cuh"
#include "internal.h"
#include "stream_pipeline.cuh"

namespace moe_lora {

namespace {

constexpr int kWarps = 11;
constexpr int kThreads = kWarps * 32;
constexpr int kCompWarps = 8;
constexpr int kCompThreads = kCompWarps * 32;
constexpr int kMaxAcc = 8;         // shrink items per compute thread (block_size * rank <= 2048)

__device__ __forceinline__ float dot8_bf16(const uint4 a, const uint4 b) {
  const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s = fmaf(__uint_as_float(wa[i] << 16), __uint_as_float(wb[i] << 16), s);
    s = fmaf(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(wb[i] & 0xFFFF0000u), s);
  }
  return s;
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
    fused_stream_cc_kernel(const __grid_constant__ stream::TmapSet maps, const FusedArgs p, const stream::Cfg cfg) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  stream::Meta &meta = *reinterpret_cast<stream::Meta *>(smem + cfg.off_meta);
  uint8_t *sh_base = smem + cfg.off_sh;
  uint8_t *ex_base = smem + cfg.off_ex;
  float *t_s = reinterpret_cast<float *>(smem + cfg.off_t);   // [real pairs][r_pad]
  volatile int *abort = &meta.abort;

  if (tid == 0) {
    for (int s = 0; s < cfg.s_sh; ++s) {
      mbar_init(&meta.full_sh[s], 1 + 32);
      mbar_init(&meta.empty_sh[s], kCompWarps);
    }
    for (int s = 0; s < cfg.s_ex; ++s) {
      mbar_init(&meta.full_ex[s], 1 + 32);
      mbar_init(&meta.empty_ex[s], kCompWarps);
    }
    meta.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < p.num_slices) {
    prefetch_tensor_map(&maps.a[lane]);
    prefetch_tensor_map(&maps.b[lane]);
  }
  wait_for_prior_grid();   // align outputs are read from here on
  stream::slot_prefix<BS>(p, meta);
  __syncthreads();
  const stream::Range rg = stream::cta_range(meta, p.num_active_loras, p.num_slices, cfg);

  if (warp == 9 || warp == 10) {
    stream::shrink_producer<BS>(p, cfg, meta, &maps, sh_base, rg, warp - 9);
  } else if (warp == 0) {
    stream::expand_producer<BS>(p, cfg, meta, &maps, ex_base, rg);
  } else {
    const int ctid = tid - 32, cwarp = warp - 1;
    const int N = p.N, E = p.num_experts, r = p.rank, r_pad = cfg.r_pad, P = p.M * p.topk;
    const int kb = cfg.ka * 2;
    uint32_t sh_iter = 0, ex_iter = 0;
    for (int gb = rg.gb0; gb <= rg.gb1; gb += rg.step) {
      const stream::BlockRef br = stream::block_ref<BS>(p, meta, gb);
      const bool e_ok = br.e >= 0 && br.e < E;
      // -- the block's real pairs, in order: row in the block and pair id
      named_barrier(1, kCompThreads);   // previous block is done with cpx / epi_f / t_s
      int f = -1;
      bool valid = false;
      if (ctid < BS) {
        f = __ldg(br.ids + ctid);
        valid = f >= 0 && f < P && e_ok;
        if ((f < 0 || f > P) && br.s == 0) flag_error(p.err, MOE_LORA_DEVERR_PAIR_ID);
      }
      const unsigned bal = __ballot_sync(0xffffffffu, valid);
      if (lane == 0) meta.wcount[cwarp] = __popc(bal);
      named_barrier(1, kCompThreads);
      int base = 0, nv = 0;
#pragma unroll
      for (int w = 0; w < kCompWarps; ++w) {
        base += (w < cwarp) ? meta.wcount[w] : 0;
        nv += meta.wcount[w];
      }
      if (valid) {
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        meta.cpx[pos] = ctid;
        meta.epi_f[pos] = f;
        meta.epi_w[pos] = route_weight(p, f);
      }
      named_barrier(1, kCompThreads);

      // -- shrink over all K: thread items (pair pi, rank row j), item = ctid + 256 i
      const int n_items = nv * r;
      float acc[kMaxAcc];
      int irow[kMaxAcc], ij[kMaxAcc];
#pragma unroll
      for (int i = 0; i < kMaxAcc; ++i) {
        acc[i] = 0.f;
        const int item = ctid + kCompThreads * i;
        const int pi = item < n_items ? item / r : 0;
        ij[i] = item < n_items ? item - pi * r : 0;
        irow[i] = item < n_items ? meta.cpx[pi] : 0;
      }
      for (int kt = 0; kt < cfg.kt_total; ++kt, ++sh_iter) {
        const int s = sh_iter % cfg.s_sh;
        mbar_wait(&meta.full_sh[s], (sh_iter / cfg.s_sh) & 1, abort, p.err);
        const uint8_t *xt = sh_base + (size_t)s * cfg.sh_stage;
        const uint8_t *at = xt + cfg.at_off;
#pragma unroll
        for (int i = 0; i < kMaxAcc; ++i) {
          if (ctid + kCompThreads * i < n_items) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 av = *reinterpret_cast<const uint4 *>(at + stream::swz(ij[i], c, 128));
              const uint4 xv = *reinterpret_cast<const uint4 *>(xt + stream::swz(irow[i], c, 128));
              acc[i] += dot8_bf16(av, xv);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta.empty_sh[s]);
      }
#pragma unroll
      for (int i = 0; i < kMaxAcc; ++i) {
        const int item = ctid + kCompThreads * i;
        if (item < n_items) t_s[(item / r) * r_pad + ij[i]] = acc[i];
      }
      for (int i = ctid; i < nv * r_pad; i += kCompThreads)   // rank columns past r stay zero
        if (i % r_pad >= r) t_s[i] = 0.f;
      named_barrier(1, kCompThreads);

      // -- expand, tile by tile: thread items (column n, pair pi), item = ctid + 256 i
      for (int nt = rg.tile_lo(gb); nt < rg.tile_hi(gb); ++nt, ++ex_iter) {
        const int s = ex_iter % cfg.s_ex;
        mbar_wait(&meta.full_ex[s], (ex_iter / cfg.s_ex) & 1, abort, p.err);
        const uint8_t *bt = ex_base + (size_t)s * cfg.ex_stage;
        uint8_t *yt = ex_base + (size_t)s * cfg.ex_stage + cfg.yt_off;
        const int n0 = nt * stream::kTileN;
        for (int item = ctid; item < stream::kTileN * nv; item += kCompThreads) {
          const int n = item & (stream::kTileN - 1), pi = item >> 7;
          const float *tp = t_s + pi * r_pad;
          float a = 0.f;
          for (int cc = 0; cc < r_pad / 8; ++cc) {
            const int atom = cc * 8 / cfg.ka, c = (cc * 8 % cfg.ka) / 8;
            const uint4 bv = *reinterpret_cast<const uint4 *>(bt + atom * (stream::kTileN * kb) + stream::swz(n, c, kb));
            const uint32_t w[4] = {bv.x, bv.y, bv.z, bv.w};
            const float4 t0 = *reinterpret_cast<const float4 *>(tp + cc * 8);
            const float4 t1 = *reinterpret_cast<const float4 *>(tp + cc * 8 + 4);
            a = fmaf(__uint_as_float(w[0] << 16), t0.x, a);
            a = fmaf(__uint_as_float(w[0] & 0xFFFF0000u), t0.y, a);
            a = fmaf(__uint_as_float(w[1] << 16), t0.z, a);
            a = fmaf(__uint_as_float(w[1] & 0xFFFF0000u), t0.w, a);
            a = fmaf(__uint_as_float(w[2] << 16), t1.x, a);
            a = fmaf(__uint_as_float(w[2] & 0xFFFF0000u), t1.y, a);
            a = fmaf(__uint_as_float(w[3] << 16), t1.z, a);
            a = fmaf(__uint_as_float(w[3] & 0xFFFF0000u), t1.w, a);
          }
          if (n0 + n < N) {
            uint16_t *dst = reinterpret_cast<uint16_t *>(yt + meta.cpx[pi] * (stream::kTileN * 2)) + n;
            a *= meta.epi_w[pi];
            if (p.add_inputs) a += bf16_bits_to_float(*dst);
            *dst = float_to_bf16_bits(a);
          }
        }
        named_barrier(1, kCompThreads);
        for (int item = ctid; item < nv * 16; item += kCompThreads) {
          const int pi = item >> 4, c16 = item & 15;
          const int nn = n0 + c16 * 8;
          if (nn < N)
            *reinterpret_cast<uint4 *>(p.y + y_base(p, meta.epi_f[pi], br.s) + nn) =
                *reinterpret_cast<const uint4 *>(yt + meta.cpx[pi] * (stream::kTileN * 2) + c16 * 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta.empty_ex[s]);
      }
    }
  }
}

template <int BS>
int launch_bs(const FusedArgs &f, const stream::Cfg &cfg, const stream::TmapSet &maps, int G, cudaStream_t s) {
  const void *fn = (const void *)fused_stream_cc_kernel<BS>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem_bytes) != cudaSuccess)
    return MOE_LORA_ERR_LAUNCH;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(G, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = cfg.smem_bytes;
  lc.stream = s;
  // May start while the align kernel before it is finishing (it waits for it
  // with griddepcontrol.wait before touching the align outputs).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&lc, fused_stream_cc_kernel<BS>, maps, f, cfg);
  return err == cudaSuccess ? 0 : MOE_LORA_ERR_LAUNCH;
}

}  // namespace

bool stream_cc_supports(const FusedArgs &f) {
  return f.rank % 8 == 0 && f.num_active_loras <= stream::kMaxSlots &&
         (long long)f.block_size * f.rank <= (long long)kCompThreads * kMaxAcc;
}

int launch_fused_stream_cc(const FusedArgs &f, cudaStream_t s) {
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  if (!stream_cc_supports(f)) return MOE_LORA_ERR_UNSUPPORTED;
  const int r16 = (f.rank + 15) / 16 * 16;
  const int r_pad = r16 <= 16 ? 16 : (r16 <= 32 ? 32 : (r16 <= 64 ? 64 : 128));
  stream::Cfg cfg;
  if (int st = stream::plan(f, dev, f.block_size * r_pad * 4, 1, &cfg)) return st;
  stream::TmapSet maps;
  if (int st = stream::make_tensor_maps(f, cfg, &maps)) return st;
  const long long bound = fused_block_bound(f.M, f.topk, f.num_experts, f.num_active_loras, f.block_size);
  if (bound <= 0) return 0;
  const int per_sm = std::max(1, (228 * 1024) / (cfg.smem_bytes + 1024));
  long long G = (long long)dev.sm_count * per_sm;
  if (G > bound * f.num_slices * cfg.nt_total) G = bound * f.num_slices * cfg.nt_total;
  if (G < 1) G = 1;
  switch (f.block_size) {
    case 16: return launch_bs<16>(f, cfg, maps, (int)G, s);
    case 32: return launch_bs<32>(f, cfg, maps, (int)G, s);
    case 64: return launch_bs<64>(f, cfg, maps, (int)G, s);
    case 128: return launch_bs<128>(f, cfg, maps, (int)G, s);
    default: return MOE_LORA_ERR_UNSUPPORTED;
  }
}

}  // namespace moe_lora
