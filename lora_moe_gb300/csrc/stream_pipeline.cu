// stream_pipeline.cu -- host side of the streaming skeleton (see
// stream_pipeline.cuh): tensor maps and the choice of ring depths.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "stream_pipeline.cuh"

namespace moe_lora {
namespace stream {

namespace {

// cuTensorMapEncodeTiled, fetched through the runtime so that the library
// does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once; the initialisation of a function-local static is
// thread-safe, so concurrent first calls from several host threads agree.
EncodeTiledFn get_encode_fn() {
  static const EncodeTiledFn fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

int round_up(int v, int a) { return (v + a - 1) / a * a; }

}  // namespace

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

int make_tensor_maps(const FusedArgs &f, const Cfg &cfg, TmapSet *maps) {
  const uint64_t LE = (uint64_t)f.max_loras * f.num_experts;
  const CUtensorMapSwizzle bsw = cfg.ka == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                              : (cfg.ka == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  for (int s = 0; s < kMaxSlices; ++s) {
    const int src = s < f.num_slices ? s : 0;   // unused entries repeat slice 0
    if (int st = encode_3d(&maps->a[s], f.lora_a[src], (uint64_t)f.K, (uint64_t)f.rank, LE, kTileK,
                           (uint32_t)cfg.r_pad, CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
    if (int st = encode_3d(&maps->b[s], f.lora_b[src], (uint64_t)f.rank, (uint64_t)f.N, LE, (uint32_t)cfg.ka, kTileN,
                           bsw))
      return st;
  }
  return 0;
}

int plan(const FusedArgs &f, const DeviceInfo &dev, int consumer_bytes, int t_bufs_max, Cfg *cfg) {
  const int BS = f.block_size;
  const int r16 = round_up(f.rank, 16);
  cfg->r_pad = r16 <= 16 ? 16 : (r16 <= 32 ? 32 : (r16 <= 64 ? 64 : 128));
  cfg->ka = cfg->r_pad >= 64 ? 64 : cfg->r_pad;
  cfg->natoms = cfg->r_pad / cfg->ka;
  const int kb = cfg->ka * 2;
  cfg->kt_total = (f.K + kTileK - 1) / kTileK;
  cfg->nt_total = (f.N + kTileN - 1) / kTileN;
  cfg->at_off = BS * 128;
  cfg->sh_stage = round_up(BS * 128 + cfg->r_pad * 128, 1024);
  cfg->yt_off = round_up(cfg->natoms * kTileN * kb, 1024);
  cfg->ex_stage = round_up(cfg->yt_off + BS * kTileN * 2, 1024);
  cfg->t_part = round_up(consumer_bytes, 1024);
  cfg->unit_sh_bytes = (long long)cfg->kt_total * (BS * 128 + cfg->r_pad * 128);
  cfg->tile_bytes = (long long)cfg->natoms * kTileN * kb + (long long)BS * kTileN * 2;
  // The Meta block sits last and needs no more than 16-byte alignment.
  const int meta_bytes = round_up((int)sizeof(Meta), 128);
  const int budget = (int)dev.max_smem_optin;

  // Choose the ring depths with the most bytes in flight (the shrink ring has
  // 2 * (lag + 1) stages in flight: two producer warps, each up to `lag` owned
  // stages ahead), each ring's credit capped at 128 KB, a little credit for a
  // second T buffer, and a small charge for the shared memory used.
  int best = -1 << 30;
  Cfg pick = *cfg;
  bool found = false;
  for (int s_sh = kMaxStages; s_sh >= 2; --s_sh) {
    const int lag = std::min(kMaxLag, (s_sh - 1) / 2);
    const int sh_fly = std::min(s_sh, 2 * (lag + 1)) * cfg->sh_stage;
    for (int s_ex = kMaxStages; s_ex >= 1; --s_ex) {
      for (int t_bufs = t_bufs_max; t_bufs >= 1; --t_bufs) {
        const int after_sh = s_ex * cfg->ex_stage + t_bufs * cfg->t_part + meta_bytes;
        const int total = s_sh * cfg->sh_stage + after_sh;
        if (total > budget) continue;
        // the M=128 shrink MMA of the tensor-core kernel reads 128 x-tile rows:
        // the rows past block_size (never used) must still lie in the allocation
        if (cfg->sh_stage + after_sh < 128 * 128) continue;
        // a one-stage expand ring cannot load the next tile while the current
        // one is in use: taken only when no deeper ring fits
        const int score = std::min(sh_fly, 128 * 1024) + std::min(s_ex * cfg->ex_stage, 128 * 1024) +
                          (t_bufs == 2 ? 8 * 1024 : 0) - total / 64 - (s_ex == 1 ? (1 << 24) : 0);
        if (score > best) {
          best = score;
          found = true;
          pick = *cfg;
          pick.s_sh = s_sh;
          pick.lag = lag;
          pick.s_ex = s_ex;
          pick.t_bufs = t_bufs;
          pick.off_sh = 0;
          pick.off_ex = s_sh * cfg->sh_stage;
          pick.off_t = pick.off_ex + s_ex * cfg->ex_stage;
          pick.off_meta = pick.off_t + t_bufs * cfg->t_part;
          pick.smem_bytes = total;
        }
      }
    }
  }
  if (!found) return MOE_LORA_ERR_UNSUPPORTED;
  *cfg = pick;
  return 0;
}

}  // namespace stream
}  // namespace moe_lora
