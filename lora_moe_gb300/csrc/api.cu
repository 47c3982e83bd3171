// api.cu -- the C ABI of libmoe_lora.so (declared in include/moe_lora.h):
// argument validation, workspace sizing and the choice of align variant and
// fused path.  Every check runs on the host before anything is enqueued.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "moe_lora.h"

namespace moe_lora {

int current_device_info(DeviceInfo *out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_LORA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MOE_LORA_ERR_DEVICE;
    cache[dev].device = dev;
    cache[dev].sm_count = prop.multiProcessorCount;
    cache[dev].major = prop.major;
    cache[dev].minor = prop.minor;
    cache[dev].max_smem_optin = prop.sharedMemPerBlockOptin;
    have[dev] = true;
  }
  *out = cache[dev];
  // The kernels are built for sm_103a only (tcgen05, TMA, clusters); an
  // arch-specific image loads on compute capability 10.3 alone.
  if (out->major != 10 || out->minor != 3) return MOE_LORA_ERR_DEVICE;
  return 0;
}

}  // namespace moe_lora

using namespace moe_lora;

namespace {

constexpr int kMaxExperts = 1024;   // vLLM PR #29257 review: num_experts <= 1024
constexpr int kMaxRank = 128;       // PR #42290 summary: the one-shot kernel supports rank <= 128
constexpr int kMaxSlots = 512;

bool valid_block_size(int bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128; }

// Ranks each forced path takes: the tensor-core kernel rank % 8 == 0, the
// cluster streaming kernel the powers of two 8 .. 128.
bool path_takes_rank(int path, int rank) {
  if (path == MOE_LORA_PATH_TCGEN05) return rank % 8 == 0;
  if (path == MOE_LORA_PATH_CUDA_CORE_STREAM) return rank >= 8 && rank <= 128 && (rank & (rank - 1)) == 0;
  return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long capacity_tokens(int M, int topk, int E, int bs) {
  return (long long)M * topk + (long long)E * (bs - 1);
}

// Shared checks of the sizes both entry points take.
int check_common(int M, int topk, int E, int max_loras, int nact, int bs, int max_ntp, int max_blocks) {
  if (M < 0 || topk < 1 || E < 1 || max_loras < 1 || nact < 0) return MOE_LORA_ERR_INVALID_ARG;
  if (E > kMaxExperts || topk > E) return MOE_LORA_ERR_UNSUPPORTED;
  if (!valid_block_size(bs)) return MOE_LORA_ERR_UNSUPPORTED;
  if (nact > max_loras) return MOE_LORA_ERR_INVALID_ARG;
  if (nact > kMaxSlots) return MOE_LORA_ERR_UNSUPPORTED;
  const long long cap = capacity_tokens(M, topk, E, bs);
  if (cap > INT32_MAX / 2) return MOE_LORA_ERR_UNSUPPORTED;
  if (max_ntp < cap || (long long)max_blocks * bs < cap) return MOE_LORA_ERR_INVALID_ARG;
  if ((long long)max_loras * max_ntp > INT32_MAX || (long long)max_loras * max_blocks > INT32_MAX)
    return MOE_LORA_ERR_UNSUPPORTED;
  return 0;
}

// The shared-memory variant runs one CTA per active slot; the global variant
// spreads each slot's pairs over many CTAs in three launches; the cluster
// variant over up to 8 CTAs of one thread-block cluster in one launch.  AUTO
// takes the cluster variant for large expert counts (vLLM PR #29257, Purpose:
// the global-memory variant exists for large num_experts) and for long pair
// lists, where it measured 10-13 us against 20-34 us for the three launches
// and 21-47 us for one CTA per slot (prefill and large-E workloads), and the
// shared-memory variant otherwise (3-5 us on the decode workloads, against
// 6-7 us clustered).  The global variant is the fallback when the cluster's
// per-warp counters do not fit in shared memory.
int resolve_align_variant(int M, int topk, int E, int variant) {
  if (variant == MOE_LORA_ALIGN_SMEM || variant == MOE_LORA_ALIGN_GLOBAL || variant == MOE_LORA_ALIGN_CLUSTER)
    return variant;
  const bool large = !align_smem_fits(E) || E >= 256 || (long long)M * topk >= 16384;
  if (!large) return MOE_LORA_ALIGN_SMEM;
  return align_cluster_fits(E) ? MOE_LORA_ALIGN_CLUSTER : MOE_LORA_ALIGN_GLOBAL;
}

}  // namespace

// Both align entry points: a null token_lora_mapping puts every token in the
// one slot, null lora_ids make slot z row z (the plain MoE align).
static int align_impl(const int32_t *topk_ids, const int32_t *token_lora_mapping, const int32_t *lora_ids,
                   const int32_t *adapter_enabled, int M, int topk, int num_experts, int max_loras,
                   int num_active_loras, int block_size, int32_t *sorted_token_ids, int32_t *expert_ids,
                   int32_t *num_tokens_post_padded, int max_num_tokens_padded, int max_num_m_blocks,
                   void *workspace, size_t workspace_bytes, int variant, int32_t *err_flag, void *stream) {
  if (int st = check_common(M, topk, num_experts, max_loras, num_active_loras, block_size, max_num_tokens_padded,
                            max_num_m_blocks))
    return st;
  if (variant < MOE_LORA_ALIGN_AUTO || variant > MOE_LORA_ALIGN_CLUSTER) return MOE_LORA_ERR_INVALID_ARG;
  if (num_active_loras == 0) return MOE_LORA_OK;
  if (!sorted_token_ids || !expert_ids || !num_tokens_post_padded) return MOE_LORA_ERR_INVALID_ARG;
  if (M > 0 && !topk_ids) return MOE_LORA_ERR_INVALID_ARG;
  const int v = resolve_align_variant(M, topk, num_experts, variant);
  if (v == MOE_LORA_ALIGN_SMEM && !align_smem_fits(num_experts)) return MOE_LORA_ERR_UNSUPPORTED;
  if (v == MOE_LORA_ALIGN_CLUSTER && !align_cluster_fits(num_experts)) return MOE_LORA_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  AlignArgs a;
  a.topk_ids = topk_ids;
  a.token_lora_mapping = token_lora_mapping;
  a.lora_ids = lora_ids;
  a.adapter_enabled = adapter_enabled;
  a.sorted_token_ids = sorted_token_ids;
  a.expert_ids = expert_ids;
  a.num_tokens_post_padded = num_tokens_post_padded;
  a.err = err_flag;
  a.M = M;
  a.topk = topk;
  a.num_experts = num_experts;
  a.max_loras = max_loras;
  a.num_active_loras = num_active_loras;
  a.block_size = block_size;
  a.max_num_tokens_padded = max_num_tokens_padded;
  a.max_num_m_blocks = max_num_m_blocks;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (v == MOE_LORA_ALIGN_SMEM) return launch_align_smem(a, s);
  if (v == MOE_LORA_ALIGN_CLUSTER) return launch_align_cluster(a, s);
  const size_t need = align_global_workspace_bytes(M, topk, num_experts, num_active_loras);
  if (!workspace || workspace_bytes < need) return MOE_LORA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MOE_LORA_ERR_MISALIGNED;
  return launch_align_global(a, workspace, s);
}

// Checks and fills what both fused entry points (sorted and naive block
// assignment) share: the operands, the options and the rank / size limits.
// *empty is set when there is nothing to do (no active slot or no token).
static int prepare_fused(const moe_lora_bf16 *x, int x_per_pair, const moe_lora_bf16 *const *lora_a,
                         const moe_lora_bf16 *const *lora_b, int num_slices, moe_lora_bf16 *y, int ldy, int y_offset,
                         const float *topk_weights, const int32_t *lora_ids, const int32_t *adapter_enabled, int M,
                         int topk, int num_experts, int K, int N, int rank, int max_loras, int num_active_loras,
                         int add_inputs, int32_t *err_flag, FusedArgs *out, bool *empty) {
  if (K < 8 || N < 8 || rank < 1) return MOE_LORA_ERR_INVALID_ARG;
  if (num_slices < 1 || num_slices > kMaxSlices || !lora_a || !lora_b) return MOE_LORA_ERR_INVALID_ARG;
  if (y_offset < 0 || ldy < 8 || (long long)y_offset + (long long)num_slices * N > ldy) return MOE_LORA_ERR_INVALID_ARG;
  if (rank > kMaxRank || rank % 4 != 0) return MOE_LORA_ERR_UNSUPPORTED;
  if (K % 8 != 0 || N % 8 != 0 || ldy % 8 != 0 || y_offset % 8 != 0) return MOE_LORA_ERR_MISALIGNED;
  const long long x_rows = x_per_pair ? (long long)M * topk : (long long)M;
  if (x_rows * K > INT32_MAX * 8LL || (long long)M * topk * ldy > INT32_MAX * 8LL) return MOE_LORA_ERR_UNSUPPORTED;
  *empty = num_active_loras == 0 || M == 0;
  if (*empty) return MOE_LORA_OK;
  if (!x || !y || !lora_ids) return MOE_LORA_ERR_INVALID_ARG;
  for (int s = 0; s < num_slices; ++s) {
    if (!lora_a[s] || !lora_b[s]) return MOE_LORA_ERR_INVALID_ARG;
    if (!aligned16(lora_a[s]) || !aligned16(lora_b[s])) return MOE_LORA_ERR_MISALIGNED;
  }
  if (!aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(topk_weights) & 3u))
    return MOE_LORA_ERR_MISALIGNED;
  FusedArgs f = {};
  f.x = x;
  for (int s = 0; s < kMaxSlices; ++s) {
    f.lora_a[s] = lora_a[s < num_slices ? s : 0];
    f.lora_b[s] = lora_b[s < num_slices ? s : 0];
  }
  f.y = y;
  f.topk_weights = topk_weights;
  f.lora_ids = lora_ids;
  f.adapter_enabled = adapter_enabled;
  f.err = err_flag;
  f.M = M;
  f.topk = topk;
  f.num_experts = num_experts;
  f.K = K;
  f.N = N;
  f.rank = rank;
  f.max_loras = max_loras;
  f.num_active_loras = num_active_loras;
  f.add_inputs = add_inputs ? 1 : 0;
  f.num_slices = num_slices;
  f.x_per_pair = x_per_pair ? 1 : 0;
  f.ldy = ldy;
  f.y_offset = y_offset;
  *out = f;
  return 0;
}

// Opt-in shared memory per block on compute capability 10.3 (227 KB): what the
// host-only queries plan against when no device is asked.
constexpr int kSmemOptinSm103 = 232448;

// Whether the cluster kernel can hold a CTA's slices of A and B (and its x
// and y rows) in shared memory with at most 16 CTAs per block.  Host
// arithmetic only.
static bool cluster_kernel_fits(const FusedArgs &f, size_t max_smem) {
  DeviceInfo dev = {};
  dev.major = 10;
  dev.minor = 3;
  dev.max_smem_optin = max_smem;
  FusedPlan plan = {};
  return plan_fused_cuda_core(f, dev, &plan) == 0;
}

// The kernel a fused call runs.
//   * Batches of at least 1024 pairs: the tensor-core kernel (when it supports
//     the sizes): blocks hold enough pairs for a real contraction.
//   * Smaller (decode) batches whose adapters, by the block bound, exceed
//     48 MB: the cluster streaming kernel (when it takes the rank), which
//     splits each block over a 4-CTA cluster and keeps every SM streaming
//     (gpt-oss-shaped w2 decode: 64 us, against 93 us on tensor cores).
//   * Other decode batches, and MOE_LORA_PATH_CUDA_CORE: the one-cluster-per-
//     block kernel (Qwen3-shaped w13 decode: 7.9 us, against 11.1 us
//     streaming) -- unless its shared memory cannot hold a CTA's share of the
//     adapter rows (N * rank or K * rank beyond what 16 CTAs hold): then the
//     tensor-core kernel when K and N span at least one 64-wide K tile and 32
//     output columns, else the streaming kernel.
static int resolve_path(const FusedArgs &f, int path, size_t max_smem) {
  int use = path;
  if (use == MOE_LORA_PATH_AUTO) {
    const double touched = (double)fused_block_bound(f.M, f.topk, f.num_experts, f.num_active_loras, f.block_size) *
                           f.num_slices * (double)(f.K + f.N) * f.rank * 2.0;
    const bool prefill = (long long)f.M * f.topk >= 1024;
    const bool tc = tcgen05_path_supports(f);
    const bool stream = cluster_stream_supports(f);
    if (prefill && tc)
      use = MOE_LORA_PATH_TCGEN05;
    else if (!prefill && touched > 48.0e6 && stream)
      use = MOE_LORA_PATH_CUDA_CORE_STREAM;
    else if (!prefill && touched > 48.0e6 && tc)
      use = MOE_LORA_PATH_TCGEN05;
    else if (cluster_kernel_fits(f, max_smem))
      use = MOE_LORA_PATH_CUDA_CORE;
    else if (tc && f.K >= 64 && f.N >= 32)
      use = MOE_LORA_PATH_TCGEN05;
    else if (stream)
      use = MOE_LORA_PATH_CUDA_CORE_STREAM;
    else
      use = MOE_LORA_PATH_CUDA_CORE;
  }
  if (use == MOE_LORA_PATH_CUDA_CORE) use = MOE_LORA_PATH_CUDA_CORE_CLUSTER;
  return use;
}

// The kernel a naive-assignment call runs (a path value), or -status.  AUTO
// takes the cluster streaming kernel when the pairs' adapters exceed 48 MB
// (gpt-oss-shaped w2 decode: 51 us, against 96 us) and it takes the rank,
// else the one-cluster-per-pair kernel (Qwen3-shaped decode: 7.6 us,
// against 12.9 us streaming), which MOE_LORA_PATH_CUDA_CORE also names.
static int resolve_naive_path(const FusedArgs &f, int path) {
  const bool stream = cluster_stream_supports(f);
  if (path == MOE_LORA_PATH_CUDA_CORE_STREAM) return stream ? MOE_LORA_PATH_CUDA_CORE_STREAM : -MOE_LORA_ERR_UNSUPPORTED;
  if (path == MOE_LORA_PATH_AUTO && stream) {
    const double touched = (double)f.M * f.topk * f.num_slices * (double)(f.K + f.N) * f.rank * 2.0;
    if (touched > 48.0e6) return MOE_LORA_PATH_CUDA_CORE_STREAM;
  }
  return MOE_LORA_PATH_CUDA_CORE_CLUSTER;
}

namespace moe_lora {

int check_align_args(const int32_t *topk_ids, const int32_t *token_lora_mapping, const int32_t *lora_ids, int M,
                     int topk, int num_experts, int max_loras, int num_active_loras, int block_size,
                     const int32_t *sorted_token_ids, const int32_t *expert_ids,
                     const int32_t *num_tokens_post_padded, int max_num_tokens_padded, int max_num_m_blocks,
                     int variant) {
  if (int st = check_common(M, topk, num_experts, max_loras, num_active_loras, block_size, max_num_tokens_padded,
                            max_num_m_blocks))
    return st;
  if (variant < MOE_LORA_ALIGN_AUTO || variant > MOE_LORA_ALIGN_CLUSTER) return MOE_LORA_ERR_INVALID_ARG;
  if (M > 0 && num_active_loras > 0 && !token_lora_mapping) return MOE_LORA_ERR_INVALID_ARG;
  if (num_active_loras > 0 && !lora_ids) return MOE_LORA_ERR_INVALID_ARG;
  if (num_active_loras == 0) return MOE_LORA_OK;
  if (!sorted_token_ids || !expert_ids || !num_tokens_post_padded) return MOE_LORA_ERR_INVALID_ARG;
  if (M > 0 && !topk_ids) return MOE_LORA_ERR_INVALID_ARG;
  return MOE_LORA_OK;
}

}  // namespace moe_lora

static int naive_impl(const moe_lora_bf16 *x, int x_per_pair, const moe_lora_bf16 *const *lora_a,
                                       const moe_lora_bf16 *const *lora_b, int num_slices, moe_lora_bf16 *y,
                                       int ldy, int y_offset, const float *topk_weights, const int32_t *topk_ids,
                                       const int32_t *token_lora_mapping, const int32_t *lora_ids,
                                       const int32_t *adapter_enabled, int M, int topk, int num_experts, int K,
                                       int N, int rank, int max_loras, int num_active_loras, int add_inputs,
                                       int path, int32_t *err_flag, void *stream,
                                       unsigned long long wait_limit_ns = 0, int withhold_b = 0) {
  if (M < 0 || topk < 1 || num_experts < 1 || max_loras < 1 || num_active_loras < 0) return MOE_LORA_ERR_INVALID_ARG;
  if (path != MOE_LORA_PATH_AUTO && path != MOE_LORA_PATH_CUDA_CORE && path != MOE_LORA_PATH_CUDA_CORE_CLUSTER &&
      path != MOE_LORA_PATH_CUDA_CORE_STREAM)
    return MOE_LORA_ERR_INVALID_ARG;
  if (!path_takes_rank(path, rank)) return MOE_LORA_ERR_UNSUPPORTED;
  if (num_experts > kMaxExperts || topk > num_experts) return MOE_LORA_ERR_UNSUPPORTED;
  if (num_active_loras > max_loras) return MOE_LORA_ERR_INVALID_ARG;
  if ((long long)M * topk > INT32_MAX / 2) return MOE_LORA_ERR_UNSUPPORTED;
  FusedArgs f;
  bool empty = false;
  if (int st = prepare_fused(x, x_per_pair, lora_a, lora_b, num_slices, y, ldy, y_offset, topk_weights, lora_ids,
                             adapter_enabled, M, topk, num_experts, K, N, rank, max_loras, num_active_loras,
                             add_inputs, err_flag, &f, &empty))
    return st;
  if (empty) return MOE_LORA_OK;
  if (!topk_ids || !token_lora_mapping) return MOE_LORA_ERR_INVALID_ARG;
  f.topk_ids = topk_ids;
  f.token_lora_mapping = token_lora_mapping;
  const int use = resolve_naive_path(f, path);
  if (use < 0) return -use;
  if (use == MOE_LORA_PATH_CUDA_CORE_STREAM) return launch_fused_cluster_stream_naive(f, static_cast<cudaStream_t>(stream));
  return launch_fused_naive(f, static_cast<cudaStream_t>(stream), wait_limit_ns, withhold_b);
}

extern "C" {

int moe_lora_version(void) { return 100; }

const char *moe_lora_status_string(int status) {
  switch (status) {
    case MOE_LORA_OK: return "ok";
    case MOE_LORA_ERR_INVALID_ARG: return "invalid argument";
    case MOE_LORA_ERR_UNSUPPORTED: return "unsupported size or option";
    case MOE_LORA_ERR_MISALIGNED: return "pointer or row not 16-byte aligned";
    case MOE_LORA_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_LORA_ERR_LAUNCH: return "CUDA launch failed";
    case MOE_LORA_ERR_DEVICE: return "no usable device (compute capability 10.3 required)";
    default: return "unknown status";
  }
}

int moe_lora_max_num_tokens_padded(int M, int topk, int num_experts, int block_size) {
  if (M < 0 || topk < 1 || num_experts < 1 || block_size < 1) return -1;
  const long long cap = capacity_tokens(M, topk, num_experts, block_size);
  return cap > INT32_MAX ? -1 : (int)cap;
}

int moe_lora_max_num_m_blocks(int M, int topk, int num_experts, int block_size) {
  const int cap = moe_lora_max_num_tokens_padded(M, topk, num_experts, block_size);
  if (cap < 0) return -1;
  return (cap + block_size - 1) / block_size;
}

int moe_lora_align_resolve_variant(int M, int topk, int num_experts, int variant) {
  if (M < 0 || topk < 1 || num_experts < 1 || variant < MOE_LORA_ALIGN_AUTO || variant > MOE_LORA_ALIGN_CLUSTER)
    return -MOE_LORA_ERR_INVALID_ARG;
  if (num_experts > kMaxExperts || topk > num_experts) return -MOE_LORA_ERR_UNSUPPORTED;
  const int v = resolve_align_variant(M, topk, num_experts, variant);
  if ((v == MOE_LORA_ALIGN_SMEM && !align_smem_fits(num_experts)) ||
      (v == MOE_LORA_ALIGN_CLUSTER && !align_cluster_fits(num_experts)))
    return -MOE_LORA_ERR_UNSUPPORTED;
  return v;
}

size_t moe_lora_align_workspace_bytes(int M, int topk, int num_experts, int num_active_loras, int block_size,
                                      int variant) {
  if (M < 0 || topk < 1 || num_experts < 1 || num_experts > kMaxExperts || num_active_loras < 0 ||
      !valid_block_size(block_size))
    return 0;
  if (resolve_align_variant(M, topk, num_experts, variant) != MOE_LORA_ALIGN_GLOBAL) return 0;
  return align_global_workspace_bytes(M, topk, num_experts, num_active_loras);
}

int moe_lora_align(const int32_t *topk_ids, const int32_t *token_lora_mapping, const int32_t *lora_ids,
                   const int32_t *adapter_enabled, int M, int topk, int num_experts, int max_loras,
                   int num_active_loras, int block_size, int32_t *sorted_token_ids, int32_t *expert_ids,
                   int32_t *num_tokens_post_padded, int max_num_tokens_padded, int max_num_m_blocks,
                   void *workspace, size_t workspace_bytes, int variant, int32_t *err_flag, void *stream) {
  if (int st = check_align_args(topk_ids, token_lora_mapping, lora_ids, M, topk, num_experts, max_loras,
                                num_active_loras, block_size, sorted_token_ids, expert_ids, num_tokens_post_padded,
                                max_num_tokens_padded, max_num_m_blocks, variant))
    return st;
  return align_impl(topk_ids, token_lora_mapping, lora_ids, adapter_enabled, M, topk, num_experts, max_loras,
                    num_active_loras, block_size, sorted_token_ids, expert_ids, num_tokens_post_padded,
                    max_num_tokens_padded, max_num_m_blocks, workspace, workspace_bytes, variant, err_flag, stream);
}

int moe_align_block_size(const int32_t *topk_ids, int M, int topk, int num_experts, int block_size,
                         int32_t *sorted_token_ids, int32_t *expert_ids, int32_t *num_tokens_post_padded,
                         int max_num_tokens_padded, int max_num_m_blocks, void *workspace, size_t workspace_bytes,
                         int variant, int32_t *err_flag, void *stream) {
  return align_impl(topk_ids, nullptr, nullptr, nullptr, M, topk, num_experts, 1, 1, block_size, sorted_token_ids,
                    expert_ids, num_tokens_post_padded, max_num_tokens_padded, max_num_m_blocks, workspace,
                    workspace_bytes, variant, err_flag, stream);
}

static int resolve_path_query(int M, int topk, int num_experts, int K, int N, int rank, int num_active_loras,
                              int block_size, int num_slices, int path, size_t max_smem) {
  if (M < 0 || topk < 1 || num_experts < 1 || K < 8 || N < 8 || rank < 1 || num_active_loras < 0 ||
      num_slices < 1 || num_slices > kMaxSlices || path < MOE_LORA_PATH_AUTO || path > MOE_LORA_PATH_CUDA_CORE_STREAM)
    return -MOE_LORA_ERR_INVALID_ARG;
  if (!valid_block_size(block_size) || rank > kMaxRank || rank % 4 != 0) return -MOE_LORA_ERR_UNSUPPORTED;
  if (!path_takes_rank(path, rank)) return -MOE_LORA_ERR_UNSUPPORTED;
  FusedArgs f = {};
  f.M = M;
  f.topk = topk;
  f.num_experts = num_experts;
  f.K = K;
  f.N = N;
  f.rank = rank;
  f.num_active_loras = num_active_loras;
  f.block_size = block_size;
  f.num_slices = num_slices;
  return resolve_path(f, path, max_smem);
}

int moe_lora_fused_naive_resolve_path(int M, int topk, int num_experts, int K, int N, int rank,
                                      int num_active_loras, int num_slices, int path) {
  if (M < 0 || topk < 1 || num_experts < 1 || K < 8 || N < 8 || rank < 1 || num_active_loras < 0 ||
      num_slices < 1 || num_slices > kMaxSlices)
    return -MOE_LORA_ERR_INVALID_ARG;
  if (path != MOE_LORA_PATH_AUTO && path != MOE_LORA_PATH_CUDA_CORE && path != MOE_LORA_PATH_CUDA_CORE_CLUSTER &&
      path != MOE_LORA_PATH_CUDA_CORE_STREAM)
    return -MOE_LORA_ERR_INVALID_ARG;
  if (rank > kMaxRank || rank % 4 != 0 || !path_takes_rank(path, rank)) return -MOE_LORA_ERR_UNSUPPORTED;
  FusedArgs f = {};
  f.M = M;
  f.topk = topk;
  f.num_experts = num_experts;
  f.K = K;
  f.N = N;
  f.rank = rank;
  f.num_active_loras = num_active_loras;
  f.num_slices = num_slices;
  f.block_size = 16;   // (no blocks under the naive assignment)
  return resolve_naive_path(f, path);
}

int moe_lora_fused_resolve_path(int M, int topk, int num_experts, int K, int N, int rank, int num_active_loras,
                                int block_size, int num_slices, int path) {
  return resolve_path_query(M, topk, num_experts, K, N, rank, num_active_loras, block_size, num_slices, path,
                            kSmemOptinSm103);
}

int moe_lora_fused_plan(int M, int topk, int num_experts, int K, int N, int rank, int num_active_loras,
                        int block_size, int num_slices, int path, int sm_count, int max_smem_per_block,
                        int32_t *out) {
  if (!out || sm_count < 1 || max_smem_per_block < 1) return MOE_LORA_ERR_INVALID_ARG;
  const int use = resolve_path_query(M, topk, num_experts, K, N, rank, num_active_loras, block_size, num_slices,
                                     path, (size_t)max_smem_per_block);
  if (use < 0) return -use;
  FusedArgs f = {};
  f.M = M;
  f.topk = topk;
  f.num_experts = num_experts;
  f.K = K;
  f.N = N;
  f.rank = rank;
  f.max_loras = num_active_loras;
  f.num_active_loras = num_active_loras;
  f.block_size = block_size;
  f.num_slices = num_slices;
  DeviceInfo dev = {};
  dev.sm_count = sm_count;
  dev.major = 10;
  dev.minor = 3;
  dev.max_smem_optin = (size_t)max_smem_per_block;
  FusedPlan plan = {};
  const int st = use == MOE_LORA_PATH_TCGEN05          ? plan_fused_tcgen05(f, dev, &plan)
                 : use == MOE_LORA_PATH_CUDA_CORE_STREAM ? plan_fused_cluster_stream(f, dev, false, &plan)
                                                         : plan_fused_cuda_core(f, dev, &plan);
  if (st) return st;
  const int32_t vals[11] = {plan.kernel, plan.grid, plan.threads, plan.smem_bytes, plan.s_sh, plan.lag, plan.s_ex,
                            plan.t_bufs, plan.tmem_cols, plan.cluster, plan.pairs_per_group};
  for (int i = 0; i < 11; ++i) out[i] = vals[i];
  return 0;
}

int moe_lora_fused_shrink_expand_ex(const moe_lora_bf16 *x, int x_per_pair, const moe_lora_bf16 *const *lora_a,
                                    const moe_lora_bf16 *const *lora_b, int num_slices, moe_lora_bf16 *y, int ldy,
                                    int y_offset, const float *topk_weights, const int32_t *sorted_token_ids,
                                    const int32_t *expert_ids, const int32_t *num_tokens_post_padded,
                                    const int32_t *lora_ids, const int32_t *adapter_enabled, int M, int topk,
                                    int num_experts, int K, int N, int rank, int max_loras, int num_active_loras,
                                    int block_size, int max_num_tokens_padded, int max_num_m_blocks, int add_inputs,
                                    int path, int32_t *err_flag, void *stream) {
  if (int st = check_common(M, topk, num_experts, max_loras, num_active_loras, block_size, max_num_tokens_padded,
                            max_num_m_blocks))
    return st;
  if (path < MOE_LORA_PATH_AUTO || path > MOE_LORA_PATH_CUDA_CORE_STREAM) return MOE_LORA_ERR_INVALID_ARG;
  if (!path_takes_rank(path, rank)) return MOE_LORA_ERR_UNSUPPORTED;
  FusedArgs f;
  bool empty = false;
  if (int st = prepare_fused(x, x_per_pair, lora_a, lora_b, num_slices, y, ldy, y_offset, topk_weights, lora_ids,
                             adapter_enabled, M, topk, num_experts, K, N, rank, max_loras, num_active_loras,
                             add_inputs, err_flag, &f, &empty))
    return st;
  if (empty) return MOE_LORA_OK;
  if (!sorted_token_ids || !expert_ids || !num_tokens_post_padded) return MOE_LORA_ERR_INVALID_ARG;
  f.sorted_token_ids = sorted_token_ids;
  f.expert_ids = expert_ids;
  f.num_tokens_post_padded = num_tokens_post_padded;
  f.block_size = block_size;
  f.max_num_tokens_padded = max_num_tokens_padded;
  f.max_num_m_blocks = max_num_m_blocks;
  DeviceInfo dev;
  if (int st = current_device_info(&dev)) return st;
  const int use = resolve_path(f, path, dev.max_smem_optin);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (use) {
    case MOE_LORA_PATH_TCGEN05: return launch_fused_tcgen05(f, s);
    case MOE_LORA_PATH_CUDA_CORE_STREAM: return launch_fused_cluster_stream(f, s);
    default: return launch_fused_cuda_core(f, s);
  }
}

int moe_lora_fused_shrink_expand_naive(const moe_lora_bf16 *x, int x_per_pair, const moe_lora_bf16 *const *lora_a,
                                       const moe_lora_bf16 *const *lora_b, int num_slices, moe_lora_bf16 *y,
                                       int ldy, int y_offset, const float *topk_weights, const int32_t *topk_ids,
                                       const int32_t *token_lora_mapping, const int32_t *lora_ids,
                                       const int32_t *adapter_enabled, int M, int topk, int num_experts, int K,
                                       int N, int rank, int max_loras, int num_active_loras, int add_inputs,
                                       int path, int32_t *err_flag, void *stream) {
  return naive_impl(x, x_per_pair, lora_a, lora_b, num_slices, y, ldy, y_offset, topk_weights, topk_ids,
                    token_lora_mapping, lora_ids, adapter_enabled, M, topk, num_experts, K, N, rank, max_loras,
                    num_active_loras, add_inputs, path, err_flag, stream);
}

int moe_lora_test_withheld_copy(const moe_lora_bf16 *x, int x_per_pair, const moe_lora_bf16 *const *lora_a,
                                const moe_lora_bf16 *const *lora_b, int num_slices, moe_lora_bf16 *y, int ldy,
                                int y_offset, const float *topk_weights, const int32_t *topk_ids,
                                const int32_t *token_lora_mapping, const int32_t *lora_ids,
                                const int32_t *adapter_enabled, int M, int topk, int num_experts, int K, int N,
                                int rank, int max_loras, int num_active_loras, int add_inputs,
                                unsigned long long wait_limit_ns, int32_t *err_flag, void *stream) {
  if (wait_limit_ns < 1000ull || wait_limit_ns > 4000000000ull) return MOE_LORA_ERR_INVALID_ARG;
  return naive_impl(x, x_per_pair, lora_a, lora_b, num_slices, y, ldy, y_offset, topk_weights, topk_ids,
                    token_lora_mapping, lora_ids, adapter_enabled, M, topk, num_experts, K, N, rank, max_loras,
                    num_active_loras, add_inputs, MOE_LORA_PATH_CUDA_CORE_CLUSTER, err_flag, stream, wait_limit_ns,
                    1);
}

int moe_lora_fused_shrink_expand(const moe_lora_bf16 *x, const moe_lora_bf16 *lora_a, const moe_lora_bf16 *lora_b,
                                 moe_lora_bf16 *y, const int32_t *sorted_token_ids, const int32_t *expert_ids,
                                 const int32_t *num_tokens_post_padded, const int32_t *lora_ids,
                                 const int32_t *adapter_enabled, int M, int topk, int num_experts, int K, int N,
                                 int rank, int max_loras, int num_active_loras, int block_size,
                                 int max_num_tokens_padded, int max_num_m_blocks, int add_inputs, int path,
                                 int32_t *err_flag, void *stream) {
  const moe_lora_bf16 *a[1] = {lora_a};
  const moe_lora_bf16 *b[1] = {lora_b};
  return moe_lora_fused_shrink_expand_ex(x, 0, a, b, 1, y, N, 0, nullptr, sorted_token_ids, expert_ids,
                                         num_tokens_post_padded, lora_ids, adapter_enabled, M, topk, num_experts, K,
                                         N, rank, max_loras, num_active_loras, block_size, max_num_tokens_padded,
                                         max_num_m_blocks, add_inputs, path, err_flag, stream);
}

}  // extern "C"
