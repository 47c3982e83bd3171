// internal.h -- argument blocks and launchers shared between the C-ABI layer
// (api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe_lora {

// Align outputs and inputs, as validated by the C-ABI layer.
struct AlignArgs {
  const int32_t *topk_ids;
  const int32_t *token_lora_mapping;  // null: every token in the one slot (plain MoE align)
  const int32_t *lora_ids;            // null: slot z is row z
  const int32_t *adapter_enabled;  // may be null
  int32_t *sorted_token_ids;
  int32_t *expert_ids;
  int32_t *num_tokens_post_padded;
  int32_t *err;                    // may be null
  int M, topk, num_experts, max_loras, num_active_loras, block_size;
  int max_num_tokens_padded, max_num_m_blocks;
};

constexpr int kMaxSlices = 4;

// Fused-stage inputs, as validated by the C-ABI layer.
struct FusedArgs {
  const uint16_t *x;                   // bf16 [M, K], or [M*topk, K] when x_per_pair
  const uint16_t *lora_a[kMaxSlices];  // per slice: bf16 [L, E, r, K]
  const uint16_t *lora_b[kMaxSlices];  // per slice: bf16 [L, E, N, r]
  uint16_t *y;                         // bf16 [M, topk, ldy]; slice s at columns y_offset + s*N
  const float *topk_weights;           // fp32 [M, topk] or null (no router-weight scaling)
  const int32_t *sorted_token_ids;        // align outputs (null for naive block assignment)
  const int32_t *expert_ids;
  const int32_t *num_tokens_post_padded;
  const int32_t *topk_ids;                // routing (naive block assignment only)
  const int32_t *token_lora_mapping;
  const int32_t *lora_ids;
  const int32_t *adapter_enabled;  // may be null
  int32_t *err;                    // may be null
  int M, topk, num_experts, K, N, rank, max_loras, num_active_loras, block_size;
  int max_num_tokens_padded, max_num_m_blocks;
  int add_inputs;
  int num_slices;
  int x_per_pair;
  int ldy, y_offset;
};

// Device helpers for the per-slice operands and the pair's rows.
__device__ __forceinline__ const uint16_t *slice_a(const FusedArgs &p, int s) {
  return s == 0 ? p.lora_a[0] : (s == 1 ? p.lora_a[1] : (s == 2 ? p.lora_a[2] : p.lora_a[3]));
}
__device__ __forceinline__ const uint16_t *slice_b(const FusedArgs &p, int s) {
  return s == 0 ? p.lora_b[0] : (s == 1 ? p.lora_b[1] : (s == 2 ? p.lora_b[2] : p.lora_b[3]));
}
// Row of x that pair f reads.
__device__ __forceinline__ int x_row(const FusedArgs &p, int f) { return p.x_per_pair ? f : f / p.topk; }
// First element of slice s's output columns in pair f's row of y.
__device__ __forceinline__ size_t y_base(const FusedArgs &p, int f, int s) {
  return (size_t)f * p.ldy + p.y_offset + (size_t)s * p.N;
}
// Router weight of pair f (1 when there are none).
__device__ __forceinline__ float route_weight(const FusedArgs &p, int f) {
  return p.topk_weights ? __ldg(p.topk_weights + f) : 1.f;
}

// Upper bound on the number of blocks all active slots can produce together:
// every pair belongs to at most one slot, so the blocks are at most
// floor(M*topk / bs) full ones plus one partly filled block per non-empty
// (slot, expert) segment.
inline long long fused_block_bound(int M, int topk, int E, int nact, int bs) {
  const long long pairs = (long long)M * topk;
  const long long segs = (long long)nact * E < pairs ? (long long)nact * E : pairs;
  return pairs / bs + segs;
}

// Pairs per warp in the global align variant, and its workspace layout:
// per slot, a [warps][E] table of per-warp expert counts followed by [E]
// segment offsets.
int align_global_pairs_per_warp(int M, int topk);
size_t align_global_workspace_bytes(int M, int topk, int E, int nact);
bool align_smem_fits(int E);

// The argument checks of moe_lora_align (sizes, variant, required pointers),
// without touching a device: 0 or a moe_lora_status code.
int check_align_args(const int32_t *topk_ids, const int32_t *token_lora_mapping, const int32_t *lora_ids, int M,
                     int topk, int num_experts, int max_loras, int num_active_loras, int block_size,
                     const int32_t *sorted_token_ids, const int32_t *expert_ids,
                     const int32_t *num_tokens_post_padded, int max_num_tokens_padded, int max_num_m_blocks,
                     int variant);

int launch_align_smem(const AlignArgs &a, cudaStream_t stream);
// The cluster variant: CTAs per slot for these sizes, whether its shared
// memory holds the per-warp counters of E experts, and the launch.
int align_cluster_size(int M, int topk);
bool align_cluster_fits(int E);
int launch_align_cluster(const AlignArgs &a, cudaStream_t stream);
int launch_align_global(const AlignArgs &a, void *workspace, cudaStream_t stream);
int launch_fused_cuda_core(const FusedArgs &f, cudaStream_t stream);
// Naive block assignment: one work item per pair, no align outputs.  For the
// test of the bounded waits only: wait_limit_ns (0: the default 4 s) bounds the
// wait for each CTA's B slice, and withhold_b leaves that copy unissued.
int launch_fused_naive(const FusedArgs &f, cudaStream_t stream, unsigned long long wait_limit_ns = 0,
                       int withhold_b = 0);
int launch_fused_tcgen05(const FusedArgs &f, cudaStream_t stream);
// Whether the tensor-core path takes these arguments (rank % 8 == 0, at most
// 128 listed slots).
bool tcgen05_path_supports(const FusedArgs &f);
// The cluster streaming kernel (CUDA cores; decode-sized blocks): sorted and
// naive block assignment.  Takes rank % 8 == 0, at most 128 listed slots.
bool cluster_stream_supports(const FusedArgs &f);
int launch_fused_cluster_stream(const FusedArgs &f, cudaStream_t stream);
int launch_fused_cluster_stream_naive(const FusedArgs &f, cudaStream_t stream);

// Device properties of the current device, cached per device.
struct DeviceInfo {
  int device;
  int sm_count;
  int major, minor;
  size_t max_smem_optin;
};
int current_device_info(DeviceInfo *out);

// The launch plan of a fused call (host arithmetic only).
struct FusedPlan {
  int kernel;                              // MOE_LORA_PATH_TCGEN05 or _CUDA_CORE_CLUSTER
  int grid, threads, smem_bytes;
  int s_sh, lag, s_ex, t_bufs, tmem_cols;  // tensor-core kernel: rings and TMEM
  int cluster, pairs_per_group;            // cluster kernel: CTAs per block, pairs per group
};
int plan_fused_tcgen05(const FusedArgs &f, const DeviceInfo &dev, FusedPlan *out);
int plan_fused_cuda_core(const FusedArgs &f, const DeviceInfo &dev, FusedPlan *out);
int plan_fused_cluster_stream(const FusedArgs &f, const DeviceInfo &dev, bool naive, FusedPlan *out);

}  // namespace moe_lora
