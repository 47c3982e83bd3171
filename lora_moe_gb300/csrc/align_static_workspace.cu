// align_static_workspace.cu -- moe_lora_align_static_workspace: the global-
// memory align variant run on a scratch buffer that lives inside this library
// instead of one the caller allocates.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocating
// routine) at the point where they align -- for example code that runs under
// an allocator that forbids device allocations on this path, plugins handed
// only input and output buffers by a host framework, or callers that must not
// grow device memory after start-up.  They still pass every input and output
// buffer; only the workspace is supplied by the library.
//
// The scratch is a file-scope __device__ array of kStaticWorkspaceBytes
// (4 MiB).  Every GPU that loads this library holds that much device memory
// for it until the process exits.  Host code may not use the array's name as
// a device address (on the host it is only a stand-in symbol), so the first
// call on each device, with that device current, looks the address up with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls on a device share the one array and it keeps the last
// call's contents: the align kernels write every workspace entry they later
// read, so nothing needs clearing, but calls that overlap on the GPU (on
// different streams, or from different host threads without ordering) race
// on the array and must not be issued.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "moe_lora.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = MOE_LORA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Device address of g_static_workspace on the current device, looked up once
// per device.  Returns nullptr (and the CUDA error in *err) on failure.
void *static_workspace_address(cudaError_t *err) {
  static std::mutex mu;
  static void *addr[kMaxDevices] = {};
  int dev = -1;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_static_workspace);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int moe_lora_align_static_workspace(const int32_t *topk_ids, const int32_t *token_lora_mapping,
                                               const int32_t *lora_ids, const int32_t *adapter_enabled, int M,
                                               int topk, int num_experts, int max_loras, int num_active_loras,
                                               int block_size, int32_t *sorted_token_ids, int32_t *expert_ids,
                                               int32_t *num_tokens_post_padded, int max_num_tokens_padded,
                                               int max_num_m_blocks, int32_t *err_flag, void *stream) {
  const size_t need = moe_lora_align_workspace_bytes(M, topk, num_experts, num_active_loras, block_size,
                                                     MOE_LORA_ALIGN_GLOBAL);
  if (need > kStaticWorkspaceBytes) return MOE_LORA_ERR_WORKSPACE;  // beyond the built-in scratch
  cudaError_t cerr = cudaSuccess;
  void *ws = nullptr;
  if (num_active_loras > 0) {
    ws = static_workspace_address(&cerr);
    if (!ws) return MOE_LORA_ERR_DEVICE;
  }
  return moe_lora_align(topk_ids, token_lora_mapping, lora_ids, adapter_enabled, M, topk, num_experts, max_loras,
                        num_active_loras, block_size, sorted_token_ids, expert_ids, num_tokens_post_padded,
                        max_num_tokens_padded, max_num_m_blocks, ws, kStaticWorkspaceBytes, MOE_LORA_ALIGN_GLOBAL,
                        err_flag, stream);
}
