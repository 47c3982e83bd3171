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
// call in each CUDA context (normally once per device: the runtime's primary
// context), with that context current, looks the address up with
// cudaGetSymbolAddress and caches it under the context's unique id; make that
// first call before any stream capture.  A context created later (after
// cudaDeviceReset, or a caller's own driver context) has a new id and gets
// its own lookup.  All calls in a context share the one array and it keeps
// the last call's contents: the align kernels write every workspace entry
// they later read, so nothing needs clearing, but calls that overlap on the
// GPU (on different streams, or from different host threads without
// ordering) race on the array and must not be issued.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "moe_lora.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = MOE_LORA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxContexts = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name) {
  void *ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(ptr);
  return nullptr;
}

// Unique id of the current context (ids are never reused within a process).
bool current_context_id(unsigned long long *id) {
  static const CtxGetCurrentFn get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_ctx || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_static_workspace in the current context, looked up
// once per context.  Returns nullptr on failure.
void *static_workspace_address() {
  static std::mutex mu;
  static unsigned long long ids[kMaxContexts];
  static void *addr[kMaxContexts];
  static int n = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  unsigned long long id = 0;
  if (!current_context_id(&id)) {
    // no context current yet: the lookup below makes the device's primary
    // context current, then the id is read again
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) return nullptr;
    if (!current_context_id(&id)) return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (ids[i] == id) return addr[i];
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) return nullptr;
  if (n < kMaxContexts) {
    ids[n] = id;
    addr[n] = p;
    ++n;
  }
  return p;
}

}  // namespace

extern "C" int moe_lora_align_static_workspace(const int32_t *topk_ids, const int32_t *token_lora_mapping,
                                               const int32_t *lora_ids, const int32_t *adapter_enabled, int M,
                                               int topk, int num_experts, int max_loras, int num_active_loras,
                                               int block_size, int32_t *sorted_token_ids, int32_t *expert_ids,
                                               int32_t *num_tokens_post_padded, int max_num_tokens_padded,
                                               int max_num_m_blocks, int32_t *err_flag, void *stream) {
  // the argument errors of moe_lora_align come first, then the size limit
  if (int st = moe_lora::check_align_args(topk_ids, token_lora_mapping, lora_ids, M, topk, num_experts, max_loras,
                                          num_active_loras, block_size, sorted_token_ids, expert_ids,
                                          num_tokens_post_padded, max_num_tokens_padded, max_num_m_blocks,
                                          MOE_LORA_ALIGN_GLOBAL))
    return st;
  const size_t need = moe_lora_align_workspace_bytes(M, topk, num_experts, num_active_loras, block_size,
                                                     MOE_LORA_ALIGN_GLOBAL);
  if (need > kStaticWorkspaceBytes) return MOE_LORA_ERR_WORKSPACE;  // beyond the built-in scratch
  void *ws = nullptr;
  if (num_active_loras > 0) {
    ws = static_workspace_address();
    if (!ws) return MOE_LORA_ERR_DEVICE;
  }
  return moe_lora_align(topk_ids, token_lora_mapping, lora_ids, adapter_enabled, M, topk, num_experts, max_loras,
                        num_active_loras, block_size, sorted_token_ids, expert_ids, num_tokens_post_padded,
                        max_num_tokens_padded, max_num_m_blocks, ws, kStaticWorkspaceBytes, MOE_LORA_ALIGN_GLOBAL,
                        err_flag, stream);
}
