/*
 * moe_lora.h -- C ABI of the GB300 (sm_103a) multi-LoRA Mixture-of-Experts
 * adapter library (libmoe_lora.so).
 *
 * Two stages make up the path:
 *
 *   moe_lora_align                 -- per active LoRA slot, group the
 *       (token, top-k) pairs by expert into block_size-padded segments.
 *       Defined by vLLM PR #29257 "Lora MoE Align Improvements", section
 *       Purpose (a per-LoRA align kernel with a shared-memory variant and a
 *       global-memory variant for large num_experts, sharing one align routine
 *       with the non-LoRA case) and its review thread (token_lora_mapping dtype;
 *       num_experts must not exceed 1024).  Output rows are per LoRA slot, as in
 *       the `.view(max_loras, -1)` of sorted_token_ids / expert_ids in the test
 *       diff of vLLM PR #32005 "Reduce the kernel overhead when num of active
 *       loras is smaller than max loras", tests/lora/test_fused_moe_lora_kernel.py.
 *
 *   moe_lora_fused_shrink_expand   -- y[m,k,:] (+)= (x[m] . A[l,e]^T) . B[l,e]^T
 *       with l = token_lora_mapping[m], e = topk_ids[m,k], the rank-r
 *       intermediate never written to global memory.  Defined by the
 *       prhub.com.cn summary of vLLM PR #42290 (one-shot fused MoE LoRA kernel
 *       and dual-stream execution), sections "Features and motivation" and
 *       "Implementation breakdown" step 1 (shrink and expand in one kernel, the
 *       rank dimension kept on chip, add_inputs choosing accumulate or
 *       overwrite) and "Key source snippets" (rank <= 128 for the one-shot
 *       kernel).  The grid is sized by num_active_loras, not max_loras, as in
 *       vLLM PR #32005, diff of vllm/lora/ops/triton_ops/fused_moe_lora_op.py
 *       (_adjust_kernel_inputs).
 *
 * Conventions for every entry point:
 *   - Pointers marked [device] must be device pointers of the current CUDA
 *     device; [host] are host pointers.  bf16 tensors are passed as
 *     moe_lora_bf16 (raw IEEE bfloat16 bit patterns, uint16).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).  Nothing is synchronised.
 *   - The caller owns every buffer.  The library allocates no memory, keeps
 *     no per-call state between calls and may be called from several host
 *     threads (moe_lora_align_static_workspace, below, is the one exception:
 *     it runs on a scratch buffer built into the library).
 *   - Return value: MOE_LORA_OK, or a moe_lora_status error code.  On an
 *     argument error nothing is enqueued.  Errors the device detects
 *     (out-of-range ids in device arrays, a wait that timed out) are OR-ed
 *     as MOE_LORA_DEVERR_* bits into *err_flag (an int32 [device] word, may be
 *     NULL), readable after the stream has synchronised; the offending entry is
 *     skipped, never dereferenced.
 *   - Every (token, top-k) pair is named by its flat index f = m*topk + k.
 *   - A fused call may start while the align call before it on the same
 *     stream is finishing (programmatic dependent launch); it reads the
 *     align's outputs only after that kernel has completed, and lora_ids /
 *     adapter_enabled, which the align does not write, possibly earlier.
 */
#ifndef MOE_LORA_H
#define MOE_LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_lora_bf16;

typedef enum {
    MOE_LORA_OK = 0,
    MOE_LORA_ERR_INVALID_ARG = 1,   /* NULL pointer, negative or inconsistent size */
    MOE_LORA_ERR_UNSUPPORTED = 2,   /* rank > 128, num_experts > 1024, bad block_size, ... */
    MOE_LORA_ERR_MISALIGNED = 3,    /* a pointer or a row is not 16-byte aligned */
    MOE_LORA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
    MOE_LORA_ERR_LAUNCH = 5,        /* a CUDA launch or attribute call failed */
    MOE_LORA_ERR_DEVICE = 6         /* the current device is not compute capability 10.3 (sm_103) */
} moe_lora_status;

/* Bits OR-ed into *err_flag by the kernels. */
#define MOE_LORA_DEVERR_EXPERT_ID 0x1   /* topk_ids / expert_ids entry outside [0, num_experts) */
#define MOE_LORA_DEVERR_LORA_ID 0x2     /* lora_ids entry outside [0, max_loras) */
#define MOE_LORA_DEVERR_CAPACITY 0x4    /* align output larger than max_num_tokens_padded */
#define MOE_LORA_DEVERR_PAIR_ID 0x8     /* sorted_token_ids entry neither a pair nor the sentinel
                                           (the streaming kernel also flags a block whose pairs
                                           do not all precede its sentinels) */
#define MOE_LORA_DEVERR_TIMEOUT 0x10    /* an on-chip wait gave up (a bounded wait ran out) */

/* Align variants (moe_lora_align `variant`). */
#define MOE_LORA_ALIGN_AUTO 0
#define MOE_LORA_ALIGN_SMEM 1     /* one CTA per active slot, counters in shared memory */
#define MOE_LORA_ALIGN_GLOBAL 2   /* many CTAs per slot, counters in the caller's workspace */
#define MOE_LORA_ALIGN_CLUSTER 3  /* a thread-block cluster of up to 8 CTAs per slot in one launch,
                                     counts exchanged through distributed shared memory (no workspace) */

/* Fused paths (moe_lora_fused_shrink_expand `path`). */
#define MOE_LORA_PATH_AUTO 0
#define MOE_LORA_PATH_CUDA_CORE 1 /* decode-sized blocks on CUDA cores (the cluster kernel below) */
#define MOE_LORA_PATH_TCGEN05 2   /* prefill-sized blocks: tcgen05 tensor-core MMAs */
#define MOE_LORA_PATH_CUDA_CORE_CLUSTER 3 /* CUDA cores: a thread-block cluster per block, K split over
                                             its CTAs, partial t summed through distributed shared memory */
#define MOE_LORA_PATH_CUDA_CORE_STREAM 4  /* CUDA cores: persistent thread-block clusters stream each
                                             block's adapters through a ring of TMA stages, K split over
                                             the cluster's CTAs for the shrink (partial t pushed through
                                             distributed shared memory), N split for the expand
                                             (rank 8, 16, 32, 64 or 128) */

/* Capacity of one LoRA row of sorted_token_ids: every pair once plus up to
 * block_size-1 padding slots for each expert: M*topk + num_experts*(block_size-1).
 * Returns -1 on invalid sizes. */
int moe_lora_max_num_tokens_padded(int M, int topk, int num_experts, int block_size);

/* Capacity of one LoRA row of expert_ids: ceil(max_num_tokens_padded / block_size).
 * Returns -1 on invalid sizes. */
int moe_lora_max_num_m_blocks(int M, int topk, int num_experts, int block_size);

/* The align variant a call with these sizes runs: MOE_LORA_ALIGN_SMEM,
 * MOE_LORA_ALIGN_GLOBAL or MOE_LORA_ALIGN_CLUSTER (never AUTO), or a negative
 * moe_lora_status code for invalid sizes or a variant these sizes do not fit.
 * Host only; no device is touched. */
int moe_lora_align_resolve_variant(int M, int topk, int num_experts, int variant);

/* Bytes of [device] workspace moe_lora_align needs for `variant` (0 for the
 * shared-memory and cluster variants; for AUTO, the size of whichever variant
 * AUTO picks for these sizes).  Returns 0 and the call needs no workspace
 * when it is 0.  AUTO picks the cluster variant for num_experts >= 256 or at
 * least 16384 pairs, and the shared-memory variant otherwise. */
size_t moe_lora_align_workspace_bytes(int M, int topk, int num_experts,
                                      int num_active_loras, int block_size, int variant);

/*
 * moe_lora_align -- group the pairs of each active LoRA slot by expert.
 *
 * For each z < num_active_loras, with l = lora_ids[z] (distinct, in
 * [0, max_loras)):
 *   cnt[e]  = number of pairs f with token_lora_mapping[f / topk] == l and
 *             topk_ids[f] == e;
 *   off[e]  = sum_{e' < e} ceil(cnt[e'] / block_size) * block_size;
 *   num_tokens_post_padded[l] = off[num_experts];
 *   sorted_token_ids[l][off[e] ...] = the pairs of expert e in ascending f,
 *       followed by the sentinel M*topk up to the next multiple of block_size;
 *   expert_ids[l][b] = e for every block b in [off[e], off[e+1]) / block_size.
 * Experts with no pair get no block.  Tokens mapped to -1, or to a slot that
 * is not in lora_ids, are dropped.  A slot whose adapter is disabled
 * (adapter_enabled[l] == 0) gets num_tokens_post_padded[l] = 0.  Pairs whose
 * expert is outside [0, num_experts) are dropped and flagged
 * (MOE_LORA_DEVERR_EXPERT_ID).  Only num_tokens_post_padded[l] for active l,
 * sorted_token_ids[l][0, ntpp) and expert_ids[l][0, ntpp / block_size) are
 * written; every other entry keeps its previous contents.  The result is
 * deterministic and identical for both variants.
 *
 *   topk_ids               [device] int32 [M, topk]
 *   token_lora_mapping     [device] int32 [M], -1 = no adapter
 *   lora_ids               [device] int32 [num_active_loras]
 *   adapter_enabled        [device] int32 [max_loras], or NULL = all enabled
 *   sorted_token_ids       [device] int32 [max_loras, max_num_tokens_padded]
 *   expert_ids             [device] int32 [max_loras, max_num_m_blocks]
 *   num_tokens_post_padded [device] int32 [max_loras]
 *   workspace              [device] >= moe_lora_align_workspace_bytes(..., variant)
 *                          bytes, 16-byte aligned; may be NULL when that is 0.
 *                          Its contents need no initialisation and are
 *                          overwritten.
 * Sizes: 1 <= topk <= num_experts <= 1024; block_size in {16, 32, 64, 128};
 * 0 <= num_active_loras <= max_loras; M >= 0 (M == 0 or num_active_loras == 0
 * writes num_tokens_post_padded[l] = 0 for each listed slot, or nothing when
 * the list is empty); max_num_tokens_padded / max_num_m_blocks must be at
 * least the capacities returned above.
 */
int moe_lora_align(const int32_t *topk_ids, const int32_t *token_lora_mapping,
                   const int32_t *lora_ids, const int32_t *adapter_enabled,
                   int M, int topk, int num_experts, int max_loras,
                   int num_active_loras, int block_size,
                   int32_t *sorted_token_ids, int32_t *expert_ids,
                   int32_t *num_tokens_post_padded,
                   int max_num_tokens_padded, int max_num_m_blocks,
                   void *workspace, size_t workspace_bytes,
                   int variant, int32_t *err_flag, void *stream);

/*
 * moe_align_block_size -- the plain (non-LoRA) MoE align: group all (token,
 * top-k) pairs by expert into block_size-padded segments.  It is the
 * single-slot case of moe_lora_align (one routine serves the LoRA and the
 * non-LoRA callers: vLLM PR #29257, section Purpose): every token belongs to
 * the one slot, whose row is row 0.  Same output rules as moe_lora_align with
 * max_loras = num_active_loras = 1:
 *   sorted_token_ids [device] int32 [max_num_tokens_padded]
 *   expert_ids       [device] int32 [max_num_m_blocks]
 *   num_tokens_post_padded [device] int32 [1]
 * workspace: moe_lora_align_workspace_bytes(M, topk, num_experts, 1,
 * block_size, variant) bytes, [device], 16-byte aligned (may be NULL when
 * that is 0).  Limits and errors as for moe_lora_align.
 */
int moe_align_block_size(const int32_t *topk_ids, int M, int topk, int num_experts, int block_size,
                         int32_t *sorted_token_ids, int32_t *expert_ids, int32_t *num_tokens_post_padded,
                         int max_num_tokens_padded, int max_num_m_blocks,
                         void *workspace, size_t workspace_bytes, int variant,
                         int32_t *err_flag, void *stream);

/*
 * moe_lora_fused_shrink_expand -- apply each covered pair's adapter.
 *
 * Reads the align outputs of the same slots and, for every block b of every
 * active slot z (l = lora_ids[z], b < num_tokens_post_padded[l] / block_size)
 * with e = expert_ids[l][b] and every pair f = sorted_token_ids[l][b*block_size + i]
 * that is not the sentinel M*topk (m = f / topk):
 *   t[j]      = sum_k x[m][k] * A[l][e][j][k]                 (j < rank, fp32)
 *   y[f][n]   = bf16( (add_inputs ? y[f][n] : 0) + sum_j B[l][e][n][j] * t[j] )
 * t stays in registers / shared memory / tensor memory.  Pairs of slots that
 * are not listed, disabled, or not covered are not touched (in both modes).
 * Tensor-core path: t enters the second product as two bf16 terms,
 * t_hi = bf16(t) and t_lo = bf16(t - t_hi), which keeps fp32-level accuracy.
 *
 *   x                [device] bf16 [M, K] row-major
 *   lora_a           [device] bf16 [max_loras, num_experts, rank, K]
 *   lora_b           [device] bf16 [max_loras, num_experts, N, rank]
 *   y                [device] bf16 [M, topk, N], read (if add_inputs) and written
 *   sorted_token_ids, expert_ids, num_tokens_post_padded: as written by moe_lora_align
 *                    with the same M, topk, num_experts, block_size and capacities
 *   lora_ids         [device] int32 [num_active_loras]
 *   adapter_enabled  [device] int32 [max_loras] or NULL
 * Sizes: 1 <= rank <= 128 with rank % 4 == 0 (the tensor-core path needs
 * rank % 8 == 0); K % 8 == 0 and N % 8 == 0; x, lora_a, lora_b, y 16-byte
 * aligned; other limits as for moe_lora_align.  The tensor-core and
 * streaming paths also need num_active_loras <= 128.
 * path: MOE_LORA_PATH_*.  AUTO picks
 *   - the tensor-core path (when it takes the sizes) for batches of at least
 *     1024 pairs;
 *   - for smaller batches whose adapters, by the block bound (block bound
 *     times (K + N) * rank * 2 bytes per slice), exceed 48 MB: the cluster
 *     streaming kernel (MOE_LORA_PATH_CUDA_CORE_STREAM) for ranks 8, 16, 32,
 *     64 and 128, else the tensor-core path;
 *   - otherwise the one-cluster-per-block kernel
 *     (MOE_LORA_PATH_CUDA_CORE_CLUSTER) -- unless it cannot hold a CTA's
 *     share of the adapter rows in shared memory (long N * rank or K * rank
 *     rows), in which case the tensor-core path when K >= 64 and N >= 32, else
 *     the streaming kernel.
 * Shapes no kernel takes return MOE_LORA_ERR_UNSUPPORTED.
 * MOE_LORA_PATH_CUDA_CORE runs MOE_LORA_PATH_CUDA_CORE_CLUSTER.
 */
int moe_lora_fused_shrink_expand(const moe_lora_bf16 *x, const moe_lora_bf16 *lora_a,
                                 const moe_lora_bf16 *lora_b, moe_lora_bf16 *y,
                                 const int32_t *sorted_token_ids, const int32_t *expert_ids,
                                 const int32_t *num_tokens_post_padded,
                                 const int32_t *lora_ids, const int32_t *adapter_enabled,
                                 int M, int topk, int num_experts, int K, int N, int rank,
                                 int max_loras, int num_active_loras, int block_size,
                                 int max_num_tokens_padded, int max_num_m_blocks,
                                 int add_inputs, int path, int32_t *err_flag, void *stream);

/* Most adapter slices one moe_lora_fused_shrink_expand_ex call takes. */
#define MOE_LORA_MAX_SLICES 4

/*
 * moe_lora_fused_shrink_expand_ex -- moe_lora_fused_shrink_expand with the
 * options the fused MoE-LoRA op carries around the same computation
 * (mul_routed_weight / topk_weights and the output `offset` in the diff of
 * vLLM PR #32005 to fused_moe_lora_op.py; the w13 / w2 stages of the
 * prhub.com.cn summary of vLLM PR #42290, step 2):
 *   - x_per_pair: x is [M*topk, K] and pair f reads row f (the w2 stage,
 *     whose input is one activation row per pair); otherwise x is [M, K] and
 *     pair f reads row f / topk;
 *   - num_slices (1..MOE_LORA_MAX_SLICES) adapter slices per layer (the
 *     separate gate and up adapters of w13): slice s has its own A_s, B_s and
 *     rank-r intermediate t_s, and writes output columns
 *     y_offset + s*N + n (n < N) of y rows that are ldy elements long;
 *   - topk_weights: when not NULL, the delta of pair f is multiplied by
 *     topk_weights[f] before it is added (mul_routed_weight):
 *         y[f][y_offset + s*N + n] =
 *             bf16( (add_inputs ? y_in : 0) + w[f] * sum_j B_s[l][e][n][j] * t_s[j] )
 *     The weight scales the delta only, never y_in.
 * Columns no slice writes are never touched.
 *
 *   x                [device] bf16 [M, K], or [M*topk, K] when x_per_pair
 *   lora_a, lora_b   [host] arrays of num_slices [device] pointers, each as in
 *                    moe_lora_fused_shrink_expand (same shapes for every slice);
 *                    the host arrays are read during the call only
 *   y                [device] bf16 [M, topk, ldy]
 *   topk_weights     [device] fp32 [M, topk], or NULL
 * Sizes: ldy % 8 == 0, y_offset % 8 == 0, y_offset + num_slices*N <= ldy;
 * the rest as for moe_lora_fused_shrink_expand, which is this call with
 * x_per_pair = 0, one slice, ldy = N, y_offset = 0 and no weights.
 */
int moe_lora_fused_shrink_expand_ex(const moe_lora_bf16 *x, int x_per_pair,
                                    const moe_lora_bf16 *const *lora_a,
                                    const moe_lora_bf16 *const *lora_b, int num_slices,
                                    moe_lora_bf16 *y, int ldy, int y_offset,
                                    const float *topk_weights,
                                    const int32_t *sorted_token_ids, const int32_t *expert_ids,
                                    const int32_t *num_tokens_post_padded,
                                    const int32_t *lora_ids, const int32_t *adapter_enabled,
                                    int M, int topk, int num_experts, int K, int N, int rank,
                                    int max_loras, int num_active_loras, int block_size,
                                    int max_num_tokens_padded, int max_num_m_blocks,
                                    int add_inputs, int path, int32_t *err_flag, void *stream);

/*
 * moe_lora_fused_shrink_expand_naive -- the general fused call without the
 * align stage (naive block assignment: the one-shot kernel's grid of
 * (num_tokens * top_k, num_slices, num_active_loras) programs, one per pair,
 * in the prhub.com.cn summary of vLLM PR #42290, "Key source snippets"; the
 * early-exit and zero-grid cases of its tests, "Implementation breakdown"
 * step 4).  Each (token, top-k) pair f is its own work item: l =
 * token_lora_mapping[f / topk], e = topk_ids[f]; the pair is covered when l is
 * one of lora_ids[0, num_active_loras), its adapter is enabled and
 * 0 <= e < num_experts, and then gets exactly the update of
 * moe_lora_fused_shrink_expand_ex.  Uncovered pairs exit at once and are not
 * touched.  A covered token with an expert id outside [0, num_experts) is
 * reported as MOE_LORA_DEVERR_EXPERT_ID, a lora_ids entry outside
 * [0, max_loras) as MOE_LORA_DEVERR_LORA_ID.  Pairs that share an adapter
 * each read it (from L2 after the first), so this path suits batches with
 * few pairs per (LoRA, expert), i.e. decode.  Runs on CUDA cores:
 *   path  MOE_LORA_PATH_CUDA_CORE_CLUSTER or MOE_LORA_PATH_CUDA_CORE (one
 *         cluster per pair, the whole share of A and B in shared memory;
 *         shapes whose rows it cannot hold return MOE_LORA_ERR_UNSUPPORTED),
 *         MOE_LORA_PATH_CUDA_CORE_STREAM (persistent CTAs streaming each
 *         pair's adapters; rank 8, 16, 32, 64 or 128), or MOE_LORA_PATH_AUTO:
 *         the streaming kernel when the pairs' adapters (M * topk * slices *
 *         (K + N) * rank * 2 bytes) exceed 48 MB and it takes the rank, else
 *         the one-cluster-per-pair kernel.  MOE_LORA_PATH_TCGEN05 is not
 *         valid here.
 *
 *   topk_ids          [device] int32 [M, topk]
 *   token_lora_mapping [device] int32 [M] (-1: no adapter)
 *   the rest as for moe_lora_fused_shrink_expand_ex.
 */
int moe_lora_fused_shrink_expand_naive(const moe_lora_bf16 *x, int x_per_pair,
                                       const moe_lora_bf16 *const *lora_a,
                                       const moe_lora_bf16 *const *lora_b, int num_slices,
                                       moe_lora_bf16 *y, int ldy, int y_offset,
                                       const float *topk_weights, const int32_t *topk_ids,
                                       const int32_t *token_lora_mapping, const int32_t *lora_ids,
                                       const int32_t *adapter_enabled, int M, int topk,
                                       int num_experts, int K, int N, int rank, int max_loras,
                                       int num_active_loras, int add_inputs, int path,
                                       int32_t *err_flag, void *stream);

/*
 * moe_lora_test_withheld_copy -- a test of the library's bounded waits, not
 * for production use.  The pages have no counterpart: it exists so that a
 * test can make one of the kernels' on-chip waits run out without faulting or
 * hanging the GPU.  It is moe_lora_fused_shrink_expand_naive on the
 * one-cluster-per-pair kernel (MOE_LORA_PATH_CUDA_CORE_CLUSTER), except that
 * no CTA issues the bulk copy of its slice of B[l][e], whose arrival it then
 * waits for with a limit of wait_limit_ns nanoseconds (1000 .. 4e9) instead
 * of 4 s.  Every CTA that reaches a covered pair's wait gives up after the
 * limit, ORs MOE_LORA_DEVERR_TIMEOUT into *err_flag, requests no further
 * copy, runs its remaining control flow (its cluster barriers stay balanced)
 * and exits; the call completes.  No copy is in flight when a CTA exits (the
 * withheld one was never issued), so the device stays usable.  The covered
 * pairs' output columns are left in an unspecified state; everything else in
 * y is untouched.  Arguments and argument errors as for the naive entry point,
 * plus MOE_LORA_ERR_INVALID_ARG for a limit outside the range.
 */
int moe_lora_test_withheld_copy(const moe_lora_bf16 *x, int x_per_pair,
                                const moe_lora_bf16 *const *lora_a,
                                const moe_lora_bf16 *const *lora_b, int num_slices,
                                moe_lora_bf16 *y, int ldy, int y_offset,
                                const float *topk_weights, const int32_t *topk_ids,
                                const int32_t *token_lora_mapping, const int32_t *lora_ids,
                                const int32_t *adapter_enabled, int M, int topk,
                                int num_experts, int K, int N, int rank, int max_loras,
                                int num_active_loras, int add_inputs,
                                unsigned long long wait_limit_ns, int32_t *err_flag,
                                void *stream);

/*
 * moe_lora_fused_resolve_path -- the kernel a fused call with these sizes
 * runs: MOE_LORA_PATH_TCGEN05, MOE_LORA_PATH_CUDA_CORE_CLUSTER or
 * MOE_LORA_PATH_CUDA_CORE_STREAM (never AUTO or CUDA_CORE), or a negative
 * moe_lora_status code if `path` is not valid for these sizes.  Host only; no
 * device is touched: where AUTO depends on shared memory it assumes the
 * 227 KB per block of compute capability 10.3.
 */
int moe_lora_fused_resolve_path(int M, int topk, int num_experts, int K, int N, int rank,
                                int num_active_loras, int block_size, int num_slices, int path);

/*
 * moe_lora_fused_naive_resolve_path -- the kernel a naive-assignment call
 * (moe_lora_fused_shrink_expand_naive / _ex) with these sizes runs:
 * MOE_LORA_PATH_CUDA_CORE_CLUSTER or MOE_LORA_PATH_CUDA_CORE_STREAM, or a
 * negative moe_lora_status code if `path` (AUTO, CUDA_CORE, CUDA_CORE_CLUSTER
 * or CUDA_CORE_STREAM) is not valid for these sizes.  Host only; no device is
 * touched.
 */
int moe_lora_fused_naive_resolve_path(int M, int topk, int num_experts, int K, int N, int rank,
                                      int num_active_loras, int num_slices, int path);

/*
 * moe_lora_fused_plan -- the launch plan a plain fused call with these sizes
 * would use on a device with `sm_count` SMs and `max_smem_per_block` bytes of
 * opt-in shared memory per block.  Host arithmetic only; no device is
 * touched.  For inspection and tests.
 *
 *   out  [host] int32 [11]: kernel (MOE_LORA_PATH_TCGEN05 or
 *        MOE_LORA_PATH_CUDA_CORE_CLUSTER), grid (0 for the cluster kernel:
 *        capped at run time by the clusters that can be resident at once),
 *        threads per CTA, dynamic shared memory bytes, then for the tensor-core
 *        kernel the shrink ring depth, the shrink producers' lag, the expand
 *        ring depth, the T buffers and the TMEM columns, and for the cluster
 *        kernel the CTAs per cluster and the pairs per group (block_size for
 *        the tensor-core kernel).
 * Returns a moe_lora_status code (MOE_LORA_ERR_UNSUPPORTED for the CUDA-core
 * streaming kernel, which has no plan here).  On a GB300 every tensor-core
 * plan has at least two expand stages except block_size 128 with rank > 64,
 * where only one fits beside the shrink stages and the T buffer.
 */
int moe_lora_fused_plan(int M, int topk, int num_experts, int K, int N, int rank,
                        int num_active_loras, int block_size, int num_slices, int path,
                        int sm_count, int max_smem_per_block, int32_t *out);

/* Size of the scratch buffer built into the library for
 * moe_lora_align_static_workspace (4 MiB). */
#define MOE_LORA_STATIC_WORKSPACE_BYTES ((size_t)4 << 20)

/*
 * moe_lora_align_static_workspace -- moe_lora_align (global-memory variant)
 * for callers that cannot allocate device memory.
 *
 * vLLM's align has no counterpart to this entry point; it exists for callers
 * that may not call cudaMalloc or any allocating routine where they align
 * (code running under an allocator that forbids device allocations there,
 * plugins that are handed only their input and output buffers, processes that
 * must not grow device memory after start-up).  They pass the same inputs and
 * outputs as to moe_lora_align; the workspace is a MOE_LORA_STATIC_WORKSPACE_BYTES
 * buffer compiled into the library (every GPU that loads the library holds it
 * until the process exits).  Nothing is allocated by this call.
 *   - Same arguments, results and errors as moe_lora_align with
 *     variant = MOE_LORA_ALIGN_GLOBAL, minus the workspace arguments.  Those
 *     argument checks come first; then it returns MOE_LORA_ERR_WORKSPACE when
 *     moe_lora_align_workspace_bytes(M, topk, num_experts, num_active_loras,
 *     block_size, MOE_LORA_ALIGN_GLOBAL) exceeds MOE_LORA_STATIC_WORKSPACE_BYTES.
 *   - The first call in each CUDA context (normally once per device, in the
 *     runtime's primary context), with that context current, looks up the
 *     buffer's device address; make that first call before any stream
 *     capture.  A new context (after cudaDeviceReset, or a caller's own
 *     driver context) gets a lookup of its own on its first call.
 *   - All calls in a context share the one buffer, which keeps the last call's
 *     contents (no entry needs clearing between calls).  Calls that overlap on
 *     the GPU -- on different streams, or from host threads without ordering
 *     between them -- race on it and must not be issued.
 */
int moe_lora_align_static_workspace(const int32_t *topk_ids, const int32_t *token_lora_mapping,
                                    const int32_t *lora_ids, const int32_t *adapter_enabled,
                                    int M, int topk, int num_experts, int max_loras,
                                    int num_active_loras, int block_size,
                                    int32_t *sorted_token_ids, int32_t *expert_ids,
                                    int32_t *num_tokens_post_padded,
                                    int max_num_tokens_padded, int max_num_m_blocks,
                                    int32_t *err_flag, void *stream);

/* Human-readable name of a moe_lora_status value (static string). */
const char *moe_lora_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int moe_lora_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LORA_H */
