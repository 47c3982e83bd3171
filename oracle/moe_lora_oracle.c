/*
 * moe_lora_oracle.c -- plain, slow, single-threaded CPU oracle for the
 * multi-LoRA Mixture-of-Experts adapter path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library under lora_moe_gb300/) neither links nor calls it, and this file
 * shares no code, header, table or helper with that path.
 *
 * What it computes, and where the definition comes from:
 *
 *  1. oracle_moe_lora_align: for every active LoRA slot, count the
 *     (token, top-k) pairs routed to each expert, pad each count up to a
 *     multiple of block_size, prefix-sum the padded counts into segment
 *     offsets, and scatter the pair indices into their expert segments.
 *     Sources: vLLM PR #29257 "Lora MoE Align Improvements", section Purpose
 *     (the per-LoRA align kernel, its shared-memory and global-memory
 *     variants, and the common align routine that serves LoRA and non-LoRA
 *     callers); its review thread (the token_lora_mapping dtype and the
 *     num_experts <= 1024 check).  The per-LoRA row view of the outputs is the
 *     `.view(max_loras, -1)` of sorted_token_ids / expert_ids in the test diff
 *     of vLLM PR #32005 "Reduce the kernel overhead when num of active loras is
 *     smaller than max loras", file tests/lora/test_fused_moe_lora_kernel.py.
 *     Readings where the pages are silent (each is listed in the design notes):
 *       - a pair is identified by its flat index f = m*topk + k;
 *       - within a segment, pairs appear in ascending f;
 *       - segments appear in ascending expert id; an expert with no pair gets
 *         no block;
 *       - padding slots hold the sentinel M*topk;
 *       - tokens whose LoRA is -1, or not in the active set, are dropped;
 *       - pairs whose expert id is outside [0, E) are dropped (and reported);
 *       - a disabled adapter gets num_tokens_post_padded = 0.
 *     Only num_tokens_post_padded[l] for active l, sorted_token_ids[l][0, ntpp)
 *     and expert_ids[l][0, ntpp/block_size) are defined; nothing else is
 *     written.
 *
 *  2. oracle_moe_lora_fused: the plain definition of the fused shrink+expand
 *     (prhub.com.cn summary of vLLM PR #42290, sections "Features and
 *     motivation" and "Implementation breakdown" step 1: shrink by lora_a,
 *     expand by lora_b, rank-r intermediate kept on chip, optional
 *     accumulation into the output via add_inputs):
 *         for every covered pair (m, k), l = token_lora_mapping[m],
 *         e = topk_ids[m][k]:
 *           t[j]       = sum_kk x[m][kk] * A[l][e][j][kk]            (j < r)
 *           ref[m][k][n] = (add_inputs ? y_in[m][k][n] : 0)
 *                          + sum_j B[l][e][n][j] * t[j]
 *         uncovered pairs keep y_in in both modes.
 *     A pair is covered iff l >= 0, l is one of lora_ids[0, num_active_loras),
 *     its adapter is enabled (adapter_enabled == NULL means all enabled), and
 *     0 <= e < E.  All arithmetic is fp64 over the exact bf16 input values;
 *     nothing is rounded to bf16.
 *
 *  3. oracle_moe_lora_fused_sampled: the same definition evaluated only at a
 *     caller-chosen list of pairs and output columns, for checks at full size.
 *
 *  4. oracle_moe_lora_fused_ex: the same definition with the options the
 *     pages name around it: router-weight scaling (mul_routed_weight with
 *     topk_weights, prhub.com.cn summary of vLLM PR #42290, step 2, and the
 *     mul_routed_weight / offset arguments in the diff of vLLM PR #32005 to
 *     fused_moe_lora_op.py), input rows per pair (the w2 stage's input is one
 *     activation row per (token, expert) pair), several adapter slices per
 *     layer (num_slices; the gate and up projections of w13 each have their
 *     own A and B) and an output column offset.  Readings where the pages are
 *     silent:
 *       - the router weight multiplies the LoRA delta only, not y_in:
 *             out = (add_inputs ? y_in : 0) + w[f] * sum_j B[n][j] * t[j];
 *       - with x_per_pair, the input row of pair f is row f of x
 *         ([M*topk][K]); otherwise row m = f / topk of x ([M][K]);
 *       - slice s has its own A_s [L][E][r][K] and B_s [L][E][N][r] and its
 *         own rank-r intermediate t_s; its N columns land at output columns
 *         y_offset + s*N + n of a row of ldy columns;
 *       - output columns that no slice writes keep y_in (either mode), and
 *         uncovered pairs keep their whole row.
 *     It can evaluate all pairs or a caller-chosen list of pairs.
 *
 * Layouts (row-major, bf16 carried as raw uint16 bit patterns):
 *   topk_ids [M][topk] int32, token_lora_mapping [M] int32, lora_ids
 *   [num_active_loras] int32, x [M][K], lora_a [max_loras][E][r][K],
 *   lora_b [max_loras][E][N][r], y_in [M][topk][N], ref [M][topk][N] double.
 *
 * Build: gcc -O2 -ffp-contract=off (no fused multiply-add, so that x86 and
 * Arm hosts round identically).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status bits returned by the oracle functions. */
#define ORACLE_BAD_EXPERT_ID 1   /* a covered token routed to an expert outside [0, E) */
#define ORACLE_BAD_LORA_ID 2     /* lora_ids[z] outside [0, max_loras) */
#define ORACLE_CAPACITY 4        /* output would exceed max_num_tokens_padded / max_num_m_blocks */
#define ORACLE_NOMEM 8

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int slot_is_active(int l, const int32_t *lora_ids, int num_active_loras)
{
    for (int z = 0; z < num_active_loras; ++z)
        if (lora_ids[z] == l)
            return 1;
    return 0;
}

int oracle_moe_lora_align(const int32_t *topk_ids, const int32_t *token_lora_mapping,
                          const int32_t *lora_ids, const int32_t *adapter_enabled,
                          int M, int topk, int num_experts, int max_loras,
                          int num_active_loras, int block_size,
                          int32_t *sorted_token_ids, int32_t *expert_ids,
                          int32_t *num_tokens_post_padded,
                          int max_num_tokens_padded, int max_num_m_blocks)
{
    const int E = num_experts;
    const int num_pairs = M * topk;
    const int sentinel = num_pairs;
    int status = 0;
    int *count = malloc(sizeof(int) * (size_t)(E > 0 ? E : 1));
    int *offset = malloc(sizeof(int) * (size_t)(E + 1));
    int *cursor = malloc(sizeof(int) * (size_t)(E > 0 ? E : 1));
    if (!count || !offset || !cursor) {
        free(count); free(offset); free(cursor);
        return ORACLE_NOMEM;
    }

    for (int z = 0; z < num_active_loras; ++z) {
        const int l = lora_ids[z];
        if (l < 0 || l >= max_loras) {
            status |= ORACLE_BAD_LORA_ID;
            continue;
        }
        int32_t *sorted = sorted_token_ids + (int64_t)l * max_num_tokens_padded;
        int32_t *experts = expert_ids + (int64_t)l * max_num_m_blocks;
        if (adapter_enabled && !adapter_enabled[l]) {
            num_tokens_post_padded[l] = 0;
            continue;
        }

        /* Count: pairs of this LoRA per expert. */
        for (int e = 0; e < E; ++e)
            count[e] = 0;
        for (int f = 0; f < num_pairs; ++f) {
            const int m = f / topk;
            if (token_lora_mapping[m] != l)
                continue;
            const int e = topk_ids[f];
            if (e < 0 || e >= E) {
                status |= ORACLE_BAD_EXPERT_ID;
                continue;
            }
            count[e] += 1;
        }

        /* Pad each count up to a multiple of block_size; exclusive prefix sum. */
        offset[0] = 0;
        for (int e = 0; e < E; ++e) {
            const int padded = (count[e] + block_size - 1) / block_size * block_size;
            offset[e + 1] = offset[e] + padded;
        }
        const int total = offset[E];
        num_tokens_post_padded[l] = total;
        if (total > max_num_tokens_padded || total / block_size > max_num_m_blocks) {
            status |= ORACLE_CAPACITY;
            continue;
        }

        /* Every slot of the segments starts as padding; each block names its expert. */
        for (int i = 0; i < total; ++i)
            sorted[i] = sentinel;
        for (int e = 0; e < E; ++e)
            for (int b = offset[e] / block_size; b < offset[e + 1] / block_size; ++b)
                experts[b] = e;

        /* Scatter pairs in ascending flat index into their expert's segment. */
        for (int e = 0; e < E; ++e)
            cursor[e] = offset[e];
        for (int f = 0; f < num_pairs; ++f) {
            const int m = f / topk;
            if (token_lora_mapping[m] != l)
                continue;
            const int e = topk_ids[f];
            if (e < 0 || e >= E)
                continue;
            sorted[cursor[e]] = f;
            cursor[e] += 1;
        }
    }
    free(count);
    free(offset);
    free(cursor);
    return status;
}

/* Is pair f covered?  On success writes the LoRA slot and expert. */
static int pair_is_covered(int f, const int32_t *topk_ids, const int32_t *token_lora_mapping,
                           const int32_t *lora_ids, const int32_t *adapter_enabled,
                           int topk, int num_experts, int max_loras, int num_active_loras,
                           int *l_out, int *e_out)
{
    const int m = f / topk;
    const int l = token_lora_mapping[m];
    const int e = topk_ids[f];
    if (l < 0 || l >= max_loras)
        return 0;
    if (!slot_is_active(l, lora_ids, num_active_loras))
        return 0;
    if (adapter_enabled && !adapter_enabled[l])
        return 0;
    if (e < 0 || e >= num_experts)
        return 0;
    *l_out = l;
    *e_out = e;
    return 1;
}

/* t[j] = sum_kk x[m][kk] * A[l][e][j][kk] for one pair. */
static void shrink_one_pair(const uint16_t *x_row, const uint16_t *a_le, int K, int rank, double *t)
{
    for (int j = 0; j < rank; ++j) {
        const uint16_t *a_row = a_le + (int64_t)j * K;
        double s = 0.0;
        for (int kk = 0; kk < K; ++kk)
            s += bf16_value(x_row[kk]) * bf16_value(a_row[kk]);
        t[j] = s;
    }
}

/* sum_j B[l][e][n][j] * t[j] for one output column. */
static double expand_one_column(const uint16_t *b_le, int n, int rank, const double *t)
{
    const uint16_t *b_row = b_le + (int64_t)n * rank;
    double s = 0.0;
    for (int j = 0; j < rank; ++j)
        s += bf16_value(b_row[j]) * t[j];
    return s;
}

int oracle_moe_lora_fused(const uint16_t *x, const uint16_t *lora_a, const uint16_t *lora_b,
                          const uint16_t *y_in, const int32_t *topk_ids,
                          const int32_t *token_lora_mapping, const int32_t *lora_ids,
                          const int32_t *adapter_enabled,
                          int M, int topk, int num_experts, int K, int N, int rank,
                          int max_loras, int num_active_loras, int add_inputs, double *ref)
{
    double *t = malloc(sizeof(double) * (size_t)(rank > 0 ? rank : 1));
    if (!t)
        return ORACLE_NOMEM;
    for (int f = 0; f < M * topk; ++f) {
        const int m = f / topk;
        const uint16_t *yin = y_in + (int64_t)f * N;
        double *out = ref + (int64_t)f * N;
        int l, e;
        if (!pair_is_covered(f, topk_ids, token_lora_mapping, lora_ids, adapter_enabled,
                             topk, num_experts, max_loras, num_active_loras, &l, &e)) {
            for (int n = 0; n < N; ++n)
                out[n] = bf16_value(yin[n]);
            continue;
        }
        const uint16_t *a_le = lora_a + ((int64_t)l * num_experts + e) * rank * K;
        const uint16_t *b_le = lora_b + ((int64_t)l * num_experts + e) * N * rank;
        shrink_one_pair(x + (int64_t)m * K, a_le, K, rank, t);
        for (int n = 0; n < N; ++n) {
            const double delta = expand_one_column(b_le, n, rank, t);
            out[n] = (add_inputs ? bf16_value(yin[n]) : 0.0) + delta;
        }
    }
    free(t);
    return 0;
}

int oracle_moe_lora_fused_sampled(const uint16_t *x, const uint16_t *lora_a,
                                  const uint16_t *lora_b, const uint16_t *y_in,
                                  const int32_t *topk_ids, const int32_t *token_lora_mapping,
                                  const int32_t *lora_ids, const int32_t *adapter_enabled,
                                  int M, int topk, int num_experts, int K, int N, int rank,
                                  int max_loras, int num_active_loras, int add_inputs,
                                  const int32_t *pairs, int num_sampled_pairs,
                                  const int32_t *columns, int num_sampled_columns,
                                  double *out /* [num_sampled_pairs][num_sampled_columns] */)
{
    (void)M;
    double *t = malloc(sizeof(double) * (size_t)(rank > 0 ? rank : 1));
    if (!t)
        return ORACLE_NOMEM;
    for (int i = 0; i < num_sampled_pairs; ++i) {
        const int f = pairs[i];
        const int m = f / topk;
        const uint16_t *yin = y_in + (int64_t)f * N;
        double *o = out + (int64_t)i * num_sampled_columns;
        int l, e;
        const int covered = pair_is_covered(f, topk_ids, token_lora_mapping, lora_ids,
                                            adapter_enabled, topk, num_experts, max_loras,
                                            num_active_loras, &l, &e);
        if (covered)
            shrink_one_pair(x + (int64_t)m * K,
                            lora_a + ((int64_t)l * num_experts + e) * rank * K, K, rank, t);
        for (int c = 0; c < num_sampled_columns; ++c) {
            const int n = columns[c];
            if (!covered) {
                o[c] = bf16_value(yin[n]);
                continue;
            }
            const double delta = expand_one_column(
                lora_b + ((int64_t)l * num_experts + e) * N * rank, n, rank, t);
            o[c] = (add_inputs ? bf16_value(yin[n]) : 0.0) + delta;
        }
    }
    free(t);
    return 0;
}

int oracle_moe_lora_fused_ex(const uint16_t *x, int x_per_pair,
                             const uint16_t *const *lora_a, const uint16_t *const *lora_b,
                             int num_slices, const uint16_t *y_in, int ldy, int y_offset,
                             const float *topk_weights, const int32_t *topk_ids,
                             const int32_t *token_lora_mapping, const int32_t *lora_ids,
                             const int32_t *adapter_enabled, int M, int topk, int num_experts,
                             int K, int N, int rank, int max_loras, int num_active_loras,
                             int add_inputs, const int32_t *pairs, int num_selected,
                             double *out /* [num_selected, or M*topk if pairs is NULL][ldy] */)
{
    double *t = malloc(sizeof(double) * (size_t)(rank > 0 ? rank : 1));
    if (!t)
        return ORACLE_NOMEM;
    const int rows = pairs ? num_selected : M * topk;
    for (int i = 0; i < rows; ++i) {
        const int f = pairs ? pairs[i] : i;
        const int m = f / topk;
        const uint16_t *yin = y_in + (int64_t)f * ldy;
        double *o = out + (int64_t)i * ldy;
        for (int c = 0; c < ldy; ++c)
            o[c] = bf16_value(yin[c]);
        int l, e;
        if (!pair_is_covered(f, topk_ids, token_lora_mapping, lora_ids, adapter_enabled,
                             topk, num_experts, max_loras, num_active_loras, &l, &e))
            continue;
        const uint16_t *x_row = x + (int64_t)(x_per_pair ? f : m) * K;
        const double w = topk_weights ? (double)topk_weights[f] : 1.0;
        for (int s = 0; s < num_slices; ++s) {
            shrink_one_pair(x_row, lora_a[s] + ((int64_t)l * num_experts + e) * rank * K, K, rank, t);
            const uint16_t *b_le = lora_b[s] + ((int64_t)l * num_experts + e) * N * rank;
            for (int n = 0; n < N; ++n) {
                const int c = y_offset + s * N + n;
                const double delta = expand_one_column(b_le, n, rank, t);
                o[c] = (add_inputs ? bf16_value(yin[c]) : 0.0) + w * delta;
            }
        }
    }
    free(t);
    return 0;
}
