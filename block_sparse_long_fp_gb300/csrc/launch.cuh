// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include "common.cuh"

namespace fp {
cudaError_t launch_pool(const BatchDesc &bd, bool fp8, const void *k_cache, const void *v_cache, int page_size,
                        int num_pages, const int *block_table, int max_pages, const float *k_scale,
                        const float *v_scale, float *k_mean, float *v_mean, int *status, cudaStream_t st,
                        bool v_dim_major = false);
cudaError_t launch_score(const BatchDesc &bd, bool fp8, const void *q, long long q_stride_tok,
                         long long q_stride_head, const float *q_scale, const float *k_mean, float softmax_scale,
                         float *score, cudaStream_t st);
// lb_state: look-back scratch of select_state_bytes(bd), 8-byte aligned
cudaError_t launch_select(const BatchDesc &bd, float alpha, int sink_blocks, int local_blocks, int rule, int top_k,
                          float top_p, const float *score, void *lb_state, int *row_ptr, int *col_idx,
                          long long col_capacity, int *nnz, unsigned char *dense_mask, int *status,
                          unsigned long long wait_ns, cudaStream_t st);
inline size_t select_state_bytes(const BatchDesc &bd) { return (size_t)((bd.total_rows + 7) / 8 + 1) * 8; }
size_t score_smem_bytes(int max_nkb);
// tensor-core score map: the two fp16 terms of the key means, then the scale
// exponent of each (128-block chunk, kv head), live in a workspace of
// score_tc_terms_bytes()
int score_tc_rows_pad(const BatchDesc &bd);
size_t score_tc_smem_bytes(int max_nkb);   // the tensor-core path needs this <= 227 KB
inline size_t score_tc_kexp_offset(const BatchDesc &bd) {
    return ((size_t)2 * score_tc_rows_pad(bd) * bd.h_kv * kHeadDim * 2 + 255) / 256 * 256;
}
inline size_t score_tc_terms_bytes(const BatchDesc &bd) {
    return score_tc_kexp_offset(bd) + (size_t)(bd.total_kb > 0 ? bd.total_kb : 1) * bd.h_kv;
}
// fused selection at the end of the tensor-core score kernel (threshold rule)
struct ScoreSelect {
    int *keep_pad;            // [score_size] ints: each row's kept blocks at its score-map offset
    int *counts;              // [total_rows, 8]: kept blocks per row warp's segment
    float alpha;
    int sink_blocks, local_blocks;
};
cudaError_t launch_score_tc(const BatchDesc &bd, bool fp8, const void *q, long long q_stride_tok,
                            long long q_stride_head, const float *q_scale, const float *k_mean, float softmax_scale,
                            float *score, void *terms_ws, int *status, unsigned long long wait_ns,
                            cudaStream_t st, const ScoreSelect *sel = nullptr, bool head_union = false);
cudaError_t launch_select_gather(const BatchDesc &bd, const int *keep_pad, const int *counts, int *row_ptr,
                                 int *col_idx, long long col_capacity, int *nnz, int *status, cudaStream_t st);

struct AttnLaunch {
    const BatchDesc *bd;
    const void *q;
    long long q_stride_tok, q_stride_head;
    const void *k_cache, *v_cache;
    int page_size, num_pages;
    const int *block_table;
    int max_pages;
    const int *row_ptr, *col_idx;
    const float *k_mean, *v_mean;
    int mean_corr;
    float softmax_scale;
    void *out;
    float *lse;
    int *status;
    int *work;
    __nv_bfloat16 *km16, *vm16;       // block-mean copies (bf16, or e4m3 in the same space)
    unsigned long long wait_ns;
    bool fp8;                         // e4m3 q / k / v with per-head scales
    const float *q_scale, *k_scale, *v_scale;
    int n_split;                      // split-KV parts per row (1: none)
    float *part_o;                    // [n_split, total_q, h_q, d] fp32 when n_split > 1
    float *part_lse;                  // [n_split, h_q, total_q] fp32 when n_split > 1
    bool v_dim_major;                 // value cache [num_pages, h_kv, d, page_size]
    int p_terms;                      // e4m3: P in 1 term (e4m3 of 256 p) or 2 (plus the residual)
};
int launch_attn(const AttnLaunch &L, cudaStream_t st);
// rows of the bf16 block-mean copies: at least one full 128-row TMA box
inline int mean_rows(const BatchDesc &bd) { return bd.total_kb > kBlock ? bd.total_kb : kBlock; }
int attn_smem_bytes();
cudaError_t launch_wait_timeout(int *status, unsigned long long limit_ns, cudaStream_t st);
}  // namespace fp
