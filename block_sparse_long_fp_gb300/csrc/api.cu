// The C ABI of libfprefill (declared in include/fprefill.h): argument
// validation, the per-batch descriptor, workspace sizing and kernel launches.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "launch.cuh"


using namespace fp;

namespace {

unsigned long long g_wait_ns = 200000000ull;    // bounded-wait limit inside kernels (200 ms)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side checks of the shape and the varlen descriptors; fills bd.
fp_status build_desc(const fp_problem *p, const fp_params *prm, BatchDesc *bd) {
    if (!p || !prm || !bd) return FP_ERR_INVALID;
    if (p->batch < 1 || p->batch > FP_MAX_BATCH) return p->batch < 1 ? FP_ERR_INVALID : FP_ERR_UNSUPPORTED;
    if (p->h_q < 1 || p->h_kv < 1 || p->h_q % p->h_kv) return FP_ERR_INVALID;
    if (p->d != kHeadDim || prm->block != kBlock) return FP_ERR_UNSUPPORTED;
    if (p->dtype != FP_BF16 && p->dtype != FP_E4M3) return FP_ERR_INVALID;
    if (!p->cu_seqlens_q || !p->seqlens_k || !p->q_start_pos) return FP_ERR_INVALID;
    if (p->cu_seqlens_q[0] != 0) return FP_ERR_INVALID;
    if (prm->sink_tokens < 0 || prm->local_tokens < 0 || !(prm->alpha >= 0.f)) return FP_ERR_INVALID;
    if (prm->kv_splits < 0 || prm->kv_splits > FP_MAX_KV_SPLITS) return FP_ERR_INVALID;
    if (prm->select_rule == FP_SELECT_TOPK && prm->top_k < 1) return FP_ERR_INVALID;
    if (prm->select_rule == FP_SELECT_TOPP && !(prm->top_p > 0.f && prm->top_p <= 1.f)) return FP_ERR_INVALID;
    if (prm->select_rule < FP_SELECT_THRESHOLD || prm->select_rule > FP_SELECT_TOPP) return FP_ERR_INVALID;
    if (prm->score_mode != FP_SCORE_PACKED && prm->score_mode != FP_SCORE_HEAD_UNION) return FP_ERR_INVALID;
    if (prm->p_terms < 0 || prm->p_terms > 2) return FP_ERR_INVALID;
    memset(bd, 0, sizeof(*bd));
    bd->batch = p->batch;
    bd->h_q = p->h_q;
    bd->h_kv = p->h_kv;
    bd->g = p->h_q / p->h_kv;
    long long rows = 0, kb = 0, sc = 0;
    int max_nkb = 1;
    for (int r = 0; r < p->batch; ++r) {
        long long lq = (long long)p->cu_seqlens_q[r + 1] - p->cu_seqlens_q[r];
        long long start = p->q_start_pos[r];
        long long lk = p->seqlens_k[r];
        if (lq < 0 || start < 0 || start % kBlock || lk != start + lq) return FP_ERR_INVALID;
        long long nqb = (lq + kBlock - 1) / kBlock, nkb = (lk + kBlock - 1) / kBlock;
        if (nkb > FP_MAX_KEY_BLOCKS) return FP_ERR_UNSUPPORTED;
        long long I0 = start / kBlock;
        ReqDesc &q = bd->req[r];
        q.q_off = p->cu_seqlens_q[r];
        q.lq = (int)lq;
        q.lk = (int)lk;
        q.start = (int)start;
        q.nqb = (int)nqb;
        q.nkb = (int)nkb;
        q.row_base = (int)rows;
        q.kb_base = (int)kb;
        q.score_base = sc;
        rows += nqb * p->h_kv;
        kb += nkb;
        sc += (long long)p->h_kv * (nqb * (I0 + 1) + nqb * (nqb - 1) / 2);
        if (nkb > max_nkb) max_nkb = (int)nkb;
    }
    if (rows > (1ll << 30) || kb > (1ll << 30) || p->cu_seqlens_q[p->batch] > (1 << 30)) return FP_ERR_UNSUPPORTED;
    bd->total_q = p->cu_seqlens_q[p->batch];
    bd->total_rows = (int)rows;
    bd->total_kb = (int)kb;
    bd->max_nkb = max_nkb;
    bd->score_size = sc;
    return FP_OK;
}

// Checks of the device operands shared by discover and the attention.
fp_status check_kv(const fp_problem *p, const BatchDesc &bd) {
    if (!p->k_cache || !p->v_cache || !p->block_table) return FP_ERR_INVALID;
    if (!aligned16(p->k_cache) || !aligned16(p->v_cache)) return FP_ERR_INVALID;
    const int ps = p->page_size;
    if (ps < 16 || !((kBlock % ps == 0) || (ps % kBlock == 0))) return FP_ERR_UNSUPPORTED;
    if (p->num_pages < 1) return FP_ERR_INVALID;
    if ((long long)p->num_pages * ps > (1ll << 31) - 1) return FP_ERR_UNSUPPORTED;
    for (int r = 0; r < bd.batch; ++r)
        if ((bd.req[r].lk + ps - 1) / ps > p->max_pages_per_seq) return FP_ERR_INVALID;
    if (p->dtype == FP_E4M3 && (!p->k_scale || !p->v_scale)) return FP_ERR_INVALID;
    if (p->v_layout != FP_V_TOKEN_MAJOR && p->v_layout != FP_V_DIM_MAJOR) return FP_ERR_INVALID;
    if (p->v_layout == FP_V_DIM_MAJOR && ps % (p->dtype == FP_E4M3 ? 128 : 64) != 0) return FP_ERR_UNSUPPORTED;
    return FP_OK;
}

fp_status check_q(const fp_problem *p) {
    if (!p->q || !aligned16(p->q)) return FP_ERR_INVALID;
    const int esz = p->dtype == FP_BF16 ? 2 : 1;
    if (p->q_stride_head < p->d || p->q_stride_tok < (long long)p->q_stride_head * (p->h_q - 1) + p->d)
        return FP_ERR_INVALID;
    if ((p->q_stride_head * esz) % 16 || (p->q_stride_tok * esz) % 16) return FP_ERR_INVALID;
    if (p->dtype == FP_E4M3 && !p->q_scale) return FP_ERR_INVALID;
    return FP_OK;
}

float softmax_scale_of(const fp_params *prm, int d) {
    return prm->softmax_scale > 0.f ? prm->softmax_scale : 1.f / sqrtf((float)d);
}

int *status_ptr(void *ws) { return reinterpret_cast<int *>(ws); }

// Scores run on the tensor cores while the column sums fit in shared memory
// (rows up to 12480 key blocks); longer rows use the fp32 CUDA-core kernel.
bool use_score_tc(const fp_problem *p, const BatchDesc &bd) {
    (void)p;
    return score_tc_smem_bytes(bd.max_nkb) <= 227 * 1024;
}

// Split-KV parts per row.  Automatic: the persistent attention kernel runs
// one CTA per SM (152 on a GB300) and takes units as SMs free up, so with U
// units of about equal length, S parts per row finish in ceil(U*S/152)/S unit
// times.  Take the S that minimises it (a larger S only when it gains >= 3%,
// since every part adds a partial output to merge), with no part shorter
// than ~16 terms; work lists of at least four units per SM are not split.
int attn_splits(const BatchDesc &bd, const fp_params *prm) {
    if (prm->kv_splits > 0) return prm->kv_splits;
    constexpr long long kSm = 152;
    const long long units = (long long)bd.total_rows * (bd.g / 2 > 0 ? bd.g / 2 : 1);
    if (units <= 0 || units >= 4 * kSm) return 1;
    const long long max_terms = bd.max_nkb + (bd.max_nkb + kBlock - 1) / kBlock;
    long long cap = max_terms / 16;
    cap = cap < FP_MAX_KV_SPLITS ? cap : FP_MAX_KV_SPLITS;
    int best = 1;
    double best_t = (double)((units + kSm - 1) / kSm);
    for (long long s = 2; s <= cap; ++s) {
        const double t = (double)((units * s + kSm - 1) / kSm) / (double)s;
        if (t < 0.97 * best_t) {
            best = (int)s;
            best_t = t;
        }
    }
    return best;
}

size_t attn_work_bytes(const BatchDesc &bd, int n_split) {
    // work schedule and, after it, the work-list cursor
    return align_up(((size_t)bd.total_rows * (bd.g / 2 > 0 ? bd.g / 2 : 1) * n_split + 1) * sizeof(int), 256);
}
size_t attn_part_o_bytes(const BatchDesc &bd, int n_split) {
    return n_split > 1 ? align_up((size_t)n_split * bd.total_q * bd.h_q * kHeadDim * sizeof(float), 256) : 0;
}
size_t attn_part_lse_bytes(const BatchDesc &bd, int n_split) {
    return n_split > 1 ? align_up((size_t)n_split * bd.h_q * bd.total_q * sizeof(float), 256) : 0;
}

size_t attn_ws_bytes(const BatchDesc &bd, int n_split) {
    size_t n = kWsHeaderBytes;
    n += attn_work_bytes(bd, n_split);
    // copies of the block means: the key means in two terms, the value means in one
    n += 3 * align_up((size_t)mean_rows(bd) * bd.h_kv * kHeadDim * 2, 256);
    n += attn_part_o_bytes(bd, n_split) + attn_part_lse_bytes(bd, n_split);
    return n;
}

}  // namespace

extern "C" {

fp_params fp_default_params(void) {
    fp_params p;
    p.block = 128;
    p.sink_tokens = 256;
    p.local_tokens = 512;
    p.alpha = 0.1f;
    p.softmax_scale = 0.f;
    p.mean_correction = 1;
    p.kv_splits = 0;
    p.select_rule = FP_SELECT_THRESHOLD;
    p.top_k = 0;
    p.top_p = 0.f;
    p.score_mode = FP_SCORE_PACKED;
    p.p_terms = 1;
    return p;
}

long long fp_num_rows(const fp_problem *p, const fp_params *prm) {
    BatchDesc bd;
    return build_desc(p, prm, &bd) == FP_OK ? bd.total_rows : -1;
}

long long fp_num_key_blocks(const fp_problem *p, const fp_params *prm) {
    BatchDesc bd;
    return build_desc(p, prm, &bd) == FP_OK ? bd.total_kb : -1;
}

long long fp_score_size(const fp_problem *p, const fp_params *prm) {
    BatchDesc bd;
    return build_desc(p, prm, &bd) == FP_OK ? bd.score_size : -1;
}

long long fp_score_offsets(const fp_problem *p, const fp_params *prm, long long *offsets, long long n) {
    BatchDesc bd;
    if (!offsets || build_desc(p, prm, &bd) != FP_OK || n < (long long)bd.total_rows + 1) return -1;
    long long k = 0;
    for (int r = 0; r < bd.batch; ++r) {
        const ReqDesc &rq = bd.req[r];
        for (int i = 0; i < rq.nqb; ++i)
            for (int h = 0; h < bd.h_kv; ++h) offsets[k++] = score_row_offset(rq, bd.h_kv, i, h);
    }
    offsets[k] = bd.score_size;
    return k + 1;
}

long long fp_total_q(const fp_problem *p) {
    if (!p || !p->cu_seqlens_q || p->batch < 1) return -1;
    return p->cu_seqlens_q[p->batch];
}

size_t fp_discover_workspace_size(const fp_problem *p, const fp_params *prm) {
    BatchDesc bd;
    if (build_desc(p, prm, &bd) != FP_OK) return 0;
    return kWsHeaderBytes + (use_score_tc(p, bd) ? align_up(score_tc_terms_bytes(bd), 256) : 0);
}

fp_status fp_discover(const fp_problem *p, const fp_params *prm, float *k_mean, float *v_mean, float *score,
                      void *ws, size_t ws_bytes, void *stream) {
    BatchDesc bd;
    fp_status s = build_desc(p, prm, &bd);
    if (s != FP_OK) return s;
    if ((s = check_kv(p, bd)) != FP_OK || (s = check_q(p)) != FP_OK) return s;
    if (!k_mean || !v_mean || !score || !aligned16(k_mean) || !aligned16(v_mean)) return FP_ERR_INVALID;
    if (!ws || ws_bytes < fp_discover_workspace_size(p, prm)) return FP_ERR_WORKSPACE;
    const bool tc = use_score_tc(p, bd);
    if (!tc && score_smem_bytes(bd.max_nkb) > 227 * 1024) return FP_ERR_UNSUPPORTED;
    const bool head_union = prm->score_mode == FP_SCORE_HEAD_UNION;
    if (head_union && !tc) return FP_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    const bool fp8 = p->dtype == FP_E4M3;
    if (bd.total_kb > 0 &&
        launch_pool(bd, fp8, p->k_cache, p->v_cache, p->page_size, p->num_pages, p->block_table,
                    p->max_pages_per_seq, p->k_scale, p->v_scale, k_mean, v_mean, status_ptr(ws), st,
                    p->v_layout == FP_V_DIM_MAJOR) != cudaSuccess)
        return FP_ERR_CUDA;
    if (bd.total_rows > 0) {
        cudaError_t e;
        if (!tc)
            e = launch_score(bd, fp8, p->q, p->q_stride_tok, p->q_stride_head, p->q_scale, k_mean,
                             softmax_scale_of(prm, p->d), score, st);
        else
            e = launch_score_tc(bd, fp8, p->q, p->q_stride_tok, p->q_stride_head, p->q_scale, k_mean,
                                softmax_scale_of(prm, p->d), score,
                                static_cast<char *>(ws) + kWsHeaderBytes,
                                status_ptr(ws), g_wait_ns, st, nullptr, head_union);
        if (e != cudaSuccess) return FP_ERR_CUDA;
    }
    return FP_OK;
}

size_t fp_select_workspace_size(const fp_problem *p, const fp_params *prm) {
    BatchDesc bd;
    if (build_desc(p, prm, &bd) != FP_OK) return 0;
    return kWsHeaderBytes + align_up(select_state_bytes(bd), 256);
}

fp_status fp_select(const fp_problem *p, const fp_params *prm, const float *score, int *row_ptr, int *col_idx,
                    long long col_capacity, int *nnz_dev, unsigned char *dense_mask_opt, void *ws, size_t ws_bytes,
                    void *stream) {
    BatchDesc bd;
    fp_status s = build_desc(p, prm, &bd);
    if (s != FP_OK) return s;
    if (!score || !row_ptr || !col_idx || !nnz_dev) return FP_ERR_INVALID;
    if (col_capacity < bd.score_size) return FP_ERR_INVALID;
    if (!ws || ws_bytes < fp_select_workspace_size(p, prm)) return FP_ERR_WORKSPACE;
    const int sink_blocks = (prm->sink_tokens + kBlock - 1) / kBlock;
    const int local_blocks = (prm->local_tokens + kBlock - 1) / kBlock;
    void *lb_state = static_cast<char *>(ws) + kWsHeaderBytes;
    if (launch_select(bd, prm->alpha, sink_blocks, local_blocks, prm->select_rule, prm->top_k, prm->top_p, score,
                      lb_state, row_ptr, col_idx, col_capacity, nnz_dev, dense_mask_opt, status_ptr(ws), g_wait_ns,
                      (cudaStream_t)stream) != cudaSuccess)
        return FP_ERR_CUDA;
    return FP_OK;
}

size_t fp_discover_select_workspace_size(const fp_problem *p, const fp_params *prm) {
    BatchDesc bd;
    if (build_desc(p, prm, &bd) != FP_OK) return 0;
    size_t n = align_up(fp_discover_workspace_size(p, prm), 256);
    n += align_up((size_t)(bd.total_rows > 0 ? bd.total_rows : 1) * 8 * sizeof(int), 256);  // kept counts
    n += align_up((size_t)(bd.score_size > 0 ? bd.score_size : 1) * sizeof(int), 256);    // kept lists / scores
    return n;
}

fp_status fp_discover_select(const fp_problem *p, const fp_params *prm, float *k_mean, float *v_mean,
                             float *score_opt, int *row_ptr, int *col_idx, long long col_capacity, int *nnz_dev,
                             void *ws, size_t ws_bytes, void *stream) {
    BatchDesc bd;
    fp_status s = build_desc(p, prm, &bd);
    if (s != FP_OK) return s;
    if ((s = check_kv(p, bd)) != FP_OK || (s = check_q(p)) != FP_OK) return s;
    if (!k_mean || !v_mean || !aligned16(k_mean) || !aligned16(v_mean)) return FP_ERR_INVALID;
    if (!row_ptr || !col_idx || !nnz_dev || col_capacity < bd.score_size) return FP_ERR_INVALID;
    if (!ws || ws_bytes < fp_discover_select_workspace_size(p, prm)) return FP_ERR_WORKSPACE;
    const bool tc = use_score_tc(p, bd);
    if (!tc && score_smem_bytes(bd.max_nkb) > 227 * 1024) return FP_ERR_UNSUPPORTED;
    const bool head_union = prm->score_mode == FP_SCORE_HEAD_UNION;
    if (head_union && !tc) return FP_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    const bool fp8 = p->dtype == FP_E4M3;
    char *w = static_cast<char *>(ws);
    size_t off = align_up(fp_discover_workspace_size(p, prm), 256);
    int *counts = reinterpret_cast<int *>(w + off);     // [rows, 8] (fused) or [rows]
    off += align_up((size_t)(bd.total_rows > 0 ? bd.total_rows : 1) * 8 * sizeof(int), 256);
    int *keep_pad = reinterpret_cast<int *>(w + off);
    const int sink_blocks = (prm->sink_tokens + kBlock - 1) / kBlock;
    const int local_blocks = (prm->local_tokens + kBlock - 1) / kBlock;
    if (bd.total_kb > 0 &&
        launch_pool(bd, fp8, p->k_cache, p->v_cache, p->page_size, p->num_pages, p->block_table,
                    p->max_pages_per_seq, p->k_scale, p->v_scale, k_mean, v_mean, status_ptr(ws), st,
                    p->v_layout == FP_V_DIM_MAJOR) != cudaSuccess)
        return FP_ERR_CUDA;
    if (bd.total_rows == 0) {
        return cudaMemsetAsync(row_ptr, 0, sizeof(int), st) == cudaSuccess &&
                       cudaMemsetAsync(nnz_dev, 0, sizeof(int), st) == cudaSuccess
                   ? FP_OK
                   : FP_ERR_CUDA;
    }
    void *terms = w + kWsHeaderBytes;
    const float scale = softmax_scale_of(prm, p->d);
    cudaError_t e;
    if (tc && prm->select_rule == FP_SELECT_THRESHOLD && !head_union) {
        // one pass: the score kernel decides each row and lists its kept blocks
        ScoreSelect sel{keep_pad, counts, prm->alpha, sink_blocks, local_blocks};
        e = launch_score_tc(bd, fp8, p->q, p->q_stride_tok, p->q_stride_head, p->q_scale, k_mean, scale, score_opt,
                            terms, status_ptr(ws), g_wait_ns, st, &sel);
        if (e == cudaSuccess)
            e = launch_select_gather(bd, keep_pad, counts, row_ptr, col_idx, col_capacity, nnz_dev, status_ptr(ws), st);
    } else {
        // the separate stages, with the score map in the workspace when none is given
        float *sc = score_opt ? score_opt : reinterpret_cast<float *>(keep_pad);
        e = tc ? launch_score_tc(bd, fp8, p->q, p->q_stride_tok, p->q_stride_head, p->q_scale, k_mean, scale, sc,
                                 terms, status_ptr(ws), g_wait_ns, st, nullptr, head_union)
               : launch_score(bd, fp8, p->q, p->q_stride_tok, p->q_stride_head, p->q_scale, k_mean, scale, sc, st);
        if (e == cudaSuccess)
            e = launch_select(bd, prm->alpha, sink_blocks, local_blocks, prm->select_rule, prm->top_k, prm->top_p, sc,
                              counts, row_ptr, col_idx, col_capacity, nnz_dev, nullptr, status_ptr(ws), g_wait_ns, st);
    }
    return e == cudaSuccess ? FP_OK : FP_ERR_CUDA;
}

int fp_attn_kv_splits(const fp_problem *p, const fp_params *prm) {
    BatchDesc bd;
    if (build_desc(p, prm, &bd) != FP_OK) return -1;
    return attn_splits(bd, prm);
}

size_t fp_attn_workspace_size(const fp_problem *p, const fp_params *prm) {
    BatchDesc bd;
    if (build_desc(p, prm, &bd) != FP_OK) return 0;
    return attn_ws_bytes(bd, attn_splits(bd, prm));
}

static fp_status run_attn(const fp_problem *p, const fp_params *prm, const int *row_ptr, const int *col_idx,
                          const float *k_mean, const float *v_mean, void *out, float *lse, void *ws, size_t ws_bytes,
                          void *stream) {
    BatchDesc bd;
    fp_status s = build_desc(p, prm, &bd);
    if (s != FP_OK) return s;
    if ((s = check_kv(p, bd)) != FP_OK || (s = check_q(p)) != FP_OK) return s;
    if (bd.g % 2) return FP_ERR_UNSUPPORTED;
    if (!out || !aligned16(out)) return FP_ERR_INVALID;
    const int n_split = attn_splits(bd, prm);
    if (!ws || ws_bytes < attn_ws_bytes(bd, n_split)) return FP_ERR_WORKSPACE;
    char *w = static_cast<char *>(ws);
    AttnLaunch L;
    memset(&L, 0, sizeof(L));
    L.bd = &bd;
    L.q = p->q;
    L.q_stride_tok = p->q_stride_tok;
    L.q_stride_head = p->q_stride_head;
    L.k_cache = p->k_cache;
    L.v_cache = p->v_cache;
    L.page_size = p->page_size;
    L.num_pages = p->num_pages;
    L.block_table = p->block_table;
    L.max_pages = p->max_pages_per_seq;
    L.row_ptr = row_ptr;
    L.col_idx = col_idx;
    L.k_mean = k_mean;
    L.v_mean = v_mean;
    L.mean_corr = prm->mean_correction ? 1 : 0;
    L.softmax_scale = softmax_scale_of(prm, p->d);
    L.out = out;
    L.lse = lse;
    L.status = status_ptr(ws);
    size_t off = kWsHeaderBytes;
    L.work = reinterpret_cast<int *>(w + off);
    off += attn_work_bytes(bd, n_split);
    L.km16 = reinterpret_cast<__nv_bfloat16 *>(w + off);
    off += 2 * align_up((size_t)mean_rows(bd) * bd.h_kv * kHeadDim * 2, 256);
    L.vm16 = reinterpret_cast<__nv_bfloat16 *>(w + off);
    off += align_up((size_t)mean_rows(bd) * bd.h_kv * kHeadDim * 2, 256);
    L.n_split = n_split;
    L.part_o = n_split > 1 ? reinterpret_cast<float *>(w + off) : nullptr;
    off += attn_part_o_bytes(bd, n_split);
    L.part_lse = n_split > 1 ? reinterpret_cast<float *>(w + off) : nullptr;
    L.wait_ns = g_wait_ns;
    L.fp8 = p->dtype == FP_E4M3;
    L.v_dim_major = p->v_layout == FP_V_DIM_MAJOR;
    L.p_terms = prm->p_terms == 2 ? 2 : 1;
    L.q_scale = p->q_scale;
    L.k_scale = p->k_scale;
    L.v_scale = p->v_scale;
    return (fp_status)launch_attn(L, (cudaStream_t)stream);
}

fp_status fp_sparse_attn(const fp_problem *p, const fp_params *prm, const int *row_ptr, const int *col_idx,
                         const float *k_mean, const float *v_mean, void *out, float *lse_opt, void *ws,
                         size_t ws_bytes, void *stream) {
    if (!row_ptr || !col_idx) return FP_ERR_INVALID;
    if (prm && prm->mean_correction && (!k_mean || !v_mean)) return FP_ERR_INVALID;
    return run_attn(p, prm, row_ptr, col_idx, k_mean, v_mean, out, lse_opt, ws, ws_bytes, stream);
}

fp_status fp_dense_attn(const fp_problem *p, const fp_params *prm, void *out, float *lse_opt, void *ws,
                        size_t ws_bytes, void *stream) {
    return run_attn(p, prm, nullptr, nullptr, nullptr, nullptr, out, lse_opt, ws, ws_bytes, stream);
}

fp_status fp_reset_status(void *ws, void *stream) {
    if (!ws) return FP_ERR_INVALID;
    return cudaMemsetAsync(ws, 0, kWsHeaderBytes, (cudaStream_t)stream) == cudaSuccess ? FP_OK : FP_ERR_CUDA;
}

fp_status fp_device_status(const void *ws, void *stream, int *device_status) {
    if (!ws || !device_status) return FP_ERR_INVALID;
    int v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
        return FP_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FP_ERR_CUDA;
    *device_status = v;
    return FP_OK;
}

const char *fp_status_string(fp_status s) {
    switch (s) {
        case FP_OK: return "ok";
        case FP_ERR_INVALID: return "invalid argument";
        case FP_ERR_UNSUPPORTED: return "unsupported shape or option";
        case FP_ERR_WORKSPACE: return "workspace missing or too small";
        case FP_ERR_CUDA: return "CUDA runtime error";
        case FP_ERR_DEVICE_BOUNDS: return "page-table or index entry out of range (device)";
        case FP_ERR_TIMEOUT: return "bounded wait timed out (device)";
    }
    return "unknown status";
}

void fp_set_wait_limit_ns(unsigned long long ns) { g_wait_ns = ns ? ns : 200000000ull; }

fp_status fp_check_wait_timeout(void *ws, unsigned long long limit_ns, void *stream) {
    if (!ws || limit_ns == 0 || limit_ns > 10000000000ull) return FP_ERR_INVALID;
    return launch_wait_timeout(status_ptr(ws), limit_ns, (cudaStream_t)stream) == cudaSuccess ? FP_OK : FP_ERR_CUDA;
}

}  // extern "C"
