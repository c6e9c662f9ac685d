/*
 * libfprefill: block-sparse causal prefill attention in the FlashPrefill
 * style (instantaneous block-pattern discovery, max-based dynamic threshold,
 * index compaction, sparse attention with block-mean correction) for one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * Sources: the FlashPrefill V1 summary ("FlashPrefill: long-context
 * acceleration 28x", mhpn.cn; sections 3.1-3.3), the FlashPrefill V2 paper
 * reading (inkeast.github.io MessageDaily; sections 4, 4.1-4.3) and the
 * FlashPrefill V2 popular article (animattoys.com; sections on mean
 * correction, PackGQA, FP8, the CSR index and paged KV).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - The caller owns and allocates every buffer; the library allocates
 *    nothing.  Pointers named "device" must be device memory, 16-byte aligned.
 *    The varlen descriptors (cu_seqlens_q, seqlens_k, q_start_pos) are small
 *    HOST arrays read synchronously during the call.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  Argument errors are returned synchronously, before anything
 *    is enqueued.  Errors found by a kernel (a page-table entry out of range,
 *    a bounded wait that timed out) are recorded in a status word inside the
 *    workspace (first error wins) and read back with fp_device_status().
 *  - Every workspace is an opaque device buffer of at least the size its
 *    *_workspace_size() query returns.  Its first 256 bytes are a header
 *    holding the status word: zero them once (fp_reset_status) before first
 *    use.  One workspace may serve all stages in turn (take the largest
 *    size); calls that overlap on the GPU must not share one.
 *  - Query rows: token-major [total_q, h_q, d]; request r owns rows
 *    cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1; its query i sits at absolute
 *    position q_start_pos[r] + i and attends causally to keys 0..position.
 *    seqlens_k[r] must equal q_start_pos[r] + (its query count): a prefill
 *    (q_start_pos = 0) or a chunk of a chunked prefill whose earlier tokens
 *    are already in the cache.  q_start_pos must be a multiple of the block.
 *  - Paged KV [V2 paper reading 4.3; V2 article, paged KV address rule]:
 *    k_cache / v_cache are [num_pages, page_size, h_kv, d] (contiguous); the
 *    key at position t of request r lives in physical page
 *    block_table[r * max_pages_per_seq + t / page_size], slot t % page_size.
 *    page_size must divide 128 or be a multiple of 128, and be >= 16.
 *  - Blocks: B = params.block = 128 tokens (query and key blocks alike).
 *    Request r has nqb_r = ceil(lq_r / B) query blocks starting at absolute
 *    block I0_r = q_start_pos[r] / B, and nkb_r = ceil(seqlens_k[r] / B) key
 *    blocks.
 *  - Rows: the index and the score map are organised in rows (r, i, h) -- a
 *    query block i of request r and a kv head h -- ordered request-major,
 *    then query block, then kv head:  row = rowbase_r + i * h_kv + h, with
 *    rowbase_r = sum_{r' < r} nqb_r' * h_kv.  R = total rows.  The absolute
 *    block of the row is I = I0_r + i; its causal key blocks are J = 0..I.
 *  - Pooled means: [sum_r nkb_r, h_kv, d] fp32; request r's blocks start at
 *    kbbase_r = sum_{r' < r} nkb_r'.
 *  - Score map: fp32, row (r, i, h) holds I + 1 values (J = 0..I) at offset
 *      scorebase_r + h_kv * (i * (I0_r + 1) + i * (i - 1) / 2)
 *                  + h * (I0_r + i + 1),
 *    scorebase_r = sum_{r' < r} h_kv * (nqb * (I0 + 1) + nqb * (nqb - 1) / 2).
 *    fp_score_size() returns the total.
 *  - CSR index [V2 paper reading 4 "CSR"; V1 3.3 "physical jump"]: row_ptr
 *    int32 [R + 1], col_idx int32 [nnz] listing the kept key blocks J of each
 *    row in ascending order.  col_capacity must be >= fp_score_size() (the
 *    causal upper bound), so selection never needs a host synchronisation.
 *  - Supported: d = 128, B = 128, h_q a multiple of 2*h_kv (query heads are
 *    processed in pairs of the same group), batch <= FP_MAX_BATCH.  Other
 *    shapes return FP_ERR_UNSUPPORTED.
 */
#ifndef FPREFILL_H
#define FPREFILL_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP_MAX_BATCH 128
#define FP_MAX_KEY_BLOCKS 16384

typedef enum {
    FP_OK = 0,
    FP_ERR_INVALID = 1,        /* bad argument (null pointer, inconsistent lengths, alignment) */
    FP_ERR_UNSUPPORTED = 2,    /* a shape or option this build does not implement */
    FP_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
    FP_ERR_CUDA = 4,           /* a CUDA runtime call failed (launch, copy) */
    FP_ERR_DEVICE_BOUNDS = 5,  /* device status: a page-table entry outside [0, num_pages), or an
                                  index entry J outside [0, I] (its tile is read as zeros) */
    FP_ERR_TIMEOUT = 6         /* device status: a bounded wait inside a kernel gave up */
} fp_status;

typedef enum {
    FP_BF16 = 0,   /* q, k_cache, v_cache hold bf16 */
    FP_E4M3 = 1    /* q, k_cache, v_cache hold fp8 e4m3 codes; value = code * scale[head] */
} fp_dtype;

typedef struct {
    int block;            /* B, tokens per block: must be 128 */
    int sink_tokens;      /* blocks holding any of the first sink_tokens are always kept (256) */
    int local_tokens;     /* the ceil(local_tokens / B) blocks ending at I are always kept (512) */
    float alpha;          /* keep J when Score[I,J] >= alpha * max_J Score[I,J] (0.1) */
    float softmax_scale;  /* logit scale; <= 0 selects 1/sqrt(d) */
    int mean_correction;  /* 1: skipped blocks J < I add their block-mean term */
    int kv_splits;        /* attention only: split each row's key list into this many
                             parts merged by their LSE (split-KV); 0 chooses (more
                             parts when the problem has too few work units to fill
                             the GPU), 1 never splits; at most FP_MAX_KV_SPLITS */
    int select_rule;      /* fp_select rule (fp_select_rule); sink and local blocks are
                             kept under every rule */
    int top_k;            /* FP_SELECT_TOPK: blocks kept per row (>= 1) */
    float top_p;          /* FP_SELECT_TOPP: share of the row's score mass kept, (0, 1] */
    int score_mode;       /* fp_discover: FP_SCORE_PACKED or FP_SCORE_HEAD_UNION */
    int p_terms;          /* FP_E4M3 attention only: the softmax weights P enter the PV
                             product as 1 e4m3 term, e4m3(256 p) [V2 paper reading 4.2 (4)],
                             or 2: that term plus the residual e4m3(256 p - term) in a second
                             PV pass, which cuts the weights' rounding from 2^-4 to about
                             2^-8 relative; 0 means 1 */
} fp_params;

/* Score modes of fp_discover.  PACKED is the reading of the V1 summary 3.1
 * with PackGQA (the g heads x B queries of a group are one set of packed
 * rows); HEAD_UNION is the alternative: each query head's row is normalised
 * on its own and the row keeps the maximum over the group's heads, so the
 * threshold keeps the union of the heads' own selections. */
typedef enum { FP_SCORE_PACKED = 0, FP_SCORE_HEAD_UNION = 1 } fp_score_mode;

/* Selection rules of fp_select.  THRESHOLD is the method's rule [V1 summary
 * 3.2]; TOPK and TOPP are the alternatives it is compared with [V1 summary
 * 4.4], kept here as ablations. */
typedef enum {
    FP_SELECT_THRESHOLD = 0,  /* Score >= alpha * max_J Score */
    FP_SELECT_TOPK = 1,       /* the top_k highest scores; among equal scores the lower J */
    FP_SELECT_TOPP = 2        /* the highest scores, down to the largest t such that the
                                 scores >= t hold at least top_p of the row's total */
} fp_select_rule;

#define FP_MAX_KV_SPLITS 32

typedef struct {
    int batch;
    int h_q;
    int h_kv;
    int d;
    fp_dtype dtype;
    /* HOST arrays */
    const int *cu_seqlens_q;      /* [batch + 1], cu_seqlens_q[0] = 0, non-decreasing */
    const int *seqlens_k;         /* [batch] */
    const int *q_start_pos;       /* [batch] */
    /* DEVICE arrays */
    const void *q;                /* [total_q, h_q, d] at the strides below */
    long long q_stride_tok;       /* elements between consecutive tokens (>= h_q * d) */
    long long q_stride_head;      /* elements between consecutive heads (>= d) */
    const void *k_cache;          /* [num_pages, page_size, h_kv, d] */
    const void *v_cache;
    int page_size;
    int num_pages;
    const int *block_table;       /* [batch, max_pages_per_seq] physical page ids */
    int max_pages_per_seq;
    const float *q_scale;         /* [h_q]   FP_E4M3 only (may be NULL for FP_BF16) */
    const float *k_scale;         /* [h_kv]  FP_E4M3 only */
    const float *v_scale;         /* [h_kv]  FP_E4M3 only */
    int v_layout;                 /* fp_v_layout of v_cache (0: token-major, like k_cache) */
} fp_problem;

/* Layout of the value cache [V2 popular article, FP8 passage: a value cache
 * stored by rows or by columns].  TOKEN_MAJOR: [num_pages, page_size, h_kv, d],
 * the layout of k_cache.  DIM_MAJOR: [num_pages, h_kv, d, page_size], each
 * (page, head, d) holding the page's tokens contiguously; page_size must be a
 * multiple of 64 for FP_BF16 and of 128 for FP_E4M3 (FP_ERR_UNSUPPORTED
 * otherwise).  The result is the same either way (up to the summation order
 * of the PV product); the attention takes DIM_MAJOR tiles as K-major operands
 * and TOKEN_MAJOR ones as MN-major operands, so neither is transposed on chip. */
typedef enum { FP_V_TOKEN_MAJOR = 0, FP_V_DIM_MAJOR = 1 } fp_v_layout;

/* Defaults of the pages: B=128, sink 256, local 512, alpha 0.1, 1/sqrt(d),
 * mean correction on [V2 paper reading, section 4 configuration]; kv_splits 0
 * (chosen by the library); the threshold rule (top_k 0, top_p 0: unused);
 * p_terms 1 (the pages' e4m3 P). */
fp_params fp_default_params(void);

/* Sizes derived from the host descriptors (element counts, not bytes). */
long long fp_num_rows(const fp_problem *p, const fp_params *prm);        /* R */
long long fp_num_key_blocks(const fp_problem *p, const fp_params *prm);  /* sum_r nkb_r */
long long fp_score_size(const fp_problem *p, const fp_params *prm);      /* floats in the score map */
long long fp_total_q(const fp_problem *p);                               /* cu_seqlens_q[batch] */

/* Offsets of the score-map rows (the closed form above), for callers that
 * index the score map or the dense mask: offsets (HOST int64, n entries)
 * receives the offset of row k = 0 .. R-1 in row order, then
 * offsets[R] = fp_score_size().  Host-only: enqueues nothing.  Returns R + 1,
 * or -1 when an argument is invalid or n < R + 1. */
long long fp_score_offsets(const fp_problem *p, const fp_params *prm, long long *offsets, long long n);

/* ---------------------------------------------------------------------------
 * fp_discover -- instantaneous pattern discovery
 * [V1 3.1 key pooling + query-block scoring; V2 4.1 block means of K and V]
 *
 *   k_mean, v_mean (device, fp32 [sum_r nkb_r, h_kv, d]): block means over the
 *     n_J = min(B, lk - J*B) tokens of each key block (FP8: of the
 *     dequantised values).
 *   score (device, fp32, fp_score_size() floats, layout above): for row
 *     (r, i, h) with absolute query block I, each of the g*B packed query rows
 *     (g = h_q / h_kv heads of the group x the block's queries) contributes
 *     exp(s_J - max_J' s_J') to S'[J], s_J = scale * q . k_mean_J for J <= I;
 *     Score[I,J] = S'[J] / max_J' S'[J'] (so each row peaks at exactly 1).
 *     FP_SCORE_HEAD_UNION: the same per query head (its B queries alone),
 *     and Score[I,J] = max over the group's heads of those rows (still
 *     peaking at 1); rows over 12480 key blocks: FP_ERR_UNSUPPORTED.
 *   ws: fp_discover_workspace_size() bytes (status header only).
 * ------------------------------------------------------------------------- */
size_t fp_discover_workspace_size(const fp_problem *p, const fp_params *prm);
fp_status fp_discover(const fp_problem *p, const fp_params *prm, float *k_mean, float *v_mean,
                      float *score, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fp_select -- max-based dynamic threshold + sink/local forcing + compaction
 * [V1 3.2 threshold alpha * max_{J<=I} Score[I,J], sink and local safety net;
 *  V1 3.3 compaction of kept indices; V2 4 CSR index]
 *
 *   keep[I,J] = sel(I,J)  or  J * B < sink_tokens  or  J >= I - ceil(local_tokens / B) + 1
 *   sel: FP_SELECT_THRESHOLD  Score[I,J] >= alpha * max_J Score[I,J];
 *        FP_SELECT_TOPK  J is among the top_k highest scores of the row
 *                        (equal scores: lower J first);
 *        FP_SELECT_TOPP  Score[I,J] >= t, t the largest value such that the
 *                        scores >= t sum to at least top_p * sum_J Score[I,J].
 *   row_ptr (device int32 [R + 1]), col_idx (device int32, col_capacity
 *   entries; the first nnz are written), nnz_dev (device int32 [1]).
 *   dense_mask_opt (device uint8, fp_score_size() bytes, may be NULL): the
 *   keep decision of every score entry, at the score map's offsets.
 *   ws: fp_select_workspace_size() bytes.
 * ------------------------------------------------------------------------- */
size_t fp_select_workspace_size(const fp_problem *p, const fp_params *prm);
fp_status fp_select(const fp_problem *p, const fp_params *prm, const float *score, int *row_ptr,
                    int *col_idx, long long col_capacity, int *nnz_dev,
                    unsigned char *dense_mask_opt, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fp_discover_select -- fp_discover and fp_select in one call
 * [V1 summary 3.1-3.3 run back to back]
 *
 * Same results as fp_discover followed by fp_select with the same params (the
 * same k_mean / v_mean, score map and CSR index).  With the threshold rule on
 * rows the tensor-core score kernel takes, that kernel decides each row and
 * lists its kept blocks itself, so the score map is neither written (unless
 * score_opt is given) nor read back.
 *   score_opt (device fp32, fp_score_size() floats, may be NULL).
 *   row_ptr, col_idx, col_capacity, nnz_dev as fp_select.
 *   ws: fp_discover_select_workspace_size() bytes.
 * ------------------------------------------------------------------------- */
size_t fp_discover_select_workspace_size(const fp_problem *p, const fp_params *prm);
fp_status fp_discover_select(const fp_problem *p, const fp_params *prm, float *k_mean, float *v_mean,
                             float *score_opt, int *row_ptr, int *col_idx, long long col_capacity,
                             int *nnz_dev, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fp_sparse_attn -- block-sparse attention with block-mean correction
 * [V2 paper reading 4.1 (mean correction), 4.2 (PackGQA, warp
 *  specialisation, FP8), 4.3 (paged KV through the page table)]
 *
 * For query position p in absolute block I of row (r, i, h):
 *   O = [ sum_{J in row} sum_{t in J, t <= p} e^{s_t - m} v_t
 *         + mc * sum_{J < I, J not in row} n_J e^{scale q.kmean_J - m} vmean_J ]
 *       / [ the same sums without v ],   s_t = scale q.k_t,
 *   mc = params.mean_correction, m a common shift; LSE = m + ln(denominator).
 *   row_ptr/col_idx: a CSR index as produced by fp_select (ascending J <= I).
 *   k_mean/v_mean: as produced by fp_discover (read only when mc = 1).
 *   out (device bf16 [total_q, h_q, d], contiguous).
 *   lse_opt (device fp32 [h_q, total_q], natural log; may be NULL).
 *   ws: fp_attn_workspace_size() bytes (work schedule, the tensor-core copies
 *   of the block means, and with split-KV the fp32 partial outputs and LSEs).
 * A row with no term at all (an empty index row, no correction) yields O = 0.
 * The mean tokens' logits run on the tensor cores: bf16 problems take the key
 * means as fp16 (a power-of-two scale per 128-block tile and kv head) against
 * the queries in fp16 (exact under a power-of-two scale per row), so a mean
 * logit errs by about 2^-12 relative; e4m3 problems take them as two e4m3
 * terms.
 *
 * Split-KV (the kept-count load balancing of the V2 popular article, "KV
 * split", for rows too long for the number of rows): with S = the split count
 * chosen from params.kv_splits, each row's terms (kept blocks, then mean
 * tiles) are cut into S consecutive parts of equal size.  Part s yields
 * O_s, LSE_s over its own terms, and O = sum_s e^{LSE_s - LSE} O_s with
 * LSE = ln sum_s e^{LSE_s}: the same O up to rounding.  The workspace size
 * depends on the split count, so query it with the same params.
 * ------------------------------------------------------------------------- */
size_t fp_attn_workspace_size(const fp_problem *p, const fp_params *prm);
/* The split count S the attention calls use for these params (>= 1), or -1
 * on an argument error. */
int fp_attn_kv_splits(const fp_problem *p, const fp_params *prm);
fp_status fp_sparse_attn(const fp_problem *p, const fp_params *prm, const int *row_ptr,
                         const int *col_idx, const float *k_mean, const float *v_mean,
                         void *out, float *lse_opt, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fp_sparse_attn_noalloc -- fp_sparse_attn for callers that cannot allocate
 * (no counterpart in the pages: an interface addition of this library).
 *
 * For callers that have no way to provide a device workspace: a plugin whose
 * host framework owns all device memory and hands it none, or a serving loop
 * held to a fixed device-memory budget where allocating mid-request could fail
 * or stall the device.  The function allocates nothing: its scratch is one
 * file-scope device array of FP_NOALLOC_SCRATCH_BYTES, reserved on every GPU
 * that loads the library until the process exits.  The caller still provides
 * the inputs and the outputs.
 *
 *   Arguments and results as fp_sparse_attn, without ws / ws_bytes; rows are
 *   split only when params.kv_splits asks for it (0 means no split here).
 *   status_dev_opt (device int32 [1], may be NULL): receives this call's
 *     device status word (FP_OK or an fp_status code), in stream order after
 *     the kernels -- the scratch itself is not visible to the caller.
 *   Returns FP_ERR_WORKSPACE when the problem needs more scratch than
 *     FP_NOALLOC_SCRATCH_BYTES (compare fp_attn_workspace_size()), before
 *     touching the GPU; other argument errors as fp_sparse_attn.
 *   Every call looks up the array's device address in the caller's current
 *     context (nothing is cached, so non-primary contexts and a device reset
 *     between calls are fine).  The first call in a context may load the
 *     library's device code into it: make that first call before any stream
 *     capture.
 *   Every call on a device shares the one array, and the array keeps the last
 *   call's contents (the call clears what must start at zero).  Calls that
 *   overlap on the GPU -- on different streams, or from different threads --
 *   race on it: serialise them.
 * ------------------------------------------------------------------------- */
#define FP_NOALLOC_SCRATCH_BYTES (8u << 20)
fp_status fp_sparse_attn_noalloc(const fp_problem *p, const fp_params *prm, const int *row_ptr,
                                 const int *col_idx, const float *k_mean, const float *v_mean,
                                 void *out, float *lse_opt, int *status_dev_opt, void *stream);

/* ---------------------------------------------------------------------------
 * fp_dense_attn -- the same kernel keeping every causal block, no correction
 * (the in-house dense baseline [V2 paper reading 5.3, 5.6]).  Same arguments
 * as fp_sparse_attn without the index and the means.
 * ------------------------------------------------------------------------- */
fp_status fp_dense_attn(const fp_problem *p, const fp_params *prm, void *out, float *lse_opt,
                        void *ws, size_t ws_bytes, void *stream);

/* Zero the status header of a workspace (enqueued on stream). */
fp_status fp_reset_status(void *ws, void *stream);

/* Wait for `stream`, then read the status word of `ws` into *device_status
 * (an fp_status value; FP_OK when no kernel recorded an error). */
fp_status fp_device_status(const void *ws, void *stream, int *device_status);

/* Time limit of every bounded wait inside the attention kernel, in
 * nanoseconds (default 200 ms; 0 restores the default).  A wait that runs out
 * records FP_ERR_TIMEOUT and the kernel returns instead of hanging. */
void fp_set_wait_limit_ns(unsigned long long ns);

/* Failure-path check of the bounded waits, with no GPU fault: launches one
 * thread that waits, through the kernels' own bounded wait, on an mbarrier
 * that nothing arrives on, for limit_ns nanoseconds (1 .. 1e10).  The wait
 * runs out, FP_ERR_TIMEOUT lands in the status word of ws (first error
 * wins), and the context stays usable: reset the status and carry on.
 * Returns FP_ERR_INVALID for a null ws or a limit out of range. */
fp_status fp_check_wait_timeout(void *ws, unsigned long long limit_ns, void *stream);

/* Static description of an fp_status value. */
const char *fp_status_string(fp_status s);

#ifdef __cplusplus
}
#endif
#endif /* FPREFILL_H */
