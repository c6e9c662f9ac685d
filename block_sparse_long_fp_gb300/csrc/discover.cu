// fp_discover kernels: block-mean pooling of K and V, and the block-score map.
//
// Pooling follows the key pooling of the FlashPrefill V1 summary, section 3.1
// (mean over each 128-token block), extended to V for the V2 mean correction
// (V2 paper reading, section 4.1: kbar_j and vbar_j).  Scoring follows V1
// section 3.1: per packed query row, logits against the pooled keys are
// normalised by the row's own maximum, exponentiated and summed over the
// query block; the row of block scores is then divided by its largest entry
// ("global re-weighting").
#include "common.cuh"
#include "launch.cuh"

namespace fp {

// ---------------------------------------------------------------------------
// pool: one CTA per pooled block; a token's h_kv*d values are contiguous in a
// page, so each thread streams one 16-byte column vector over a strided
// subset of the block's tokens and the partial sums meet in shared memory.
// ---------------------------------------------------------------------------
template <bool kFp8>
__global__ void __launch_bounds__(256)
pool_kernel(const __grid_constant__ BatchDesc bd, const uint8_t *__restrict__ k_cache,
            const uint8_t *__restrict__ v_cache, int page_size, int num_pages,
            const int *__restrict__ block_table, int max_pages,
            const float *__restrict__ k_scale, const float *__restrict__ v_scale,
            float *__restrict__ k_mean, float *__restrict__ v_mean, int *status, int v_dim_major) {
    constexpr int kEsz = kFp8 ? 1 : 2;
    constexpr int kEpv = 16 / kEsz;  // elements per 16-byte vector
    __shared__ float red[256 * kEpv];

    const int kb = blockIdx.x;
    const int r = req_of_kb(bd, kb);
    const ReqDesc &rq = bd.req[r];
    const int J = kb - rq.kb_base;
    const int t0 = J * kBlock;
    const int t1 = min(rq.lk, t0 + kBlock);
    const int n = t1 - t0;

    const int vpt = bd.h_kv * kHeadDim / kEpv;       // vectors per token
    const int width = vpt < 256 ? vpt : 256;         // vectors handled by this CTA
    const int ngroups = 256 / width;
    const int vec = blockIdx.y * width + threadIdx.x % width;
    const int grp = threadIdx.x / width;
    const long long tok_bytes = (long long)bd.h_kv * kHeadDim * kEsz;

    float ak[kEpv], av[kEpv];
#pragma unroll
    for (int e = 0; e < kEpv; ++e) ak[e] = av[e] = 0.f;

    const int *bt = block_table + (long long)r * max_pages;
#pragma unroll 4
    for (int t = t0 + grp; t < t1; t += ngroups) {
        int pg = __ldg(bt + t / page_size);
        if (pg < 0 || pg >= num_pages) {
            set_status(status, FP_ERR_DEVICE_BOUNDS);
            continue;
        }
        long long off = ((long long)pg * page_size + t % page_size) * tok_bytes + (long long)vec * 16;
        int4 kv = __ldg(reinterpret_cast<const int4 *>(k_cache + off));
        int4 vv;
        if (!v_dim_major) {
            vv = __ldg(reinterpret_cast<const int4 *>(v_cache + off));
        } else {
            // [num_pages, h_kv, d, page_size]: this vector's kEpv values of token t
            // sit page_size elements apart
            const long long e0 = ((long long)pg * bd.h_kv * kHeadDim + (long long)vec * kEpv) * page_size + t % page_size;
            uint32_t w4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w = 0;
#pragma unroll
                for (int b = 0; b < 4 / kEsz; ++b) {
                    const long long e = e0 + (long long)(q * (4 / kEsz) + b) * page_size;
                    const uint32_t x = kFp8 ? (uint32_t)__ldg(v_cache + e)
                                            : (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(v_cache) + e);
                    w |= x << (8 * kEsz * b);
                }
                w4[q] = w;
            }
            vv = make_int4((int)w4[0], (int)w4[1], (int)w4[2], (int)w4[3]);
        }
        const uint32_t *kw = reinterpret_cast<const uint32_t *>(&kv);
        const uint32_t *vw = reinterpret_cast<const uint32_t *>(&vv);
        if constexpr (!kFp8) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kw[w]));
                float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vw[w]));
                ak[2 * w] += a.x; ak[2 * w + 1] += a.y;
                av[2 * w] += b.x; av[2 * w + 1] += b.y;
            }
        } else {
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                __nv_fp8x2_storage_t ks = (__nv_fp8x2_storage_t)(kw[w / 2] >> (16 * (w & 1)));
                __nv_fp8x2_storage_t vs = (__nv_fp8x2_storage_t)(vw[w / 2] >> (16 * (w & 1)));
                float2 a = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(ks, __NV_E4M3)));
                float2 b = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(vs, __NV_E4M3)));
                ak[2 * w] += a.x; ak[2 * w + 1] += a.y;
                av[2 * w] += b.x; av[2 * w + 1] += b.y;
            }
        }
    }

    const int col = threadIdx.x % width;
    const float inv_n = 1.f / (float)n;
    const int head = vec * kEpv / kHeadDim;
    const float ks = kFp8 ? __ldg(k_scale + head) : 1.f;
    const float vs = kFp8 ? __ldg(v_scale + head) : 1.f;
    float *kout = k_mean + (long long)kb * bd.h_kv * kHeadDim + (long long)vec * kEpv;
    float *vout = v_mean + (long long)kb * bd.h_kv * kHeadDim + (long long)vec * kEpv;

    for (int pass = 0; pass < 2; ++pass) {
        const float *acc = pass == 0 ? ak : av;
#pragma unroll
        for (int e = 0; e < kEpv; ++e) red[(grp * width + col) * kEpv + e] = acc[e];
        __syncthreads();
        if (grp == 0) {
            float s[kEpv];
#pragma unroll
            for (int e = 0; e < kEpv; ++e) s[e] = 0.f;
            for (int q = 0; q < ngroups; ++q)
#pragma unroll
                for (int e = 0; e < kEpv; ++e) s[e] += red[(q * width + col) * kEpv + e];
            float mul = inv_n * (pass == 0 ? ks : vs);
            float *out = pass == 0 ? kout : vout;
#pragma unroll
            for (int e = 0; e < kEpv; e += 4)
                *reinterpret_cast<float4 *>(out + e) =
                    make_float4(s[e] * mul, s[e + 1] * mul, s[e + 2] * mul, s[e + 3] * mul);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// score: one CTA per score row (request, query block i, kv head h).  For each
// of the g query heads of the group, a 128-query tile is held in shared memory
// (fp32, pre-multiplied by scale*log2(e)); two passes over the pooled keys of
// blocks 0..I (64 at a time): the first finds every query's maximum, the
// second sums exp2(s - max) down the query dimension.  fp32 FMA throughout so
// that scores near the threshold are decided like the float64 definition.
// ---------------------------------------------------------------------------
constexpr int kScTileCols = 64;
constexpr int kScoreThreads = 256;

template <bool kFp8>
__global__ void __launch_bounds__(kScoreThreads, 2)
score_kernel(const __grid_constant__ BatchDesc bd, const uint8_t *__restrict__ q, long long q_stride_tok,
             long long q_stride_head, const float *__restrict__ q_scale,
             const float *__restrict__ k_mean, float scale_log2, float *__restrict__ score) {
    extern __shared__ __align__(16) float smem[];
    float *Qs = smem;                                  // [128 d][128 rows]
    float *Ks = Qs + kHeadDim * kBlock;                // [128 d][64 cols]
    float *part = Ks + kHeadDim * kScTileCols;         // [16][64]
    float *rowm = part + 16 * kScTileCols;             // [128]
    float *colsum = rowm + kBlock;                     // [max_nkb]

    const int row = bd.total_rows - 1 - blockIdx.x;    // heavy (late) rows first
    const int r = req_of_row(bd, row);
    const ReqDesc &rq = bd.req[r];
    const int local = row - rq.row_base;
    const int i = local / bd.h_kv;
    const int h = local % bd.h_kv;
    const int I = rq.start / kBlock + i;
    const int ncol = I + 1;
    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;            // 8 rows x 4 cols per thread

    for (int c = tid; c < ncol; c += kScoreThreads) colsum[c] = 0.f;

    for (int hh = h * bd.g; hh < (h + 1) * bd.g; ++hh) {
        const float qmul = scale_log2 * (kFp8 ? __ldg(q_scale + hh) : 1.f);
        __syncthreads();
        // Q tile -> Qs (transposed), rows past the request are zero
        for (int v = tid; v < kBlock * kHeadDim / 8; v += kScoreThreads) {
            int rr = v / (kHeadDim / 8), c8 = (v % (kHeadDim / 8)) * 8;
            int qi = i * kBlock + rr;
            float x[8];
            if (qi < rq.lq) {
                const uint8_t *src = q + ((long long)(rq.q_off + qi) * q_stride_tok +
                                          (long long)hh * q_stride_head + c8) * (kFp8 ? 1 : 2);
                if constexpr (!kFp8) {
                    int4 w = __ldg(reinterpret_cast<const int4 *>(src));
                    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 f = __bfloat1622float2(b[e]);
                        x[2 * e] = f.x; x[2 * e + 1] = f.y;
                    }
                } else {
                    uint2 w = __ldg(reinterpret_cast<const uint2 *>(src));
                    const uint32_t ww[2] = {w.x, w.y};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_fp8x2_storage_t s2 = (__nv_fp8x2_storage_t)(ww[e / 2] >> (16 * (e & 1)));
                        float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(s2, __NV_E4M3)));
                        x[2 * e] = f.x; x[2 * e + 1] = f.y;
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) Qs[(c8 + e) * kBlock + rr] = x[e] * qmul;
        }

        float m[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) m[a] = -INFINITY;

        for (int pass = 0; pass < 2; ++pass) {
            for (int c0 = 0; c0 < ncol; c0 += kScTileCols) {
                __syncthreads();
                for (int v = tid; v < kScTileCols * kHeadDim / 4; v += kScoreThreads) {
                    int cc = v / (kHeadDim / 4), d4 = (v % (kHeadDim / 4)) * 4;
                    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (c0 + cc < ncol)
                        f = __ldg(reinterpret_cast<const float4 *>(
                            k_mean + ((long long)(rq.kb_base + c0 + cc) * bd.h_kv + h) * kHeadDim + d4));
                    Ks[(d4 + 0) * kScTileCols + cc] = f.x;
                    Ks[(d4 + 1) * kScTileCols + cc] = f.y;
                    Ks[(d4 + 2) * kScTileCols + cc] = f.z;
                    Ks[(d4 + 3) * kScTileCols + cc] = f.w;
                }
                __syncthreads();
                float acc[8][4];
#pragma unroll
                for (int a = 0; a < 8; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
                for (int k = 0; k < kHeadDim; ++k) {
                    float4 qa = *reinterpret_cast<const float4 *>(Qs + k * kBlock + ty * 8);
                    float4 qb = *reinterpret_cast<const float4 *>(Qs + k * kBlock + ty * 8 + 4);
                    float4 kk = *reinterpret_cast<const float4 *>(Ks + k * kScTileCols + tx * 4);
                    float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                    float kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
                    for (int a = 0; a < 8; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qv[a], kv[b], acc[a][b]);
                }
                if (pass == 0) {
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        if (c0 + tx * 4 + b < ncol)
#pragma unroll
                            for (int a = 0; a < 8; ++a) m[a] = fmaxf(m[a], acc[a][b]);
                } else {
                    float cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int a = 0; a < 8; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b) cs[b] += fast_exp2(acc[a][b] - m[a]);
#pragma unroll
                    for (int b = 0; b < 4; ++b) part[ty * kScTileCols + tx * 4 + b] = cs[b];
                    __syncthreads();
                    if (tid < kScTileCols && c0 + tid < ncol) {
                        float s = 0.f;
                        for (int yy = 0; yy < 16; ++yy) s += part[yy * kScTileCols + tid];
                        colsum[c0 + tid] += s;
                    }
                }
            }
            if (pass == 0) {
                // row maxima: the 16 threads sharing rows are adjacent lanes
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    float v = m[a];
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    int qi = i * kBlock + ty * 8 + a;
                    m[a] = qi < rq.lq ? v : INFINITY;   // rows past the request add exp2(-inf) = 0
                }
            }
        }
    }
    __syncthreads();
    // re-normalise by the row maximum and store
    float mx = 0.f;
    for (int c = tid; c < ncol; c += kScoreThreads) mx = fmaxf(mx, colsum[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) part[tid / 32] = mx;
    __syncthreads();
    if (tid == 0) {
        float v = part[0];
        for (int w = 1; w < kScoreThreads / 32; ++w) v = fmaxf(v, part[w]);
        rowm[0] = v;
    }
    __syncthreads();
    const float inv = 1.f / rowm[0];
    float *out = score + score_row_offset(rq, bd.h_kv, i, h);
    for (int c = tid; c < ncol; c += kScoreThreads) out[c] = colsum[c] == rowm[0] ? 1.f : colsum[c] * inv;
}

size_t score_smem_bytes(int max_nkb) {
    return sizeof(float) * ((size_t)kHeadDim * kBlock + (size_t)kHeadDim * kScTileCols +
                            16 * kScTileCols + kBlock + (size_t)max_nkb);
}

cudaError_t launch_pool(const BatchDesc &bd, bool fp8, const void *k_cache, const void *v_cache,
                        int page_size, int num_pages, const int *block_table, int max_pages,
                        const float *k_scale, const float *v_scale, float *k_mean, float *v_mean,
                        int *status, cudaStream_t st, bool v_dim_major) {
    const int epv = fp8 ? 16 : 8;
    const int vpt = bd.h_kv * kHeadDim / epv;
    dim3 grid(bd.total_kb, vpt > 256 ? vpt / 256 : 1);
    if (fp8)
        pool_kernel<true><<<grid, 256, 0, st>>>(bd, (const uint8_t *)k_cache, (const uint8_t *)v_cache,
                                                page_size, num_pages, block_table, max_pages, k_scale,
                                                v_scale, k_mean, v_mean, status, v_dim_major ? 1 : 0);
    else
        pool_kernel<false><<<grid, 256, 0, st>>>(bd, (const uint8_t *)k_cache, (const uint8_t *)v_cache,
                                                 page_size, num_pages, block_table, max_pages, k_scale,
                                                 v_scale, k_mean, v_mean, status, v_dim_major ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_score(const BatchDesc &bd, bool fp8, const void *q, long long q_stride_tok,
                         long long q_stride_head, const float *q_scale, const float *k_mean,
                         float softmax_scale, float *score, cudaStream_t st) {
    size_t smem = score_smem_bytes(bd.max_nkb);
    const float scale_log2 = softmax_scale * 1.4426950408889634f;
    cudaError_t e;
    if (fp8) {
        e = cudaFuncSetAttribute(score_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        score_kernel<true><<<bd.total_rows, kScoreThreads, smem, st>>>(
            bd, (const uint8_t *)q, q_stride_tok, q_stride_head, q_scale, k_mean, scale_log2, score);
    } else {
        e = cudaFuncSetAttribute(score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        score_kernel<false><<<bd.total_rows, kScoreThreads, smem, st>>>(
            bd, (const uint8_t *)q, q_stride_tok, q_stride_head, q_scale, k_mean, scale_log2, score);
    }
    return cudaGetLastError();
}

}  // namespace fp
