// Block-score map on tcgen05 tensor cores (bf16 inputs).
//
// The scores of the FlashPrefill V1 summary, section 3.1 (per packed query
// row: logits against the pooled keys, normalised by the row's own maximum,
// exponentiated and summed over the query block; then each score row divided
// by its largest entry) decide, through a threshold, which blocks are kept.
// Decisions must not move relative to the float64 definition, so the pooled
// keys enter the MMA as three bf16 terms, kmean = hi + mid + lo (24
// significant bits, like fp32); Q is exactly representable in bf16 (and e4m3
// inputs would be too, but those use the fp32 CUDA-core kernel).
//
// One CTA per score row (request, query block I, kv head h):
//   for each query head of the group (128-query tile, M = 128):
//     pass 0: S = Q Kmean^T over the row's key blocks 0..I, 64 at a time -> row max
//     pass 1: the same S again -> exp2((s - max) * scale * log2 e), summed down
//             the 128 queries (a transpose-reduce across each warp's 32 rows)
//             and accumulated into the score row in global memory;
//   finally the row is divided by its maximum.
// Warp 0 issues TMA loads (Q per head, the three mean terms per 64-block
// chunk, 3-stage ring), warp 1 issues the MMAs into four 64-column TMEM
// buffers, warps 4-7 read S from TMEM (one query row per thread).
#include "common.cuh"
#include "launch.cuh"
#include "sm100.cuh"

namespace fp {

using namespace sm100;

namespace {

constexpr int kScThreads = 256;
constexpr int kChunk = 64;                                 // key blocks per chunk (MMA N)
constexpr int kQBytes = kBlock * kHeadDim * 2;             // 32 KB
constexpr int kTermBytes = kChunk * kHeadDim * 2;          // 16 KB: one term of one chunk
constexpr int kStageBytes = 3 * kTermBytes;                // 48 KB
constexpr int kStages = 3;
constexpr int kTmemBufs = 4;
constexpr int kSmQ = 0;
constexpr int kSmStage = 2 * kQBytes;                      // 64 KB
constexpr int kSmPart = kSmStage + kStages * kStageBytes;  // 208 KB
constexpr int kSmCtl = kSmPart + 2 * 4 * kChunk * 4;       // + 2 KB partial sums
constexpr int kScoreTcSmem = kSmCtl + 256 + 1024;

enum { B_QF = 0, B_QE = 2, B_SF = 4, B_SE = 7, B_TF = 10, B_TE = 14, B_N = 18 };

struct ScoreTcArgs {
    float *score;
    float scale_log2;
    int rows_pad;             // rows of each mean term in the split array
    int *status;
    unsigned long long wait_ns;
};

// A barrier among the four row warps that cannot hang: each warp's lane 0
// adds one arrival to a shared counter and spins (bounded, like the mbarrier
// waits) until all four warps of this generation have arrived.  Returns false
// if the CTA is aborting.
__device__ __forceinline__ bool rows_sync(unsigned *ctr, unsigned &gen, int lane, volatile int *abort_flag,
                                          int *status, unsigned long long wait_ns) {
    gen += 4;
    bool ok = true;
    __threadfence_block();          // this lane's shared / global writes before the arrival
    __syncwarp();
    if (lane == 0) {
        atomicAdd(ctr, 1u);
        volatile unsigned *vc = ctr;
        const uint64_t t0 = global_ns();
        for (uint32_t it = 0; *vc < gen; ++it) {
            if ((it & 63u) == 63u) {
                if (*abort_flag) { ok = false; break; }
                if (global_ns() - t0 > wait_ns) {
                    set_status(status, FP_ERR_TIMEOUT);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
            }
        }
    }
    __syncwarp();
    __threadfence_block();          // the other warps' writes are visible from here on
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok;
}

// Column sums of a 32x32 block held one row per lane (v[c] = column c of
// this lane's row): after the butterfly, lane L holds the sum of column L.
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const bool up = lane & 16;
        const float send = up ? v[k] : v[k + 16];
        const float keep = up ? v[k + 16] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const bool up = lane & 8;
        const float send = up ? v[k] : v[k + 8];
        const float keep = up ? v[k + 8] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool up = lane & 4;
        const float send = up ? v[k] : v[k + 4];
        const float keep = up ? v[k + 4] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool up = lane & 2;
        const float send = up ? v[k] : v[k + 2];
        const float keep = up ? v[k + 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const bool up = lane & 1;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__global__ void __launch_bounds__(kScThreads, 1)
score_tc_kernel(const __grid_constant__ BatchDesc bd, const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ CUtensorMap tmM, const ScoreTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *part = reinterpret_cast<float *>(smem + kSmPart);            // [2][4 warps][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kSmCtl);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kSmCtl + B_N * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kSmCtl + B_N * 8 + 4);
    float *red = reinterpret_cast<float *>(smem + kSmCtl + B_N * 8 + 16);   // [4]
    unsigned *sync_ctr = reinterpret_cast<unsigned *>(smem + kSmCtl + B_N * 8 + 32);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int k) { return smem_u32(&bars[k]); };

    const int row = bd.total_rows - 1 - blockIdx.x;           // heavy (late) rows first
    const int r = req_of_row(bd, row);
    const ReqDesc &rq = bd.req[r];
    const int local = row - rq.row_base;
    const int il = local / bd.h_kv;
    const int h = local % bd.h_kv;
    const int I = rq.start / kBlock + il;
    const int ncol = I + 1;
    const int nch = (ncol + kChunk - 1) / kChunk;
    const int g = bd.g;
    float *out = a.score + score_row_offset(rq, bd.h_kv, il, h);

    if (threadIdx.x == 0) {
        for (int k = 0; k < B_N; ++k) mbar_init(bar(k), (k >= B_TE && k < B_TE + kTmemBufs) ? 128u : 1u);
        *abort_flag = 0;
        *sync_ctr = 0u;
        fence_barrier_init();
        fence_proxy_async();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmM);
            int item = 0;
            for (int hh = 0; hh < g && !*abort_flag; ++hh) {
                const int qb = hh & 1;
                if (hh >= 2 && !mbar_wait(bar(B_QE + qb), ((hh >> 1) - 1) & 1, abort_flag, a.status, a.wait_ns))
                    break;
                mbar_expect_tx(bar(B_QF + qb), kQBytes);
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_3d(sbase + kSmQ + qb * kQBytes + hf * (kQBytes / 2), &tmQ, bar(B_QF + qb), hf * 64,
                                h * g + hh, rq.q_off + il * kBlock);
                for (int pass = 0; pass < 2; ++pass)
                    for (int c = 0; c < nch; ++c, ++item) {
                        const int s = item % kStages, use = item / kStages;
                        if (item >= kStages &&
                            !mbar_wait(bar(B_SE + s), (use - 1) & 1, abort_flag, a.status, a.wait_ns))
                            goto producer_done;
                        mbar_expect_tx(bar(B_SF + s), kStageBytes);
                        const uint32_t dst = sbase + kSmStage + s * kStageBytes;
                        for (int t = 0; t < 3; ++t)
                            for (int hf = 0; hf < 2; ++hf)
                                tma_load_3d(dst + t * kTermBytes + hf * (kTermBytes / 2), &tmM, bar(B_SF + s),
                                            hf * 64, h, t * a.rows_pad + rq.kb_base + c * kChunk);
                    }
            }
        producer_done:;
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(128, kChunk, false);
            int item = 0;
            for (int hh = 0; hh < g; ++hh) {
                const int qb = hh & 1;
                if (!mbar_wait(bar(B_QF + qb), (hh >> 1) & 1, abort_flag, a.status, a.wait_ns)) goto mma_done;
                const uint32_t qa = sbase + kSmQ + qb * kQBytes;
                for (int pass = 0; pass < 2; ++pass)
                    for (int c = 0; c < nch; ++c, ++item) {
                        const int s = item % kStages, b = item % kTmemBufs;
                        if (!mbar_wait(bar(B_SF + s), (item / kStages) & 1, abort_flag, a.status, a.wait_ns))
                            goto mma_done;
                        if (item >= kTmemBufs &&
                            !mbar_wait(bar(B_TE + b), ((item / kTmemBufs) - 1) & 1, abort_flag, a.status,
                                       a.wait_ns))
                            goto mma_done;
                        tc_fence_after();
                        const uint32_t kb = sbase + kSmStage + s * kStageBytes;
#pragma unroll
                        for (int t = 0; t < 3; ++t)
#pragma unroll
                            for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                                const uint32_t off = (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32;
                                const uint32_t boff = t * kTermBytes + (kk >> 2) * (kTermBytes / 2) + (kk & 3) * 32;
                                mma_ss(tmem + b * kChunk, smem_desc_sw128(qa + off, 16, 1024),
                                       smem_desc_sw128(kb + boff, 16, 1024), idS, (t | kk) != 0);
                            }
                        tc_commit(bar(B_TF + b));
                        tc_commit(bar(B_SE + s));
                    }
                tc_commit(bar(B_QE + qb));
            }
        mma_done:;
        }
    } else if (warp >= 4) {
        // ================= row warpgroup: one query row per thread =================
        const int quarter = warp - 4;
        const int rowt = quarter * 32 + lane;
        const bool row_valid = il * kBlock + rowt < rq.lq;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        int item = 0;
        bool ok = true;
        unsigned gen = 0;
        for (int hh = 0; hh < g && ok; ++hh) {
            const float c2 = a.scale_log2;
            float m = -INFINITY;
            float mc2 = 0.f;
            for (int pass = 0; pass < 2 && ok; ++pass) {
                if (pass == 1) mc2 = (m == -INFINITY || !row_valid) ? 0.f : m * c2;
                for (int c = 0; c < nch; ++c, ++item) {
                    const int b = item % kTmemBufs;
                    const bool got = mbar_wait(bar(B_TF + b), (item / kTmemBufs) & 1, abort_flag, a.status, a.wait_ns);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    tc_fence_after();
                    uint32_t u0[32], u1[32];
                    tmem_ld32(lane_base + b * kChunk, u0);
                    tmem_ld32(lane_base + b * kChunk + 32, u1);
                    tmem_ld_wait();
                    reg_fence(u0);
                    reg_fence(u1);
                    tc_fence_before();
                    mbar_arrive(bar(B_TE + b));
                    const int J0 = c * kChunk;
                    if (pass == 0) {
                        float m4[4] = {m, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            if (J0 + e < ncol) m4[e & 3] = fmaxf(m4[e & 3], __uint_as_float(u0[e]));
                            if (J0 + 32 + e < ncol) m4[(e + 2) & 3] = fmaxf(m4[(e + 2) & 3], __uint_as_float(u1[e]));
                        }
                        m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                    } else {
                        float v0[32], v1[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            v0[e] = (row_valid && J0 + e < ncol) ? fast_exp2(fmaf(__uint_as_float(u0[e]), c2, -mc2)) : 0.f;
                            v1[e] = (row_valid && J0 + 32 + e < ncol) ? fast_exp2(fmaf(__uint_as_float(u1[e]), c2, -mc2)) : 0.f;
                        }
                        const float s0 = transpose_reduce32(v0, lane);
                        const float s1 = transpose_reduce32(v1, lane);
                        float *pp = part + (item & 1) * 4 * kChunk + quarter * kChunk;
                        pp[lane] = s0;
                        pp[32 + lane] = s1;
                        if (!rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns)) { ok = false; break; }
                        const int t = threadIdx.x - 128;
                        if (t < kChunk && J0 + t < ncol) {
                            const float *q = part + (item & 1) * 4 * kChunk;
                            const float v = (q[t] + q[kChunk + t]) + (q[2 * kChunk + t] + q[3 * kChunk + t]);
                            out[J0 + t] = hh == 0 ? v : out[J0 + t] + v;
                        }
                    }
                }
            }
        }
        // re-normalise the row by its maximum
        if (ok) ok = rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns);
        if (ok) {
            const int t = threadIdx.x - 128;
            float mx = 0.f;
            for (int J = t; J < ncol; J += 128) mx = fmaxf(mx, out[J]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) red[quarter] = mx;
            if (!rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns)) mx = 0.f;
            mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
            const float inv = 1.f / mx;
            if (!*abort_flag)
            for (int J = t; J < ncol; J += 128) {
                const float v = out[J];
                out[J] = v == mx ? 1.f : v * inv;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// fp32 block means -> three bf16 terms (hi, mid, lo) whose sum carries 24
// significant bits; rows past the last block are zero.
__global__ void split_means_kernel(const float *__restrict__ km, __nv_bfloat16 *__restrict__ terms, long long n,
                                   long long n_pad) {
    for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < n_pad;
         k += (long long)gridDim.x * blockDim.x) {
        const float x = k < n ? km[k] : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const float r1 = x - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        terms[k] = hi;
        terms[n_pad + k] = mid;
        terms[2 * n_pad + k] = __float2bfloat16_rn(r2);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_sc() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

bool map3(CUtensorMap *m, const void *base, long long n1, long long n2, long long s1, long long s2, int box2) {
    EncodeTiledFn fn = encode_fn_sc();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)n1, (cuuint64_t)n2};
    cuuint64_t strides[2] = {(cuuint64_t)(s1 * 2), (cuuint64_t)(s2 * 2)};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box2};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int score_tc_rows_pad(const BatchDesc &bd) { return bd.total_kb > kChunk ? bd.total_kb : kChunk; }

cudaError_t launch_score_tc(const BatchDesc &bd, const void *q, long long q_stride_tok, long long q_stride_head,
                            const float *k_mean, float softmax_scale, float *score, __nv_bfloat16 *terms,
                            int *status, unsigned long long wait_ns, cudaStream_t st) {
    const int rows_pad = score_tc_rows_pad(bd);
    const long long n = (long long)bd.total_kb * bd.h_kv * kHeadDim;
    const long long n_pad = (long long)rows_pad * bd.h_kv * kHeadDim;
    split_means_kernel<<<512, 256, 0, st>>>(k_mean, terms, n, n_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap tmQ, tmM;
    if (!map3(&tmQ, q, bd.h_q, bd.total_q, q_stride_head, q_stride_tok, kBlock)) return cudaErrorInvalidValue;
    if (!map3(&tmM, terms, bd.h_kv, 3LL * rows_pad, kHeadDim, (long long)bd.h_kv * kHeadDim, kChunk))
        return cudaErrorInvalidValue;
    ScoreTcArgs a;
    a.score = score;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.rows_pad = rows_pad;
    a.status = status;
    a.wait_ns = wait_ns;
    e = cudaFuncSetAttribute(score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreTcSmem);
    if (e != cudaSuccess) return e;
    score_tc_kernel<<<bd.total_rows, kScThreads, kScoreTcSmem, st>>>(bd, tmQ, tmM, a);
    return cudaGetLastError();
}

}  // namespace fp
