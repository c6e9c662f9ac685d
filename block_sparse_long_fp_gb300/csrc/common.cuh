// Shared definitions of the CUDA library: the per-batch descriptor passed by
// value to every kernel, request lookup, the device status word, and small
// numeric helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fprefill.h"

namespace fp {

constexpr int kBlock = 128;     // tokens per query / key block
constexpr int kHeadDim = 128;   // d

// 2^e as a float, for |e| <= 126
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// The power-of-two exponent that brings a largest magnitude (its fp32 bit
// pattern) into [2^14, 2^15): under fp16's largest finite value, with 2^29
// of range below it, so that fp16 holds bf16 values and e4m3 codes exactly and
// the two fp16 terms of an fp32 value carry 22 significant bits.  0 for a zero
// (or subnormal) maximum; clamped so that 2^e and 2^-e stay normal floats.
__host__ __device__ __forceinline__ int fp16_scale_exp(uint32_t max_bits) {
    const int E = (int)((max_bits >> 23) & 0xffu);
    if (E == 0) return 0;
    const int e = 141 - E;
    return e < -100 ? -100 : (e > 100 ? 100 : e);
}

// One request of a varlen batch, as every kernel sees it (computed on the
// host from the host descriptors).
struct ReqDesc {
    int q_off;        // first query row (cu_seqlens_q[r])
    int lq;           // queries
    int lk;           // keys (= start + lq)
    int start;        // absolute position of query 0 (multiple of kBlock)
    int nqb;          // ceil(lq / B)
    int nkb;          // ceil(lk / B)
    int row_base;     // first index/score row of the request
    int kb_base;      // first pooled block of the request
    long long score_base;  // first score-map entry of the request
};

struct BatchDesc {
    int batch;
    int h_q, h_kv, g;
    int total_q;
    int total_rows;
    int total_kb;
    int max_nkb;
    long long score_size;
    ReqDesc req[FP_MAX_BATCH];
};

// Status header at the start of every workspace.
struct WsHeader {
    int status;
    int pad[63];
};
constexpr size_t kWsHeaderBytes = 256;

__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Fused selection: a score row of ncol entries is cut into 8 segments of
// this many (a multiple of 32), one per row warp of the score kernel.
__host__ __device__ __forceinline__ int score_segment(int ncol) { return ((ncol + 7) / 8 + 31) / 32 * 32; }

// Request owning global row `row` (rows are request-major).
__device__ __forceinline__ int req_of_row(const BatchDesc &bd, int row) {
    int lo = 0, hi = bd.batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (bd.req[mid].row_base <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Request owning global pooled block `kb`.
__device__ __forceinline__ int req_of_kb(const BatchDesc &bd, int kb) {
    int lo = 0, hi = bd.batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (bd.req[mid].kb_base <= kb) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Offset of score row (i, h) of request `rq` (the layout in fprefill.h).
__host__ __device__ __forceinline__ long long score_row_offset(const ReqDesc &rq, int h_kv, int i, int h) {
    long long I0 = rq.start / kBlock;
    return rq.score_base + (long long)h_kv * (i * (I0 + 1) + (long long)i * (i - 1) / 2) +
           (long long)h * (I0 + i + 1);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace fp
