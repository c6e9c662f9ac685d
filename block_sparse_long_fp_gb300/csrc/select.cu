// fp_select kernels: the max-based dynamic threshold with the sink / local
// safety net (FlashPrefill V1 summary, section 3.2; V2 paper reading, section
// 4: 256 sink tokens, 512 local tokens, alpha = 0.1) and the compaction of the
// kept key blocks into a CSR index (V1 section 3.3 "index-driven physical
// jump"; V2 section 4 CSR output).  The top-k and top-p rules the V1 summary
// (section 4.4) compares the threshold with are kept as ablations.
//
// One launch, no host synchronisation: one warp per row decides and counts;
// each CTA of eight rows learns the kept count of all earlier rows by a
// decoupled look-back over the CTAs' published totals (a bounded wait); then
// each warp writes row_ptr and its kept blocks at row_ptr[row].
#include <limits.h>

#include <atomic>

#include "common.cuh"
#include "launch.cuh"
#include "sm100.cuh"

namespace fp {

struct SelectArgs {
    float alpha;
    int sink_blocks;
    int local_blocks;
    int rule;                 // fp_select_rule
    int top_k;
    float top_p;
};

// A row's decision: keep J when s > t, or s == t and J <= jt (jt: the last of
// the equal scores that still fit, top-k only), or J is a sink / local block.
struct RowRule {
    float t;
    int jt;
};

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Row maximum of a score row, reduced across the warp in a fixed order.
__device__ __forceinline__ float warp_row_max(const float *s, int n, int lane) {
    float mx = -INFINITY;
    for (int c = lane; c < n; c += 32) mx = fmaxf(mx, s[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    return mx;
}

// Scores are >= 0, so their bit patterns order like their values: the top-k
// and top-p thresholds are found by a binary search over the bit pattern (31
// steps), each step one pass over the row by the warp.  Every kernel that
// decides a row calls this with the same row, so all reach the same decision.
__device__ RowRule row_rule(const float *s, int n, int lane, const SelectArgs &a) {
    RowRule rr{0.f, INT_MAX};
    if (a.rule == FP_SELECT_THRESHOLD) {
        rr.t = a.alpha * warp_row_max(s, n, lane);      // keep s >= alpha * max
        return rr;
    }
    unsigned lo = 0u, hi = 0x7f800000u;
    if (a.rule == FP_SELECT_TOPK) {
        const int k = a.top_k < n ? a.top_k : n;
        while (lo < hi) {                                // the largest u with #(bits >= u) >= k
            const unsigned mid = lo + (hi - lo + 1u) / 2u;
            int c = 0;
            for (int J = lane; J < n; J += 32) c += __float_as_uint(__ldg(s + J)) >= mid;
            if (warp_sum(c) >= k) lo = mid;
            else hi = mid - 1u;
        }
        rr.t = __uint_as_float(lo);
        int gt = 0;
        for (int J = lane; J < n; J += 32) gt += __float_as_uint(__ldg(s + J)) > lo;
        const int need = k - warp_sum(gt);              // equal scores to keep, lowest J first (>= 1)
        int seen = 0;
        rr.jt = -1;
        for (int J0 = 0; J0 < n; J0 += 32) {
            const int J = J0 + lane;
            const unsigned m = __ballot_sync(0xffffffffu, J < n && __float_as_uint(__ldg(s + J)) == lo);
            const int c = __popc(m);
            if (seen + c >= need) {
                unsigned mm = m;
                for (int q = 1; q < need - seen; ++q) mm &= mm - 1u;
                rr.jt = J0 + __ffs(mm) - 1;
                break;
            }
            seen += c;
        }
        return rr;
    }
    // top-p: the largest u whose scores >= u hold top_p of the row's total.  A
    // subset's sum never rounds above its superset's (same order, adding
    // non-negative terms), so the mass is monotone in u.
    float tot = 0.f;
    for (int J = lane; J < n; J += 32) tot += __ldg(s + J);
    const float target = a.top_p * warp_sum(tot);
    while (lo < hi) {
        const unsigned mid = lo + (hi - lo + 1u) / 2u;
        float m = 0.f;
        for (int J = lane; J < n; J += 32) {
            const float v = __ldg(s + J);
            m += __float_as_uint(v) >= mid ? v : 0.f;
        }
        if (warp_sum(m) >= target) lo = mid;
        else hi = mid - 1u;
    }
    rr.t = __uint_as_float(lo);
    return rr;
}

__device__ __forceinline__ bool keep_block(float s, const RowRule &rr, int J, int I, const SelectArgs &a) {
    return s > rr.t || (s == rr.t && J <= rr.jt) || J < a.sink_blocks || J >= I - a.local_blocks + 1;
}

// Look-back state of one CTA: bits [62, 64) status (0: nothing yet, 1: the
// CTA's own total, 2: the inclusive total of all rows up to its last), [32,
// 62) the call's epoch (a state left by an earlier call reads as nothing
// yet, so the array needs no clearing), [0, 32) the value.
constexpr unsigned long long kLbAgg = 1ull << 62, kLbPrefix = 2ull << 62;
__device__ __forceinline__ unsigned long long lb_word(unsigned long long status, unsigned epoch, int v) {
    return status | ((unsigned long long)(epoch & 0x3fffffffu) << 32) | (unsigned)v;
}
__device__ __forceinline__ void lb_publish(unsigned long long *p, unsigned long long w) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long lb_read(const unsigned long long *p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

constexpr int kRegRow = 1024;      // rows of up to this many blocks decide from registers

// at most 64 registers, so that four CTAs fit on an SM: the 512 CTAs of a
// 4096-row map then run in one wave (at 128 registers two fit, and the last
// CTAs started ~9 us late), at the cost of a few spilled bytes
__global__ void __launch_bounds__(256, 4)
select_kernel(const __grid_constant__ BatchDesc bd, SelectArgs a, const float *__restrict__ score,
              unsigned long long *__restrict__ lb_state, unsigned epoch, int *__restrict__ row_ptr,
              int *__restrict__ col_idx, long long col_capacity, int *__restrict__ nnz,
              unsigned char *__restrict__ dense_mask, int *status, unsigned long long wait_ns) {
    __shared__ int cnt[8];
    __shared__ int cta_base;
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int row = blockIdx.x * 8 + w;
    const bool have = row < bd.total_rows;
    int I = 0, c = 0;
    long long off = 0;
    RowRule rr{0.f, INT_MAX};
    // threshold rule on a row of at most kRegRow blocks: the row is read once,
    // 32 scores per lane in registers (all loads in flight at once), and the
    // maximum, the count and the compaction work from there; keep bit k of
    // `kept` = block 32 k + lane
    const bool in_regs = a.rule == FP_SELECT_THRESHOLD;
    uint32_t kept = 0u;
    if (have) {
        const int r = req_of_row(bd, row);
        const ReqDesc &rq = bd.req[r];
        const int local = row - rq.row_base;
        const int i = local / bd.h_kv, h = local % bd.h_kv;
        I = rq.start / kBlock + i;
        off = score_row_offset(rq, bd.h_kv, i, h);
        const float *s = score + off;
        if (in_regs && I < kRegRow) {
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int J = 32 * k + lane;
                v[k] = J <= I ? __ldg(s + J) : -INFINITY;
            }
            float mx = v[0];
#pragma unroll
            for (int k = 1; k < 32; ++k) mx = fmaxf(mx, v[k]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            rr.t = a.alpha * mx;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int J = 32 * k + lane;
                const bool kb = J <= I && keep_block(v[k], rr, J, I, a);
                kept |= (uint32_t)kb << k;
                if (dense_mask && J <= I) dense_mask[off + J] = (unsigned char)kb;
            }
            c = __popc(kept);
        } else {
            rr = row_rule(s, I + 1, lane, a);
            for (int J = lane; J <= I; J += 32) {
                const bool k = keep_block(__ldg(s + J), rr, J, I, a);
                c += k;
                if (dense_mask) dense_mask[off + J] = (unsigned char)k;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    if (lane == 0) cnt[w] = c;
    __syncthreads();
    if (w == 0) {
        int agg = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) agg += cnt[k];
        int excl = 0;
        if (blockIdx.x > 0) {
            if (lane == 0) lb_publish(lb_state + blockIdx.x, lb_word(kLbAgg, epoch, agg));
            // warp-wide look-back over windows of 128 earlier CTAs: lane L reads
            // CTAs end - (32 q + L), q = 0..3, all four loads in flight; the
            // nearest CTA with an inclusive total ends the walk and the CTAs
            // between that published their own totals are added; a window of
            // 128 own totals moves the window back (bounded like every wait here)
            const uint64_t t0 = sm100::global_ns();
            for (int end = blockIdx.x - 1;;) {
                unsigned long long st[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int b = end - 32 * q - lane;
                    st[q] = b >= 0 ? lb_read(lb_state + b) : lb_word(kLbPrefix, epoch, 0);
                }
                bool done = false, step = true;
                int add = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const bool mine = ((st[q] >> 32) & 0x3fffffffu) == (epoch & 0x3fffffffu);
                    const unsigned kind = mine ? (unsigned)(st[q] >> 62) : 0u;   // 0: not yet published
                    const int val = (int)(unsigned)st[q];
                    const unsigned pre = __ballot_sync(0xffffffffu, kind == 2u);
                    const unsigned rdy = __ballot_sync(0xffffffffu, kind != 0u);
                    if (!done && step) {
                        if (pre) {
                            const int pl = __ffs(pre) - 1;                           // nearest inclusive total
                            const unsigned need = pl == 31 ? 0xffffffffu : ((2u << pl) - 1u);
                            if ((rdy & need) == need) {
                                add += lane <= pl ? val : 0;
                                done = true;
                            } else {
                                step = false;                                        // not all published yet
                            }
                        } else if (rdy == 0xffffffffu) {
                            add += val;
                        } else {
                            step = false;
                        }
                    }
                }
                if (done || step) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) add += __shfl_xor_sync(0xffffffffu, add, o);
                    excl += add;
                    if (done) break;
                    end -= 128;
                    continue;
                }
                if (__any_sync(0xffffffffu, sm100::global_ns() - t0 > wait_ns)) {   // warp-uniform
                    if (lane == 0) set_status(status, FP_ERR_TIMEOUT);
                    break;
                }
            }
        }
        if (lane == 0) {
            lb_publish(lb_state + blockIdx.x, lb_word(kLbPrefix, epoch, excl + agg));
            cta_base = excl;
        }
    }
    __syncthreads();
    if (!have) return;
    int pos = cta_base;
    for (int k = 0; k < w; ++k) pos += cnt[k];
    if (lane == 0) {
        row_ptr[row] = pos;
        if (row == bd.total_rows - 1) {
            row_ptr[row + 1] = pos + c;
            *nnz = pos + c;
        }
    }
    if ((long long)pos + c > col_capacity) {
        if (lane == 0) set_status(status, FP_ERR_INVALID);
        return;
    }
    if (in_regs && I < kRegRow) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (32 * k > I) break;
            const bool kb = (kept >> k) & 1u;
            const unsigned m = __ballot_sync(0xffffffffu, kb);
            if (kb) col_idx[pos + __popc(m & ((1u << lane) - 1u))] = 32 * k + lane;
            pos += __popc(m);
        }
        return;
    }
    const float *s = score + off;
    for (int J0 = 0; J0 <= I; J0 += 32) {
        const int J = J0 + lane;
        const bool k = J <= I && keep_block(__ldg(s + J), rr, J, I, a);
        const unsigned m = __ballot_sync(0xffffffffu, k);
        if (k) col_idx[pos + __popc(m & ((1u << lane) - 1u))] = J;
        pos += __popc(m);
    }
}

// Exclusive scan of the row counts into row_ptr[0..n], nnz = row_ptr[n]; row
// k's count is the sum of counts[k * per_row .. k * per_row + per_row).
__global__ void __launch_bounds__(1024)
scan_kernel(const int *__restrict__ counts, int n, int per_row, int *__restrict__ row_ptr, int *__restrict__ nnz) {
    __shared__ int warp_tot[32];
    const int tid = threadIdx.x;
    const int per = (n + 1023) / 1024;
    const int b = tid * per, e = min(n, b + per);
    auto count = [&](int k) {
        int c = 0;
        for (int q = 0; q < per_row; ++q) c += counts[(long long)k * per_row + q];
        return c;
    };
    int sum = 0;
    for (int k = b; k < e; ++k) sum += count(k);
    // inclusive scan of the per-thread sums
    int lane = tid % 32, w = tid / 32;
    int v = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[w] = v;
    __syncthreads();
    if (w == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += u;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    int run = v - sum + (w > 0 ? warp_tot[w - 1] : 0);
    for (int k = b; k < e; ++k) {
        row_ptr[k] = run;
        run += count(k);
    }
    if (tid == 1023) {
        int total = warp_tot[31];
        row_ptr[n] = total;
        *nnz = total;
    }
}

// fused path: row warp w of the score kernel wrote the kept blocks of segment
// w of the row at keep_pad[row offset + w * score_segment(I + 1)], and their
// count at counts8[row * 8 + w]; after the scan, one warp per row joins the
// segments into col_idx[row_ptr[row]..]
__global__ void __launch_bounds__(256)
select_gather_kernel(const __grid_constant__ BatchDesc bd, const int *__restrict__ keep_pad,
                     const int *__restrict__ counts8, const int *__restrict__ row_ptr, int *__restrict__ col_idx,
                     long long col_capacity, int *status) {
    const int row = blockIdx.x * 8 + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= bd.total_rows) return;
    const int r = req_of_row(bd, row);
    const ReqDesc &rq = bd.req[r];
    const int local = row - rq.row_base;
    const int i = local / bd.h_kv, h = local % bd.h_kv;
    const int *src = keep_pad + score_row_offset(rq, bd.h_kv, i, h);
    const int I = rq.start / kBlock + i;
    const int seg = score_segment(I + 1);
    const int b = row_ptr[row], n = row_ptr[row + 1] - b;
    if ((long long)b + n > col_capacity) {
        if (lane == 0) set_status(status, FP_ERR_INVALID);
        return;
    }
    int pos = b;
    for (int w = 0; w < 8; ++w) {
        const int c = __ldg(counts8 + (long long)row * 8 + w);
        for (int k = lane; k < c; k += 32) col_idx[pos + k] = __ldg(src + w * seg + k);
        pos += c;
    }
}

cudaError_t launch_select_gather(const BatchDesc &bd, const int *keep_pad, const int *counts, int *row_ptr,
                                 int *col_idx, long long col_capacity, int *nnz, int *status, cudaStream_t st) {
    const int grid = (bd.total_rows + 7) / 8;
    scan_kernel<<<1, 1024, 0, st>>>(counts, bd.total_rows, 8, row_ptr, nnz);
    select_gather_kernel<<<grid, 256, 0, st>>>(bd, keep_pad, counts, row_ptr, col_idx, col_capacity, status);
    return cudaGetLastError();
}

cudaError_t launch_select(const BatchDesc &bd, float alpha, int sink_blocks, int local_blocks, int rule,
                          int top_k, float top_p, const float *score, void *lb_state, int *row_ptr, int *col_idx,
                          long long col_capacity, int *nnz, unsigned char *dense_mask, int *status,
                          unsigned long long wait_ns, cudaStream_t st) {
    SelectArgs a{alpha, sink_blocks, local_blocks, rule, top_k, top_p};
    if (bd.total_rows == 0) {
        if (cudaMemsetAsync(row_ptr, 0, sizeof(int), st) != cudaSuccess) return cudaGetLastError();
        return cudaMemsetAsync(nnz, 0, sizeof(int), st);
    }
    // a new epoch per call: look-back states of earlier calls read as empty.
    // A graph replays the epoch it captured, so a call being captured clears
    // the states instead (a memset node ahead of the kernel in the graph).
    static std::atomic<unsigned> calls{0};
    const unsigned epoch = (calls.fetch_add(1u) % 0x3ffffffeu) + 1u;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return cudaGetLastError();
    if (cap != cudaStreamCaptureStatusNone && cudaMemsetAsync(lb_state, 0, select_state_bytes(bd), st) != cudaSuccess)
        return cudaGetLastError();
    const int grid = (bd.total_rows + 7) / 8;
    select_kernel<<<grid, 256, 0, st>>>(bd, a, score, static_cast<unsigned long long *>(lb_state), epoch, row_ptr,
                                        col_idx, col_capacity, nnz, dense_mask, status, wait_ns);
    return cudaGetLastError();
}

}  // namespace fp
