// Block-score map on tcgen05 tensor cores.
//
// The scores of the FlashPrefill V1 summary, section 3.1 (per packed query
// row: logits against the pooled keys, normalised by the row's own maximum,
// exponentiated and summed over the query block; then each score row divided
// by its largest entry) decide, through a threshold, which blocks are kept.
// Decisions must not move relative to the float64 definition (a block's score
// may move by far less than 1e-4 of the threshold), so the MMAs run on fp16
// operands near fp32 accuracy:
//  * the pooled keys of each chunk of 128 blocks and kv head are scaled by a
//    power of two 2^e (their largest magnitude lands in [2^14, 2^15)) and
//    enter as two fp16 terms, kmean * 2^e = hi + lo (22 significant bits);
//  * each query row is scaled by its own power of two 2^f the same way; bf16
//    values (8 significant bits) and e4m3 codes are exact in fp16 then;
//  * products of fp16 values are exact in the fp32 accumulator, and scaling
//    by powers of two commutes with its rounding, so 2^-(e+f) joins the
//    exponent's fp32 constant and the logits are those of the unscaled
//    operands.
//
// One CTA per score row (request, query block I, kv head h).  The g query
// heads of the group go in pairs (A, B), each head a 128-query tile (M = 128),
// and each pair takes two passes over the row's key blocks 0..I, 128 at a time:
//   pass 0: S = Q Kmean^T -> row max
//   pass 1: the same S again -> exp2((s - max) * scale * log2 e), summed down
//           the 128 queries (a transpose-reduce across each warp's 32 rows)
//           into per-warp column sums in shared memory;
// then S' = the sum of all warps' column sums (fixed order) and the row is
// divided by its maximum.  The passes of consecutive pairs overlap: phase k
// (k = 0 .. pairs) runs pass 0 of pair k and pass 1 of pair k - 1 chunk by
// chunk, so the row warps' exponentials of one pair run while the tensor
// cores compute the next pair's maxima, and each chunk of key means is loaded
// once per phase.  Warp 0 issues TMA loads (the two mean terms of a chunk,
// shared by both heads and both passes, in a ring of stages), warp 1 issues
// the MMAs, warpgroup A (warps 4-7) and warpgroup B (warps 8-11) each own one
// head slot of the pairs and its TMEM S buffer, one query row per thread.  A
// row warp pulls a whole chunk of S into registers before it works on it, so
// the buffer is free for the next MMA at once.  Each warpgroup also writes its
// head's query tile into TMEM, where the MMA takes it as the A operand (the
// MMAs read only the mean terms from shared memory); there are two query
// buffers, one per pair in flight, and pair k's queries go in at the start of
// phase k, once pair k - 2 is done.  While shared memory has room (rows of up
// to 1072 blocks), warp 0 also stages each head slot's next query tile there
// by TMA during the phase before, so a row thread reads its row from shared
// memory (one row per thread straight from global memory touches 32 lines per
// load instruction); longer rows read their queries from global memory,
// prefetched into L2 one phase ahead.
#include <type_traits>

#include "common.cuh"
#include "launch.cuh"
#include "sm100.cuh"

namespace fp {

using namespace sm100;

namespace {

constexpr int kScThreads = 384;

// Layout of one build of the kernel for a chunk of kChunk key blocks (MMA N;
// also the span of one scale of the key means).
template <int C, bool kQs = false>
struct ScoreCfg {
    static constexpr int kChunk = C;
    static constexpr int kTerms = 2;                           // fp16 terms of the key means
    static constexpr int kBufs = C == 64 ? 2 : 1;              // TMEM S buffers per head slot
    static constexpr int kTermBytes = C * kHeadDim * 2;        // one term of one chunk
    static constexpr int kStageBytes = kTerms * kTermBytes;
    static constexpr int kStages = C == 64 ? 3 : 2;
    static constexpr int kTmemBufs = 2 * kBufs;
    static constexpr int kSmStage = 0;
    // kQs: the query tiles of the two head slots staged in shared memory by
    // TMA (128 rows x 128 B per box, 128-byte swizzle; bf16 two boxes per tile)
    static constexpr int kQTileBytes = 128 * kHeadDim * 2;
    static constexpr int kSmQs = kSmStage + kStages * kStageBytes;
    static constexpr int kSmCtl = kSmQs + (kQs ? 2 * kQTileBytes : 0);
    static constexpr int kSmAcc = kSmCtl + 512;                // column sums [8 or 2][max_nkb]
    // TMEM: the S buffers (kBufs per head slot), then the query tiles as MMA
    // A operands (128 rows x 128 fp16 = 64 columns each), two buffers of two
    // head slots, so the next pair's queries go in while this pair runs
    static constexpr int kTmemQ = kTmemBufs * C;
    // barriers: Q full/empty per (buffer, head slot), stage full/empty, TMEM
    // full/empty per (head slot, S buffer)
    static constexpr int B_QF = 0, B_QE = 4, B_SF = 8, B_SE = 8 + kStages, B_TF = 8 + 2 * kStages;
    static constexpr int B_TE = B_TF + 4, B_DR = B_TE + 4;                  // B_DR: the MMAs' drain
    // kQs: query tile landed / read, per head slot
    static constexpr int B_QL = B_DR + 1, B_QR = B_QL + 2, B_N = B_QR + 2;
    static_assert(kTmemQ + 256 <= 512, "TMEM budget");
    static_assert(B_N * 8 + 128 <= 512, "control block");
    // shared: one column-sum array per head slot instead of one per row warp
    static size_t smem_bytes(int max_nkb, bool shared = false) {
        return (size_t)kSmAcc + (shared ? 2 : 8) * sizeof(float) * max_nkb + 1024;
    }
};

struct ScoreTcArgs {
    float *score;
    float scale_log2;
    const int8_t *kexp;       // e of each (chunk, kv head): at [chunk's first block][h]
    const uint8_t *q8;        // e4m3 queries (codes); strides in elements
    const __nv_bfloat16 *q16; // bf16 queries
    long long q_stride_tok, q_stride_head;
    const float *q_scale;     // e4m3 only: per query head
    int rows_pad;             // rows of each mean term in the term array
    int acc_stride;           // floats per warp accumulator (>= the row length)
    // fused selection (null: scores only): each row's kept blocks, ascending,
    // into keep_pad at the row's score-map offset, and their count
    int *keep_pad;
    int *counts;
    float alpha;
    int sink_blocks;
    int local_blocks;
    int head_union;           // FP_SCORE_HEAD_UNION: each head normalised alone, max over heads
    int *status;
    unsigned long long wait_ns;
};

// A barrier among the eight row warps that cannot hang: each warp's lane 0
// adds one arrival to a shared counter and spins (bounded, like the mbarrier
// waits) until all eight warps of this generation have arrived.  Returns false
// if the CTA is aborting.
__device__ __forceinline__ bool rows_sync(unsigned *ctr, unsigned &gen, int lane, uint32_t abort_flag,
                                          int *status, unsigned long long wait_ns) {
    gen += 8;
    bool ok = true;
    __threadfence_block();          // this lane's shared / global writes before the arrival
    __syncwarp();
    if (lane == 0) {
        atomicAdd(ctr, 1u);
        volatile unsigned *vc = ctr;
        const uint64_t t0 = global_ns();
        for (uint32_t it = 0; *vc < gen; ++it) {
            if ((it & 63u) == 63u) {
                if (ld_shared_volatile(abort_flag)) { ok = false; break; }
                if (global_ns() - t0 > wait_ns) {
                    set_status(status, FP_ERR_TIMEOUT);
                    st_shared_volatile(abort_flag, 1);
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

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}


// Column sums of a 32x32 block held one row per lane (v[c] = column c of
// this lane's row): after the butterfly, lane L holds the sum of column L.
// Each stage halves the columns a lane holds: it keeps one half, sends the
// other to its partner and adds what it receives, in pairs (add.rn.f32x2),
// each sum rounded exactly as a scalar add would.
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
    auto stage = [&](auto half_c, int mask) {
        constexpr int h = decltype(half_c)::value;
        const bool up = lane & mask;
#pragma unroll
        for (int k = 0; k < h; k += 2) {
            const float r0 = __shfl_xor_sync(0xffffffffu, up ? v[k] : v[k + h], mask);
            const float r1 = __shfl_xor_sync(0xffffffffu, up ? v[k + 1] : v[k + 1 + h], mask);
            float a0, a1;
            f2_unpack(f2_add(f2_pack(up ? v[k + h] : v[k], up ? v[k + 1 + h] : v[k + 1]), f2_pack(r0, r1)), a0, a1);
            v[k] = a0;
            v[k + 1] = a1;
        }
    };
    stage(std::integral_constant<int, 16>{}, 16);
    stage(std::integral_constant<int, 8>{}, 8);
    stage(std::integral_constant<int, 4>{}, 4);
    stage(std::integral_constant<int, 2>{}, 2);
    const bool up = lane & 1;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

// kFp8: the query tiles are e4m3 codes, converted exactly to fp16 (no row
// scale), and the head's scale joins the exponent.  bf16 queries get a row
// scale.
// kShared: the four warps of a head slot add their column sums into one array
// (shared-memory atomics, so the order of the additions varies from run to
// run) instead of one array each: rows past 3120 blocks (up to 12480) then
// still fit.  Without it every sum is added in a fixed order.
template <bool kFp8, int kCh, bool kShared, bool kQs>
__global__ void __launch_bounds__(kScThreads, 1)
score_tc_kernel(const __grid_constant__ BatchDesc bd, const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ CUtensorMap tmM, const ScoreTcArgs a) {
    using Cfg = ScoreCfg<kCh, kQs>;
    static_assert(!(kQs && kShared), "staged queries only with per-warp column sums");
    static_assert(kCh == 128, "the key means' scales span 128-block chunks");
    constexpr int kChunk = Cfg::kChunk, kTermBytes = Cfg::kTermBytes;
    static_assert(Cfg::kBufs == 1, "one TMEM S buffer per head slot");
    constexpr int kStageBytes = Cfg::kStageBytes, kStages = Cfg::kStages, kSmStage = Cfg::kSmStage;
    constexpr int kSmCtl = Cfg::kSmCtl, kSmAcc = Cfg::kSmAcc, kTmemQ = Cfg::kTmemQ;
    constexpr int B_QF = Cfg::B_QF, B_QE = Cfg::B_QE, B_SF = Cfg::B_SF, B_SE = Cfg::B_SE;
    constexpr int B_TF = Cfg::B_TF, B_TE = Cfg::B_TE, B_DR = Cfg::B_DR, B_N = Cfg::B_N;
    constexpr int B_QL = Cfg::B_QL, B_QR = Cfg::B_QR, kSmQs = Cfg::kSmQs;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned; derived from smem_raw by an offset, and the barriers
    // and the abort flag addressed in the shared window (no generic pointer
    // kept live)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *acc = reinterpret_cast<float *>(smem + kSmAcc);              // [4 warps][acc_stride]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kSmCtl);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kSmCtl + B_N * 8);
    const uint32_t abort_flag = smem_u32(smem) + kSmCtl + B_N * 8 + 4;
    float *red = reinterpret_cast<float *>(smem + kSmCtl + B_N * 8 + 16);   // [8]
    unsigned *sync_ctr = reinterpret_cast<unsigned *>(smem + kSmCtl + B_N * 8 + 48);
    float *red_h = reinterpret_cast<float *>(smem + kSmCtl + B_N * 8 + 64);    // [16]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars_a = smem_u32(bars);
    auto bar = [&](int k) { return bars_a + 8u * (uint32_t)k; };

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
    const long long row_off = score_row_offset(rq, bd.h_kv, il, h);
    float *out = a.score ? a.score + row_off : nullptr;

    const int npairs = (g + 1) / 2;

    if (threadIdx.x == 0) {
        for (int k = 0; k < B_N; ++k)
            mbar_init(bar(k), ((k >= B_TE && k < B_TE + 4) || (k >= B_QF && k < B_QF + 4) || (k >= B_QR && k < B_QR + 2))
                                  ? 128u : 1u);
        st_shared_volatile(abort_flag, 0);
        *sync_ctr = 0u;
        fence_barrier_init();
        fence_proxy_async();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        if (warp == 0 && lane == 0) {
            // ================= TMA producer =================
            // phase k runs pass 0 of pair k and pass 1 of pair k - 1 (k = 0 .. npairs):
            // each chunk of key means is loaded once per phase for both
            tma_prefetch_desc(&tmM);
            // kQs: head slot w's query tile of pair p (128 query rows of head hq)
            int nq[2] = {0, 0};                    // query tiles issued per head slot
            auto load_q = [&](int p, int w) {
                constexpr int kBoxes = kFp8 ? 1 : 2;
                mbar_expect_tx(bar(B_QL + w), kBoxes * 128 * 128);
                for (int hf = 0; hf < kBoxes; ++hf)
                    tma_load_3d(sbase + kSmQs + w * Cfg::kQTileBytes + hf * 128 * 128, &tmQ, bar(B_QL + w), hf * 64,
                                h * g + 2 * p + w, rq.q_off + il * kBlock);
                ++nq[w];
            };
            if constexpr (kQs) {
                tma_prefetch_desc(&tmQ);
                for (int w = 0; w < (g > 1 ? 2 : 1); ++w) load_q(0, w);
            }
            int step = 0;
            for (int k = 0; k <= npairs && !ld_shared_volatile(abort_flag); ++k) {
                for (int c = 0; c < nch; ++c, ++step) {
                    const int s = step % kStages, use = step / kStages;
                    if (step >= kStages && !mbar_wait(bar(B_SE + s), (use - 1) & 1, abort_flag, a.status, a.wait_ns))
                        goto producer_done;
                    mbar_expect_tx(bar(B_SF + s), kStageBytes);
                    const uint32_t dst = sbase + kSmStage + s * kStageBytes;
                    for (int t = 0; t < Cfg::kTerms; ++t)
                        for (int hf = 0; hf < 2; ++hf)
                            tma_load_3d(dst + t * kTermBytes + hf * (kTermBytes / 2), &tmM, bar(B_SF + s), hf * 64, h,
                                        t * a.rows_pad + rq.kb_base + c * kChunk);
                    // kQs: pair k + 1's queries, once the row warps have read pair k's
                    // (early in phase k; the chunks armed so far keep the MMAs busy)
                    if (kQs && c == (nch > 1 ? 1 : 0) && k + 1 < npairs)
                        for (int w = 0; w < ((2 * k + 3 < g) ? 2 : 1); ++w) {
                            if (!mbar_wait(bar(B_QR + w), k & 1, abort_flag, a.status, a.wait_ns)) goto producer_done;
                            load_q(k + 1, w);
                        }
                }
            }
        producer_done:
            // after an abort, the copies of the last stages armed land before the
            // CTA leaves (otherwise the MMAs have consumed every stage already)
            if (ld_shared_volatile(abort_flag)) {
                for (int j = step > kStages ? step - kStages : 0; j < step; ++j)
                    mbar_wait_drain(bar(B_SF + j % kStages), (j / kStages) & 1);
                // each slot's last query tile (every earlier one was read)
                for (int w = 0; w < 2; ++w)
                    if (nq[w] > 0) mbar_wait_drain(bar(B_QL + w), (nq[w] - 1) & 1);
            }
        } else if (warp == 1 && lane == 0) {
            // ================= MMA issuer =================
            // per chunk of phase k: S of pass 1 of pair k - 1 for each head slot,
            // then S of pass 0 of pair k, each slot's S into its own TMEM buffer
            constexpr uint32_t idS = idesc_f16(128, kChunk, false);
            int step = 0;
            int uses[2] = {0, 0};                  // S productions per head slot
            auto issue = [&](int w, int qb, uint64_t kd) -> bool {
                const int u = uses[w]++;
                if (u >= 1 && !mbar_wait(bar(B_TE + w), (u - 1) & 1, abort_flag, a.status, a.wait_ns)) return false;
                tc_fence_after();
                // descriptors differ only in the start address: add offsets (in 16-byte units)
                const uint32_t dt = tmem + w * kChunk;
                const uint32_t qt = tmem + kTmemQ + (2 * qb + w) * 64;   // A: 16 d-values per 8 columns
#pragma unroll
                for (int t = 0; t < Cfg::kTerms; ++t)
#pragma unroll
                    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                        const uint32_t boff = t * kTermBytes + (kk >> 2) * (kTermBytes / 2) + (kk & 3) * 32;
                        mma_ts(dt, qt + kk * 8, kd + (boff >> 4), idS, (t | kk) != 0);
                    }
                tc_commit(bar(B_TF + w));
                return true;
            };
            for (int k = 0; k <= npairs; ++k) {
                const int n1 = k >= 1 ? ((2 * k - 1 < g) ? 2 : 1) : 0;     // head slots of pair k - 1
                const int n0 = k < npairs ? ((2 * k + 1 < g) ? 2 : 1) : 0;  // head slots of pair k
                for (int c = 0; c < nch; ++c, ++step) {
                    const int s = step % kStages;
                    if (!mbar_wait(bar(B_SF + s), (step / kStages) & 1, abort_flag, a.status, a.wait_ns)) goto mma_done;
                    const uint64_t kd = smem_desc_sw128(sbase + kSmStage + s * kStageBytes, 16, 1024);
                    for (int w = 0; w < n1; ++w)
                        if (!issue(w, (k - 1) & 1, kd)) goto mma_done;
                    if (c == nch - 1)                  // pair k - 1 is done with its query buffer
                        for (int w = 0; w < n1; ++w) tc_commit(bar(B_QE + 2 * ((k - 1) & 1) + w));
                    for (int w = 0; w < n0; ++w) {
                        if (c == 0 && !mbar_wait(bar(B_QF + 2 * (k & 1) + w), (k >> 1) & 1, abort_flag, a.status, a.wait_ns))
                            goto mma_done;
                        if (!issue(w, k & 1, kd)) goto mma_done;
                    }
                    tc_commit(bar(B_SE + s));
                }
            }
        mma_done:
            if (ld_shared_volatile(abort_flag)) {   // after an abort, every MMA issued is done
                tc_commit(bar(B_DR));               // before the CTA leaves
                mbar_wait_drain(bar(B_DR), 0);
            }
        }
    } else {
        // ================= row warpgroups: one head each, one query row per thread =================
        const int w = (warp - 4) / 4;                     // head slot of the pair
        const int quarter = warp % 4;
        const int rowt = quarter * 32 + lane;
        const bool row_valid = il * kBlock + rowt < rq.lq;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        // this warp's 32 rows, summed (kShared: the head slot's 128 rows)
        float *my_acc = acc + (kShared ? w : w * 4 + quarter) * a.acc_stride;
        unsigned gen = 0;
        bool ok = true;
        if constexpr (kShared) {
            for (int J = quarter * 32 + lane; J < ncol; J += 128) my_acc[J] = 0.f;
            ok = rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns);   // cleared before any add
        } else {
            for (int J = lane; J < ncol; J += 32) my_acc[J] = 0.f;
            __syncwarp();
        }
        int u = 0;
        // head hq's query rows -> query buffer qb in TMEM as the MMA's A operand,
        // in fp16: e4m3 codes exactly as they are; bf16 rows scaled by 2^f_out
        // (exact: 8 significant bits within fp16's range).  Returns false if
        // the CTA is aborting.
        auto put_queries = [&](int pr_q, int &f_out) -> bool {
            const int qb = pr_q & 1;
            if (pr_q >= 2) {                       // the buffer's previous pair is done with it
                const bool got = mbar_wait(bar(B_QE + 2 * qb + w), ((pr_q >> 1) & 1) ^ 1, abort_flag, a.status,
                                           a.wait_ns);
                if (!__all_sync(0xffffffffu, got)) return false;
            }
            const int hq = h * g + 2 * pr_q + w;
            const long long el = (long long)(rq.q_off + il * kBlock + rowt) * a.q_stride_tok + (long long)hq * a.q_stride_head;
            const uint32_t qdst = lane_base + kTmemQ + (2 * qb + w) * 64;
            // kQs: this row of the staged tile, 16-byte piece j of each 128-byte
            // box row at j ^ (row & 7) (128-byte swizzle)
            const uint32_t qrow = sbase + kSmQs + w * Cfg::kQTileBytes + rowt * 128;
            if constexpr (kQs) {
                const bool got = mbar_wait(bar(B_QL + w), pr_q & 1, abort_flag, a.status, a.wait_ns);
                if (!__all_sync(0xffffffffu, got)) return false;
            }
            if constexpr (!kFp8) {
                uint32_t qw[64];
                const uint4 *src = reinterpret_cast<const uint4 *>(a.q16 + el);
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    uint4 c;
                    if constexpr (kQs) c = ld_shared_v4(qrow + (v >> 3) * 128 * 128 + (((v & 7) ^ (rowt & 7)) << 4));
                    else c = row_valid ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
                    if (kQs && !row_valid) c = make_uint4(0, 0, 0, 0);
                    qw[4 * v] = c.x; qw[4 * v + 1] = c.y; qw[4 * v + 2] = c.z; qw[4 * v + 3] = c.w;
                }
                // the row's largest magnitude: bf16 bit patterns without the sign
                // order like their values
                uint32_t mx2 = 0u;
#pragma unroll
                for (int k = 0; k < 64; ++k) mx2 = __vmaxu2(mx2, qw[k] & 0x7fff7fffu);
                if constexpr (kQs) mbar_arrive(bar(B_QR + w));   // read: the tile may be reloaded
                const uint32_t mx16 = (mx2 >> 16) > (mx2 & 0xffffu) ? (mx2 >> 16) : (mx2 & 0xffffu);
                const int f = fp16_scale_exp(mx16 << 16);
                const float sf = pow2f(f);
#pragma unroll
                for (int k = 0; k < 64; ++k) {
                    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qw[k]));
                    qw[k] = pack_f16x2(x.x * sf, x.y * sf);
                }
                tmem_st32(qdst, *reinterpret_cast<const uint32_t(*)[32]>(qw));
                tmem_st32(qdst + 32, *reinterpret_cast<const uint32_t(*)[32]>(qw + 32));
                f_out = f;
            } else {
                uint4 cq[8];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    if constexpr (kQs) cq[v] = row_valid ? ld_shared_v4(qrow + ((v ^ (rowt & 7)) << 4)) : make_uint4(0, 0, 0, 0);
                    else cq[v] = row_valid ? __ldg(reinterpret_cast<const uint4 *>(a.q8 + el) + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qw[32];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 c = cq[half * 4 + v];
                        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const __nv_fp8x2_storage_t c2v = (__nv_fp8x2_storage_t)(cw[k / 2] >> (16 * (k & 1)));
                            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(c2v, __NV_E4M3);
                            qw[8 * v + k] = (uint32_t)hr.x | ((uint32_t)hr.y << 16);
                        }
                    }
                    tmem_st32(qdst + half * 32, qw);
                }
                if constexpr (kQs) mbar_arrive(bar(B_QR + w));   // read: the tile may be reloaded
                f_out = 0;
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(B_QF + 2 * qb + w));
            return true;
        };
        // the next pair's query row into L2 ahead of its load (bf16: two 128-byte lines)
        auto prefetch_queries = [&](int pr_q) {
            if (!row_valid) return;
            const int hq = h * g + 2 * pr_q + w;
            const long long el = (long long)(rq.q_off + il * kBlock + rowt) * a.q_stride_tok + (long long)hq * a.q_stride_head;
            const size_t p = __cvta_generic_to_global(kFp8 ? static_cast<const void *>(a.q8 + el)
                                                           : static_cast<const void *>(a.q16 + el));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
            if constexpr (!kFp8) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + 128));
        };
        // phase k: this slot's head of pair k (pass 0: the row max) and of pair
        // k - 1 (pass 1: the exponentials), chunk by chunk in the MMA's order
        int fq = 0, fq_prev = 0;                          // row scale exponents (pair k, pair k - 1)
        float m_prev = -INFINITY;                         // pair k - 1's row max (unscaled logits)
        for (int k = 0; k <= npairs && ok; ++k) {
            const bool has0 = k < npairs && 2 * k + w < g;
            const bool has1 = k >= 1 && 2 * (k - 1) + w < g;
            // a slot with no head left (odd g) stops; under the union of heads it
            // still takes part in the pairs' syncs
            if (!has0 && !has1 && !a.head_union) break;
            if (has0) {
                if (!kQs && 2 * (k + 1) + w < g) prefetch_queries(k + 1);
                if (!put_queries(k, fq)) { ok = false; break; }
            }
            float c2q1 = 0.f, mc2 = 0.f;                // pass 1 of pair k - 1
            if (has1) {
                const float c2 = kFp8 ? a.scale_log2 * __ldg(a.q_scale + h * g + 2 * (k - 1) + w) : a.scale_log2;
                c2q1 = c2 * pow2f(-fq_prev);            // undoes the row's query scale
                mc2 = !row_valid ? INFINITY : (m_prev == -INFINITY ? 0.f : m_prev * c2);
            }
            const float fq0 = pow2f(-fq);
            float m = -INFINITY;                        // pair k's row max
            for (int c = 0; c < nch && (has0 || has1); ++c) {
                // the scale exponent of this chunk's key means (read before the wait)
                const float fk = pow2f(-(int)__ldg(a.kexp + (long long)(rq.kb_base + c * kChunk) * bd.h_kv + h));
                // the next S of this slot, whole into registers; the buffer is then
                // free for the next MMA while this warp works on the values
                uint32_t sv[kChunk / 32][32];
                auto pull = [&]() -> bool {
                    const bool got = mbar_wait(bar(B_TF + w), u & 1, abort_flag, a.status, a.wait_ns);
                    if (!__all_sync(0xffffffffu, got)) return false;
                    ++u;
                    tc_fence_after();
                    const uint32_t colb = lane_base + w * kChunk;
#pragma unroll
                    for (int sl = 0; sl < kChunk / 32; ++sl) tmem_ld32(colb + sl * 32, sv[sl]);
                    tmem_ld_wait();
#pragma unroll
                    for (int sl = 0; sl < kChunk / 32; ++sl) reg_fence(sv[sl]);
                    tc_fence_before();
                    mbar_arrive(bar(B_TE + w));
                    return true;
                };
                if (has1) {
                    if (!pull()) { ok = false; break; }
                    // exponents as paired FMAs: (s0, s1) * c2 * 2^-(f+e) - mc2, the
                    // scaled logits times an exact power-of-two correction of the
                    // constant (an invalid row has mc2 = +inf, so its terms are
                    // exactly 0); columns past the row are masked only in its
                    // last, partial chunk
                    const float c2c = c2q1 * fk;
                    const uint64_t cc = f2_pack(c2c, c2c), nm = f2_pack(-mc2, -mc2);
#pragma unroll
                    for (int sl = 0; sl < kChunk / 32; ++sl) {
                        const int J0 = c * kChunk + sl * 32;
                        float v0[32];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float z0, z1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[sl][e]), __uint_as_float(sv[sl][e + 1])), cc, nm),
                                      z0, z1);
                            v0[e] = fast_exp2(z0);
                            v0[e + 1] = fast_exp2(z1);
                        }
                        if (J0 + 32 > ncol) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (J0 + e >= ncol) v0[e] = 0.f;
                        }
                        // lane L now gets the sum of column J0 + L over this warp's 32 rows
                        const float s0 = transpose_reduce32(v0, lane);
                        if (J0 + lane < ncol) {
                            if constexpr (kShared) atomicAdd(my_acc + J0 + lane, s0);
                            else my_acc[J0 + lane] += s0;
                        }
                    }
                }
                if (has0) {
                    if (!pull()) { ok = false; break; }
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int sl = 0; sl < kChunk / 32; ++sl) {
                        const int J0 = c * kChunk + sl * 32;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (J0 + e < ncol) m4[e & 3] = fmaxf(m4[e & 3], __uint_as_float(sv[sl][e]));
                    }
                    // the chunk's largest scaled logit, unscaled exactly (powers of two)
                    m = fmaxf(m, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * fq0 * fk);
                }
            }
            if (!ok) break;
            m_prev = m;
            fq_prev = fq;
            if (a.head_union && k >= 1) {
                // union of heads: pair k - 1's two heads are complete in the
                // accumulators (four warps each).  Each head's row is normalised by
                // its own maximum and folded into the output row by maximum; the
                // accumulators are cleared for the next pair.
                const int pr = k - 1;
                const int t = threadIdx.x - 128;
                const int st = a.acc_stride;
                auto head_sum = [&](int ww, int J) {
                    if constexpr (kShared) return acc[ww * st + J];
                    const float *b0 = acc + ww * 4 * st;
                    return (b0[J] + b0[st + J]) + (b0[2 * st + J] + b0[3 * st + J]);
                };
                const bool h1 = 2 * pr + 1 < g;
                ok = rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns);
                if (!ok) break;
                float m0 = 0.f, m1 = 0.f;
                for (int J = t; J < ncol; J += 256) {
                    m0 = fmaxf(m0, head_sum(0, J));
                    if (h1) m1 = fmaxf(m1, head_sum(1, J));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
                    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
                }
                if (lane == 0) {
                    red_h[warp - 4] = m0;
                    red_h[8 + warp - 4] = m1;
                }
                ok = rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns);
                if (!ok) break;
                float M0 = 0.f, M1 = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    M0 = fmaxf(M0, red_h[q]);
                    M1 = fmaxf(M1, red_h[8 + q]);
                }
                const float i0 = 1.f / M0, i1 = h1 ? 1.f / M1 : 0.f;
                for (int J = t; J < ncol; J += 256) {
                    const float v0 = head_sum(0, J);
                    float uu = v0 == M0 ? 1.f : v0 * i0;
                    if (h1) {
                        const float v1 = head_sum(1, J);
                        uu = fmaxf(uu, v1 == M1 ? 1.f : v1 * i1);
                    }
                    if (pr > 0) uu = fmaxf(uu, out[J]);
                    out[J] = uu;
#pragma unroll
                    for (int q = 0; q < (kShared ? 2 : 8); ++q) acc[q * st + J] = 0.f;
                }
                ok = rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns);
                if (!ok) break;
            }
        }
        // S' = the eight warps' sums (fixed order); re-normalise by its maximum
        // (the union of heads has written its row pair by pair)
        if (ok && !a.head_union) ok = rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns);
        if (ok && !a.head_union) {
            const int t = threadIdx.x - 128;
            const int st = a.acc_stride;
            auto colsum = [&](int J) {
                if constexpr (kShared) return acc[J] + acc[st + J];
                return ((acc[J] + acc[st + J]) + (acc[2 * st + J] + acc[3 * st + J])) +
                       ((acc[4 * st + J] + acc[5 * st + J]) + (acc[6 * st + J] + acc[7 * st + J]));
            };
            float mx = 0.f;
            for (int J = t; J < ncol; J += 256) mx = fmaxf(mx, colsum(J));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) red[warp - 4] = mx;
            const bool ok2 = rows_sync(sync_ctr, gen, lane, abort_flag, a.status, a.wait_ns);
            mx = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) mx = fmaxf(mx, red[k]);
            const float inv = 1.f / mx;
            auto score_of = [&](int J) {
                const float v = colsum(J);
                return v == mx ? 1.f : v * inv;
            };
            if (ok2 && !a.keep_pad) {
                for (int J = t; J < ncol; J += 256) out[J] = score_of(J);
            } else if (ok2) {
                // fused selection [V1 summary 3.2-3.3]: the row's maximum is exactly 1,
                // so a block is kept when its score >= alpha, or it is a sink or local
                // block.  Row warp w takes segment w of the row (score_segment()),
                // writes its kept blocks, ascending, from the segment's start, and
                // records their count: no further sync, the gather joins the segments.
                const int wr = warp - 4;
                const int seg = score_segment(ncol);
                const int j0 = wr * seg, j1 = min(ncol, j0 + seg);
                int *dst = a.keep_pad + row_off + j0;
                int pos = 0;
                for (int J0 = j0; J0 < j1; J0 += 32) {
                    const int J = J0 + lane;
                    const float sc = J < j1 ? score_of(J) : 0.f;
                    const bool k = J < j1 && (sc >= a.alpha || J < a.sink_blocks || J >= I - a.local_blocks + 1);
                    if (J < j1 && out) out[J] = sc;
                    const unsigned m = __ballot_sync(0xffffffffu, k);
                    if (k) dst[pos + __popc(m & ((1u << lane) - 1u))] = J;
                    pos += __popc(m);
                }
                if (lane == 0) a.counts[row * 8 + wr] = pos;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// fp32 block means -> the score kernel's operands.  One CTA per chunk of 128
// blocks of a request (from its first block) and kv head: the chunk's largest
// magnitude sets the power of two 2^e (fp16_scale_exp), and
//   kmean * 2^e = hi + lo,  hi = fp16(kmean * 2^e),  lo = fp16(kmean * 2^e - hi)
// (the difference is exact in fp32; together 22 significant bits).  e goes to
// kexp at [the chunk's first block][h].  Term t of block row k, head h, starts
// at terms + t * n_pad + (k * h_kv + h) * d; rows past the last request's
// blocks (up to rows_pad) are zero.
constexpr int kSplitThreads = 1024;
__global__ void __launch_bounds__(kSplitThreads)
split_means_kernel(const __grid_constant__ BatchDesc bd, const float *__restrict__ km, __half *__restrict__ terms,
                   int8_t *__restrict__ kexp, long long n_pad, int rows_pad) {
    int b = blockIdx.x, r = 0;
    for (; r < bd.batch; ++r) {
        const int nc = (bd.req[r].nkb + 127) / 128;
        if (b < nc) break;
        b -= nc;
    }
    if (r == bd.batch) return;
    const ReqDesc &rq = bd.req[r];
    const int h = blockIdx.y;
    const int row0 = rq.kb_base + b * 128;
    const int nrow = min(128, rq.nkb - b * 128);
    const int col = (threadIdx.x % 32) * 4;          // four dims
    const int rw = threadIdx.x / 32;                 // rows rw, rw + 32, ...
    float4 v[4];
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int rr = rw + 32 * k;
        v[k] = rr < nrow ? __ldg(reinterpret_cast<const float4 *>(km + ((long long)(row0 + rr) * bd.h_kv + h) * kHeadDim + col))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
    }
    __shared__ float red[kSplitThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int k = 1; k < kSplitThreads / 32; ++k) mx = fmaxf(mx, red[k]);
    const int e = fp16_scale_exp(__float_as_uint(mx));
    const float sf = pow2f(e);
    const bool last = r == bd.batch - 1;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int rr = rw + 32 * k;
        if (rr >= nrow && !(last && row0 + rr < rows_pad)) continue;
        const float x[4] = {v[k].x * sf, v[k].y * sf, v[k].z * sf, v[k].w * sf};
        uint32_t hw[2], lw[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const __half2 hi = __floats2half2_rn(x[2 * q], x[2 * q + 1]);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(x[2 * q] - hf.x, x[2 * q + 1] - hf.y);
            hw[q] = *reinterpret_cast<const uint32_t *>(&hi);
            lw[q] = *reinterpret_cast<const uint32_t *>(&lo);
        }
        const long long o = ((long long)(row0 + rr) * bd.h_kv + h) * kHeadDim + col;
        *reinterpret_cast<uint2 *>(terms + o) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2 *>(terms + n_pad + o) = make_uint2(lw[0], lw[1]);
    }
    if (threadIdx.x == 0) kexp[(long long)row0 * bd.h_kv + h] = (int8_t)e;
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
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// the queries [tokens][h_q][d] (bf16 or e4m3 codes) as 128-row boxes of one
// head and 128 bytes of d, 128-byte swizzle
bool map_queries(CUtensorMap *m, const void *base, int h_q, long long total_q, long long s_head, long long s_tok,
                 bool fp8) {
    EncodeTiledFn fn = encode_fn_sc();
    if (!fn) return false;
    const int esz = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)h_q, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {(cuuint64_t)(s_head * esz), (cuuint64_t)(s_tok * esz)};
    cuuint32_t box[3] = {(cuuint32_t)(128 / esz), 1, 128};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// rows of each mean term: at least one box of the widest chunk
int score_tc_rows_pad(const BatchDesc &bd) { return bd.total_kb > 128 ? bd.total_kb : 128; }

// the build that serves rows of up to max_nkb blocks: 128-block chunks, with a
// column-sum array per row warp (fixed summation order) while it fits, then
// one per head slot
static bool score_tc_shared(int max_nkb) { return ScoreCfg<128>::smem_bytes(max_nkb) > 227 * 1024; }
// query tiles staged by TMA while shared memory has room for them (rows of up
// to 1072 blocks)
static bool score_tc_staged(int max_nkb) { return ScoreCfg<128, true>::smem_bytes(max_nkb) <= 227 * 1024; }
size_t score_tc_smem_bytes(int max_nkb) {
    if (score_tc_staged(max_nkb)) return ScoreCfg<128, true>::smem_bytes(max_nkb);
    return ScoreCfg<128>::smem_bytes(max_nkb, score_tc_shared(max_nkb));
}

cudaError_t launch_score_tc(const BatchDesc &bd, bool fp8, const void *q, long long q_stride_tok,
                            long long q_stride_head, const float *q_scale, const float *k_mean, float softmax_scale,
                            float *score, void *terms_ws, int *status, unsigned long long wait_ns,
                            cudaStream_t st, const ScoreSelect *sel, bool head_union) {
    const int rows_pad = score_tc_rows_pad(bd);
    const long long n_pad = (long long)rows_pad * bd.h_kv * kHeadDim;
    __half *terms = static_cast<__half *>(terms_ws);
    int8_t *kexp = static_cast<int8_t *>(terms_ws) + score_tc_kexp_offset(bd);
    int chunks = 0;
    for (int r = 0; r < bd.batch; ++r) chunks += (bd.req[r].nkb + 127) / 128;
    if (chunks > 0) split_means_kernel<<<dim3(chunks, bd.h_kv), kSplitThreads, 0, st>>>(bd, k_mean, terms, kexp, n_pad, rows_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap tmQ, tmM;
    const bool shared = score_tc_shared(bd.max_nkb);
    const bool staged = score_tc_staged(bd.max_nkb);
    if (!map3(&tmM, terms, bd.h_kv, (long long)ScoreCfg<128>::kTerms * rows_pad, kHeadDim,
              (long long)bd.h_kv * kHeadDim, 128))
        return cudaErrorInvalidValue;
    ScoreTcArgs a;
    a.score = score;
    a.kexp = kexp;
    a.q8 = (const uint8_t *)q;
    a.q16 = (const __nv_bfloat16 *)q;
    a.q_stride_tok = q_stride_tok;
    a.q_stride_head = q_stride_head;
    a.q_scale = q_scale;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.rows_pad = rows_pad;
    a.acc_stride = bd.max_nkb;
    a.keep_pad = sel ? sel->keep_pad : nullptr;
    a.counts = sel ? sel->counts : nullptr;
    a.alpha = sel ? sel->alpha : 0.f;
    a.sink_blocks = sel ? sel->sink_blocks : 0;
    a.local_blocks = sel ? sel->local_blocks : 0;
    a.head_union = head_union ? 1 : 0;
    a.status = status;
    a.wait_ns = wait_ns;
    if (staged) {
        if (!map_queries(&tmQ, q, bd.h_q, bd.total_q, q_stride_head, q_stride_tok, fp8)) return cudaErrorInvalidValue;
    } else {
        tmQ = tmM;                       // not read: the row warps load the queries themselves
    }
    const int smem = (int)score_tc_smem_bytes(bd.max_nkb);
    auto kern = staged   ? (fp8 ? score_tc_kernel<true, 128, false, true> : score_tc_kernel<false, 128, false, true>)
                : shared ? (fp8 ? score_tc_kernel<true, 128, true, false> : score_tc_kernel<false, 128, true, false>)
                         : (fp8 ? score_tc_kernel<true, 128, false, false> : score_tc_kernel<false, 128, false, false>);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<bd.total_rows, kScThreads, smem, st>>>(bd, tmQ, tmM, a);
    return cudaGetLastError();
}

}  // namespace fp
