// Block-sparse causal attention with block-mean correction on tcgen05 (sm_103a).
//
// What it computes: the sparse attention of the FlashPrefill V2 paper reading,
// section 4.1 -- kept key blocks exactly, every skipped earlier block J < I as
// one mean token (kmean_J, vmean_J) of weight n_J (the V2 popular article,
// mean-correction section: the block's token count) -- over a
// paged KV cache (V2 section 4.3: the address of a key is the page-table entry
// of its page plus its offset in the page, fetched asynchronously), with the
// g query heads of a kv group packed so that each kept KV tile is fetched once
// for the group (PackGQA, V2 section 4.2 (1)).
//
// How (sm_103a design, not the Hopper one of the pages):
//  * a work unit = (index row (request, query block I, kv head h), a pair of
//    query heads of the group): two 128-query tiles Q0, Q1;
//  * persistent CTAs, one per SM, take units off a list grouped by (request,
//    kv head) for L2 reuse, longest rows first; warp 2 prepares the next
//    unit's metadata (kept-block bitmap, mean tiles) while the current one
//    runs;
//  * warp 0 issues TMA loads (Q once; K and V tiles through the page table
//    into a two-stage ring each; mean tiles from the bf16 copies of the block
//    means);
//  * warp 1 issues tcgen05 MMAs: S_t = Q_t K^T into TMEM, then O_t += P_t V
//    with P_t read from TMEM (it overwrites S_t as packed bf16);
//  * warps 4-7 / 8-11 are the softmax warpgroups of tile 0 / tile 1: they read
//    S from TMEM, apply the causal mask or the mean-token bias log2(n_J),
//    keep the running max (rescaling O in TMEM only when the max grows by
//    more than 2^8) and write P back to TMEM;
//  * the MMA issue order S0(j) S1(j) PV0(j) S0(j+1) PV1(j) S1(j+1) ... lets
//    one tile's softmax overlap the other tile's MMAs (the pingpong of V2
//    section 4.2 (3), with TMEM accumulators instead of registers);
//  * item list of a unit: the kept blocks (CSR row, ascending), then the
//    tiles of block means that contain at least one skipped block; the dense
//    path walks J = 0..I with no mean tiles;
//  * a mean token's logit goes into the exponent, where one bf16 term of the
//    key means would move it by up to 2^-9 * scale * sum_c |q_c kmean_c| (e4m3:
//    2^-4).  A mean tile covers 128 blocks.  e4m3 takes the key means as two
//    terms, hi + lo, both 16 KB tiles in its K slot (4 more MMAs).  bf16 takes
//    them as one fp16 term (2^-12) scaled by a power of two per tile and kv
//    head, against queries converted in place to fp16 once the unit's kept
//    blocks are done with them (exact, under a power-of-two scale per row);
//    the exponent's constant undoes both scales.
// Every mbarrier wait is bounded (status FP_ERR_TIMEOUT instead of a hang).
#include <stdio.h>
#include <stdlib.h>

#include <type_traits>

#include "common.cuh"
#include "sm100.cuh"
#include "launch.cuh"

namespace fp {

using namespace sm100;

constexpr int kAttnThreads = 384;     // 3 warpgroups: control (TMA, MMA, unit metadata), softmax tile 0, tile 1
// register split (setmaxnreg): the launch grants 168 per thread; the control
// warpgroup gives some back so the softmax warpgroups can hold a whole
// 128-column row of S: 104*128 + 2*192*128 <= 168*384.
constexpr int kRegsControl = 104;
constexpr int kRegsSoftmax = 192;
static_assert(kRegsControl * 128 + 2 * kRegsSoftmax * 128 <= 168 * kAttnThreads, "register split");
constexpr int kTileBytes = kBlock * kHeadDim * 2;          // 32 KB: one 128 x 128 bf16 tile
constexpr int kHalfBytes = kTileBytes / 2;                 // 64 columns of d
constexpr int kSmemQ = 0;
constexpr int kSmemK = 2 * kTileBytes;
constexpr int kSmemV = 4 * kTileBytes;
constexpr int kSmemCtl = 6 * kTileBytes;                   // 192 KB
constexpr int kBitmapWords = FP_MAX_KEY_BLOCKS / 32;
constexpr int kMaxCorrTiles = FP_MAX_KEY_BLOCKS / kBlock;   // mean tiles span 128 blocks

// BAR_DR: the MMA thread's drain before the CTA leaves
// A bf16 unit whose first term is a mean tile: its queries land on BAR_QL,
// the softmax threads convert their rows to fp16 and arrive on BAR_QC, and one
// of them then completes BAR_Q for the MMA thread
enum { BAR_Q = 0, BAR_QE = 1, BAR_KF = 2, BAR_KE = 4, BAR_VF = 6, BAR_VE = 8, BAR_SF = 10, BAR_PF = 12,
       BAR_OF = 14, BAR_MF = 16, BAR_ME = 18, BAR_DR = 20, BAR_QL = 21, BAR_QC = 22, NUM_BARS = 23 };
// arrivals on a metadata-empty barrier: the TMA thread, the MMA thread and
// one lane of each of the eight softmax warps
constexpr int kMetaConsumers = 10;

// What the metadata warp prepares for one unit, double-buffered so that it
// runs one unit ahead of the others.
struct UnitMeta {
    int pos;                          // position in the work list; -1: no more units
    int unit;                         // unit id
    int n_items;                      // terms of this unit's part (kept blocks, then mean tiles)
    int n_corr;                       // mean tiles of the whole row
    int jb;                           // the part's first term in the row's list
    int n_kept;                       // kept blocks of the row (terms before the mean tiles)
    int pad[2];
    int z0[32];                       // first lookup round: pool row of box (term jb + k / nsub, k % nsub)
    uint32_t bitmap[kBitmapWords];    // kept blocks J < I
    int corr[kMaxCorrTiles];          // mean tiles holding a skipped block
};
constexpr int kSmemMisc = kSmemCtl + NUM_BARS * 8;         // TMEM address, abort flag
constexpr int kSmemMeta = kSmemCtl + 256;
constexpr int kSmemAttn = kSmemMeta + 2 * (int)sizeof(UnitMeta) + 1024;
static_assert(NUM_BARS * 8 + 8 <= 256, "control block");
static_assert(sizeof(UnitMeta) % 16 == 0, "metadata buffers");

// Row `row` of a 128 x 128 bf16 query tile in shared memory (two 64-column
// halves, 128-byte rows, swizzled within each row) converted in place to fp16
// under the row's own power-of-two scale 2^f: exact, since bf16 carries 8
// significant bits and the scale puts the row's largest magnitude just under
// fp16's largest value.  Returns 2^-f, which undoes the scale in the exponent.
// The conversion is elementwise, so the swizzle does not matter; a lane starts
// at the chunk its row number picks, so the 32 rows of a warp spread over the
// banks.
__device__ __noinline__ float q_to_f16(uint32_t tile, int row) {
    // two passes over the row (the maximum, then the conversion), so that few
    // registers are live: the control warps run it under a small budget
    auto addr = [&](int c) { return tile + (c >> 3) * kHalfBytes + row * 128 + (((c & 7) + row) & 7) * 16; };
    uint32_t mx2 = 0u;                             // bf16 bit patterns without the sign order like values
#pragma unroll 4
    for (int c = 0; c < 16; ++c) {
        const uint4 w = ld_shared_v4(addr(c));
        mx2 = __vmaxu2(__vmaxu2(mx2, w.x & 0x7fff7fffu),
                       __vmaxu2(w.y & 0x7fff7fffu, __vmaxu2(w.z & 0x7fff7fffu, w.w & 0x7fff7fffu)));
    }
    const uint32_t mx16 = (mx2 >> 16) > (mx2 & 0xffffu) ? (mx2 >> 16) : (mx2 & 0xffffu);
    const int f = fp16_scale_exp(mx16 << 16);
    const float sf = pow2f(f);
    auto cvt = [&](uint32_t x) {
        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x));
        const __half2 h = __floats2half2_rn(v.x * sf, v.y * sf);
        return *reinterpret_cast<const uint32_t *>(&h);
    };
#pragma unroll 4
    for (int c = 0; c < 16; ++c) {
        const uint4 w = ld_shared_v4(addr(c));
        st_shared_v4(addr(c), make_uint4(cvt(w.x), cvt(w.y), cvt(w.z), cvt(w.w)));
    }
    return pow2f(-f);
}

struct AttnArgs {
    const int *row_ptr;       // null in dense mode
    const int *col_idx;
    const int *work;          // unit ids in schedule order
    int *next_unit;           // work-list cursor (zeroed by the schedule kernel)
    int n_units;
    const int *block_table;
    int max_pages;
    int page_size;
    int num_pages;
    int n_pairs;              // query-head pairs per kv head
    int n_split;              // split-KV parts per row (1: none)
    float *part_o;            // n_split > 1: fp32 partial outputs [n_split, total_q, h_q, d]
    float *part_lse;          // n_split > 1: partial LSEs [n_split, h_q, total_q]
    int mean_corr;
    int mean_rows;            // row offset of the lo term of the key means (e4m3)
    const int8_t *kexp;       // bf16: scale exponent of each mean tile's key means, at [tile's first block][h]
    float scale_log2;         // softmax scale * log2(e)
    const float *q_scale;     // e4m3 only: per query head / kv head scales
    const float *k_scale;
    const float *v_scale;
    __nv_bfloat16 *out;
    float *lse;
    int *status;
    unsigned long long wait_ns;
};

// 128 bytes of P (64 packed bf16 pairs) -> bf16x2 word
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// one work unit: index row (request r, query block I, kv head h) and a pair of
// query heads hq0, hq0 + 1 of the group
struct Unit {
    int row, r, il, h, I, hq0, rp0, n_kept, split;
};

// unit id = (row * n_pairs + pair) * n_split + part
__device__ __forceinline__ Unit decode_unit(const BatchDesc &bd, const AttnArgs &a, int unit) {
    Unit U;
    U.split = unit % a.n_split;
    const int rp = unit / a.n_split;
    U.row = rp / a.n_pairs;
    const int pair = rp % a.n_pairs;
    U.r = req_of_row(bd, U.row);
    const ReqDesc &rq = bd.req[U.r];
    const int local = U.row - rq.row_base;
    U.il = local / bd.h_kv;
    U.h = local % bd.h_kv;
    U.I = rq.start / kBlock + U.il;
    U.hq0 = U.h * bd.g + 2 * pair;
    U.rp0 = a.row_ptr ? __ldg(a.row_ptr + U.row) : 0;
    U.n_kept = a.row_ptr ? __ldg(a.row_ptr + U.row + 1) - U.rp0 : U.I + 1;
    return U;
}

// kFp8: q, k, v (and the block-mean tiles) are e4m3 codes with per-head
// scales; both MMAs run as kind::f8f6f4 and P is stored in TMEM as e4m3 of
// 256 * p (the scaling of the V2 paper reading, section 4.2 (4), which keeps
// the weights in e4m3's normal range; it cancels in the ratio).
//
// Persistent: one CTA per SM walks the work list (a shared cursor: each SM
// takes the next unit when it is ready).
// Barrier phases run on counters that span units: `it` counts the CTA's
// items (K/V ring slots, S and P handshakes), `kq` its non-empty units (Q and
// O handshakes), `k` all its units (metadata buffers).  The next unit's Q,
// K and V loads and its first S MMAs overlap the current unit's epilogue.
// kLse (e4m3 only): also keep the sum of the unrounded weights, for an LSE
// that counts the weights e4m3 flushes (wanted when the caller asks for the
// LSE or rows are split; it costs ~10% of the e4m3 kernel)
// kVdm: the value cache is dim-major ([num_pages, h_kv, d, page_size]): a kept
// block's V tile arrives as d rows of keys and is a K-major operand of PV
// kPlo (e4m3 only): P enters PV in two e4m3 terms, hi = e4m3(256 p) and the
// residual lo = e4m3(256 p - hi) in the next 32 TMEM columns, through a second
// PV pass: e4m3's 1/16 relative rounding of the largest weights drops to
// about 1/256
// kMean: the mean-tile code is compiled in (bf16 builds without it serve the
// dense path and launches without the mean correction: less code in the loops).
template <bool kFp8, bool kLse, bool kVdm, bool kPlo = false, bool kMean = true>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_kernel(const __grid_constant__ BatchDesc bd, const __grid_constant__ CUtensorMap tmQ,
            const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
            const __grid_constant__ CUtensorMap tmKm, const __grid_constant__ CUtensorMap tmVm,
            const AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned (128-byte swizzle atoms).  smem, the barriers and the
    // abort flag are derived from smem_raw by offsets (not through an integer
    // round trip of a generic pointer), so every role addresses them in the
    // shared window: no 64-bit pointer stays live, and the kernel spills
    // nothing (with one it reloaded at every wait site, and extra code in the
    // MMA thread put a local load beside each MMA)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kSmemCtl);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kSmemMisc);
    const uint32_t abort_flag = smem_u32(smem) + kSmemMisc + 4;   // shared-window address
    UnitMeta *meta = reinterpret_cast<UnitMeta *>(smem + kSmemMeta);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars_a = smem_u32(bars);
    auto bar = [&](int k) { return bars_a + 8u * (uint32_t)k; };
    // a 128 x 128 tile is 32 KB of bf16 in two 64-column boxes, or 16 KB of
    // e4m3 in one 128-column box; smem slots are 32 KB either way
    constexpr int kT = kFp8 ? kTileBytes / 2 : kTileBytes;
    constexpr int kNH = kFp8 ? 1 : 2;
    constexpr int kMeanSpan = kBlock;                        // blocks per mean tile
    const bool sparse = a.row_ptr != nullptr;

    // ---- set-up (once per CTA) ---------------------------------------------------
    if (threadIdx.x == 0) {
        for (int k = 0; k < NUM_BARS; ++k) {
            uint32_t cnt = 1u;
            if (k == BAR_PF || k == BAR_PF + 1) cnt = 128u;
            if (k == BAR_MF || k == BAR_MF + 1) cnt = 32u;
            if (k == BAR_ME || k == BAR_ME + 1) cnt = kMetaConsumers;
            if (k == BAR_QC) cnt = 256u;
            mbar_init(bar(k), cnt);
        }
        st_shared_volatile(abort_flag, 0);
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
    // a CTA of this launch (or an earlier one on this workspace) timed out:
    // do no work, so a broken launch ends in one wait limit, not one per CTA
    const bool dead = a.status && *reinterpret_cast<volatile int *>(a.status) == FP_ERR_TIMEOUT;

    // each role's code sits under its own register budget
    if (warp < 4) {
        setmaxnreg_dec<kRegsControl>();
        if (dead) {
        } else if (warp == 2) {
            // ================= unit metadata =================
            // takes the next unit off the work list, builds its kept-block
            // bitmap and the list of mean tiles holding a skipped block
            for (int k = 0;; ++k) {
                const int b = k & 1;
                UnitMeta &M = meta[b];
                if (k >= 2) {
                    const bool got = mbar_wait(bar(BAR_ME + b), ((k >> 1) & 1) ^ 1, abort_flag, a.status, a.wait_ns);
                    if (!__all_sync(0xffffffffu, got)) break;
                }
                int pos = 0;
                if (lane == 0) pos = atomicAdd(a.next_unit, 1);
                pos = __shfl_sync(0xffffffffu, pos, 0);
                const bool end = pos >= a.n_units;
                int unit = 0, n_corr = 0, n_kept = 0, split = 0;
                if (!end) {
                    unit = __ldg(a.work + pos);
                    const Unit U = decode_unit(bd, a, unit);
                    n_kept = U.n_kept;
                    split = U.split;
                    // the unit's queries into L2 now, so that their load when the
                    // unit starts (exposed, at a unit switch) hits L2, not DRAM
                    if (lane == 0) {
                        const int q_row0 = bd.req[U.r].q_off + U.il * kBlock;
                        for (int t = 0; t < 2; ++t)
                            for (int hf = 0; hf < kNH; ++hf) tma_prefetch_l2_3d(&tmQ, hf * 64, U.hq0 + t, q_row0);
                    }
                    const int I = U.I;
                    if (sparse && a.mean_corr && I > 0) {
                        const int nw = (I + 31) / 32;
                        for (int w = lane; w < nw; w += 32) M.bitmap[w] = 0u;
                        __syncwarp();
                        for (int j = lane; j < U.n_kept; j += 32) {
                            const int J = __ldg(a.col_idx + U.rp0 + j);
                            if (J >= 0 && J < I) atomicOr(&M.bitmap[J >> 5], 1u << (J & 31));
                        }
                        __syncwarp();
                        const int ntiles = (I + kMeanSpan - 1) / kMeanSpan;
                        for (int c0 = 0; c0 < ntiles; c0 += 32) {
                            const int c = c0 + lane;
                            bool any = false;
                            if (c < ntiles) {
                                for (int w = 0; w < kMeanSpan / 32; ++w) {
                                    const int J0 = c * kMeanSpan + w * 32;
                                    if (J0 >= I) break;
                                    const uint32_t valid = (I - J0 >= 32) ? 0xffffffffu : ((1u << (I - J0)) - 1u);
                                    if (~M.bitmap[J0 >> 5] & valid) any = true;
                                }
                            }
                            const unsigned m = __ballot_sync(0xffffffffu, any);
                            if (any) M.corr[n_corr + __popc(m & ((1u << lane) - 1u))] = c;
                            n_corr += __popc(m);
                        }
                    }
                }
                // this part's share of the row's terms
                const int n_terms = n_kept + n_corr;
                const int jb = (int)((long long)split * n_terms / a.n_split);
                const int je = (int)((long long)(split + 1) * n_terms / a.n_split);
                if (!end) {
                    // the first round of page lookups, ahead of the producer (the
                    // same rule as its own rounds: one box per lane)
                    const Unit U = decode_unit(bd, a, unit);
                    const ReqDesc &rq = bd.req[U.r];
                    const int rpb = a.page_size < kBlock ? a.page_size : kBlock;
                    const int nsub = kBlock / rpb;
                    const int jj = jb + lane / nsub;
                    int z = a.num_pages * a.page_size;                 // zero-filled rows
                    if (jj < n_kept) {
                        const int J = sparse ? __ldg(a.col_idx + U.rp0 + jj) : jj;
                        const int tok = J * kBlock + (lane % nsub) * rpb;
                        const int lp = tok / a.page_size;
                        const int npages_req = (rq.lk + a.page_size - 1) / a.page_size;
                        if (J < 0 || J > U.I) set_status(a.status, FP_ERR_DEVICE_BOUNDS);   // not a block of the row
                        else if (tok < rq.lk && lp < npages_req) {
                            const int pg = __ldg(a.block_table + (long long)U.r * a.max_pages + lp);
                            if (pg >= 0 && pg < a.num_pages) z = pg * a.page_size + tok % a.page_size;
                            else set_status(a.status, FP_ERR_DEVICE_BOUNDS);
                        }
                    }
                    M.z0[lane] = z;
                }
                if (lane == 0) {
                    M.pos = end ? -1 : pos;
                    M.unit = unit;
                    M.n_items = je - jb;
                    M.n_corr = n_corr;
                    M.jb = jb;
                    M.n_kept = n_kept;
                }
                __syncwarp();
                mbar_arrive(bar(BAR_MF + b));
                if (end) break;
            }
        } else if (warp == 0) {
            // ================= TMA producer =================
            // Lane 0 waits on the rings and issues the copies.  The page-table
            // lookups (the index entry, then the page of each sub-box) are done
            // by the whole warp, one round of 32 / nsub items at a time, a round
            // ahead, so their latency hides behind the copies of the round
            // before; K and V of an item share them.
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
            }
            const int rpb = a.page_size < kBlock ? a.page_size : kBlock;   // rows per box
            const int nsub = kBlock / rpb;                                 // boxes per tile: 1, 2, 4 or 8
            const int per = 32 / nsub;                                     // items per lookup round
            const int oob = a.num_pages * a.page_size;                     // zero-filled rows
            uint32_t it = 0;
            int kq = 0;
            // for the drain after an abort (lane 0): the Q phase armed last (-1:
            // none), and the tile (0: K, 1: V) whose slot wait gave up, if one did
            int q_ph = -1, fail_op = -1, q_bar = BAR_Q, nql = 0;
            for (int k = 0;; ++k) {
                const int b = k & 1;
                const UnitMeta &M = meta[b];
                bool got = true;
                if (lane == 0) got = mbar_wait(bar(BAR_MF + b), (k >> 1) & 1, abort_flag, a.status, a.wait_ns);
                if (!__shfl_sync(0xffffffffu, got, 0)) break;
                __syncwarp();                               // lane 0's acquire covers the warp's reads
                if (M.pos < 0) break;
                const int n_items = M.n_items;
                if (n_items > 0) {
                    const Unit U = decode_unit(bd, a, M.unit);
                    const ReqDesc &rq = bd.req[U.r];
                    const int *bt = a.block_table + (long long)U.r * a.max_pages;
                    const int npages_req = (rq.lk + a.page_size - 1) / a.page_size;
                    // this lane's lookup for item j0 + lane / nsub, box lane % nsub:
                    // the page id (in flight until used) and the row inside the page;
                    // page -1: past the request (zero fill), -2: not a kept item
                    auto look = [&](int j0, int &pg, int &off) {
                        const int jj = j0 + lane / nsub;
                        pg = -2;
                        off = 0;
                        if (jj < U.n_kept) {
                            const int J = sparse ? __ldg(a.col_idx + U.rp0 + jj) : jj;
                            const int tok = J * kBlock + (lane % nsub) * rpb;
                            const int lp = tok / a.page_size;
                            off = tok % a.page_size;
                            if (J < 0 || J > U.I) {               // not a block of the row: zero fill
                                set_status(a.status, FP_ERR_DEVICE_BOUNDS);
                                pg = -1;
                            } else {
                                pg = (tok < rq.lk && lp < npages_req) ? __ldg(bt + lp) : -1;
                            }
                        }
                    };
                    // row of the paged pool a looked-up box starts at
                    auto row_of = [&](int pg, int off) {
                        if (pg == -1 || pg == -2) return oob;
                        if (pg < 0 || pg >= a.num_pages) {
                            set_status(a.status, FP_ERR_DEVICE_BOUNDS);
                            return oob;
                        }
                        return pg * a.page_size + off;
                    };
                    bool good = true;
                    if (lane == 0) {
                        // Q of the previous unit is free once its last S MMAs are done
                        if (kq > 0 && !mbar_wait(bar(BAR_QE), (kq - 1) & 1, abort_flag, a.status, a.wait_ns)) good = false;
                        if (good) {
                            const int q_row0 = rq.q_off + U.il * kBlock;
                            // a bf16 unit that starts with a mean tile: the converter
                            // turns the queries to fp16 first, then completes BAR_Q
                            const bool conv_first = !kFp8 && kMean && sparse && a.mean_corr && M.jb >= U.n_kept;
                            q_bar = conv_first ? BAR_QL : BAR_Q;
                            q_ph = conv_first ? (nql++ & 1) : (kq & 1);
                            mbar_expect_tx(bar(q_bar), 2 * kT);
                            for (int t = 0; t < 2; ++t)
                                for (int hf = 0; hf < kNH; ++hf)
                                    tma_load_3d(sbase + kSmemQ + t * kTileBytes + hf * kHalfBytes, &tmQ, bar(q_bar),
                                                hf * 64, U.hq0 + t, q_row0);
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, good, 0)) break;
                    // terms jb .. jb + n_items - 1 of the row (this unit's part); the
                    // metadata warp looked up the first round, this warp the rest
                    const int jb = M.jb;
                    int pg_n, off_n;
                    look(jb + per, pg_n, off_n);
                    int z_cur = M.z0[lane];
                    for (int jl = 0; jl < n_items && good; ++jl, ++it) {
                        const int j = jb + jl;
                        const int lj = jl % per;
                        if (lj == 0 && jl > 0) {            // next round: take it, look up the one after
                            z_cur = row_of(pg_n, off_n);
                            look(j + per, pg_n, off_n);
                        }
                        const bool kept = !kMean || j < U.n_kept;
                        int zs[8];
#pragma unroll
                        for (int sub = 0; sub < 8; ++sub)
                            zs[sub] = __shfl_sync(0xffffffffu, z_cur, (lj * nsub + sub) & 31);
                        if (lane == 0) {
                            const int s = it & 1, ph = (it >> 1) & 1;
                            const int c = kept ? 0 : M.corr[j - U.n_kept];
                            for (int op = 0; op < 2 && good; ++op) {       // 0: K tile, 1: V tile
                                const uint32_t full = bar(op == 0 ? BAR_KF + s : BAR_VF + s);
                                if (it >= 2 && !mbar_wait(bar(op == 0 ? BAR_KE + s : BAR_VE + s), ph ^ 1, abort_flag,
                                                          a.status, a.wait_ns)) {
                                    good = false;
                                    fail_op = op;
                                    break;
                                }
                                const uint32_t dst = sbase + (op == 0 ? kSmemK : kSmemV) + s * kTileBytes;
                                // e4m3 mean K tiles carry a second (lo) term in the slot's upper half;
                                // kPlo V tiles arrive twice (both halves of the slot)
                                const bool two = (kFp8 && !kept && op == 0) || (kPlo && op == 1);
                                mbar_expect_tx(full, two ? 2 * kT : kT);
                                if (kept && kVdm && op == 1) {
                                    // d rows of 128 / esz keys per box (K-major): bf16 as two
                                    // 64-key halves, e4m3 as one box; a pool row z is page
                                    // z / page_size, key z % page_size (past the pool: zeros)
#pragma unroll
                                    for (int hf = 0; hf < kNH; ++hf) {
                                        const int z = zs[(hf * 64) / rpb] + (hf * 64) % rpb;
                                        tma_load_3d(dst + hf * kHalfBytes, &tmV, full, z % a.page_size, U.h * kHeadDim,
                                                    z / a.page_size);
                                        if (kPlo)
                                            tma_load_3d(dst + kT, &tmV, full, z % a.page_size, U.h * kHeadDim, z / a.page_size);
                                    }
                                } else if (kept) {
                                    const CUtensorMap *tm = op == 0 ? &tmK : &tmV;
#pragma unroll
                                    for (int sub = 0; sub < 8; ++sub)
                                        if (sub < nsub)
                                            for (int hf = 0; hf < kNH; ++hf) {
                                                tma_load_3d(dst + hf * kHalfBytes + sub * rpb * 128, tm, full, hf * 64,
                                                            U.h, zs[sub]);
                                                if (kPlo && op == 1)
                                                    tma_load_3d(dst + kT + sub * rpb * 128, tm, full, 0, U.h, zs[sub]);
                                            }
                                } else if (kFp8) {
                                    // e4m3 mean tile: K slot <- hi, and lo in its upper half; V slot
                                    // <- the value means (twice with kPlo)
                                    const CUtensorMap *tm = op == 0 ? &tmKm : &tmVm;
                                    tma_load_3d(dst, tm, full, 0, U.h, rq.kb_base + c * kBlock);
                                    if (two)
                                        tma_load_3d(dst + kHalfBytes, tm, full, 0, U.h,
                                                    (op == 0 ? a.mean_rows : 0) + rq.kb_base + c * kBlock);
                                } else {
                                    // bf16 mean tile: K slot <- the scaled fp16 key means of its 128
                                    // blocks, V slot <- the bf16 value means
                                    const int row0 = rq.kb_base + c * kMeanSpan;
                                    for (int hf = 0; hf < kNH; ++hf)
                                        tma_load_3d(dst + hf * kHalfBytes, op == 0 ? &tmKm : &tmVm, full, hf * 64, U.h, row0);
                                }
                            }
                        }
                        good = __shfl_sync(0xffffffffu, good, 0);
                    }
                    if (!good) break;
                    ++kq;
                }
                __syncwarp();                               // the warp's reads of the metadata are done
                if (lane == 0) mbar_arrive(bar(BAR_ME + b));
            }
            // after an abort, the copies armed last land before the CTA leaves
            // (otherwise every copy has been consumed already)
            if (lane == 0 && ld_shared_volatile(abort_flag)) {
                if (q_ph >= 0) mbar_wait_drain(bar(q_bar), q_ph);
                // items before `it` were armed in full, except the one whose slot
                // wait gave up: its K only when the V wait was the one that gave up
                const int nk = fail_op == 0 ? (int)it - 1 : (int)it;
                const int nv = fail_op >= 0 ? (int)it - 1 : (int)it;
                for (int i = nk - 2; i < nk; ++i)
                    if (i >= 0) mbar_wait_drain(bar(BAR_KF + (i & 1)), (i >> 1) & 1);
                for (int i = nv - 2; i < nv; ++i)
                    if (i >= 0) mbar_wait_drain(bar(BAR_VF + (i & 1)), (i >> 1) & 1);
            }
        } else if (warp == 1 && lane == 0) {
            // ================= MMA issuer =================
            constexpr uint32_t idS = kFp8 ? idesc_e4m3(128, 128, false) : idesc_bf16(128, 128, false);
            constexpr uint32_t idPV = kFp8 ? idesc_e4m3(128, 128, true) : idesc_bf16(128, 128, true);
            constexpr uint32_t idS16 = idesc_f16(128, 128, false);   // bf16 mean tiles: fp16 queries and keys
            constexpr int kKSteps = kFp8 ? 4 : 8;                // K = 32 (e4m3) or 16 (bf16) per MMA
            constexpr int kKeysPerStep = kFp8 ? 32 : 16;
            // descriptors differ only in the start address: add offsets (in 16-byte units)
            const uint64_t qdesc = smem_desc_sw128(sbase + kSmemQ, 16, 1024);
            const uint64_t kdesc = smem_desc_sw128(sbase + kSmemK, 16, 1024);
            const uint64_t vdesc = smem_desc_sw128(sbase + kSmemV, kFp8 ? 16 : kHalfBytes, 1024);
            const uint64_t kvdesc = smem_desc_sw128(sbase + kSmemV, 16, 1024);   // K-major V tiles (kVdm)
            // two: a mean tile.  e4m3: its keys come as hi + lo terms (the lo tile
            // sits in the upper half of the slot); bf16: queries and keys are fp16
            auto issue_S = [&](int t, int s, bool two) {
                const uint64_t qd = qdesc + ((t * kTileBytes) >> 4);
                const uint64_t kd = kdesc + ((s * kTileBytes) >> 4);
                const uint32_t id = !kFp8 && two ? idS16 : idS;
#pragma unroll
                for (int kk = 0; kk < kKSteps; ++kk) {
                    const uint32_t off = (kFp8 ? kk * 32 : (kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                    if constexpr (kFp8) mma_ss_f8(tmem + t * 256, qd + off, kd + off, idS, kk > 0);
                    else mma_ss(tmem + t * 256, qd + off, kd + off, id, kk > 0);
                }
                if constexpr (kFp8) {
                    if (two) {
#pragma unroll 1
                        for (int kk = 0; kk < kKSteps; ++kk)
                            mma_ss_f8(tmem + t * 256, qd + kk * 2, kd + (kHalfBytes >> 4) + kk * 2, idS, true);
                    }
                }
            };
            // kept: a kept block's tile, K-major when the value cache is dim-major
            // (the same descriptors and steps as the K operand of S); mean tiles
            // and token-major tiles are MN-major
            // kPlo: 256 virtual keys, A = [P_hi | P_lo] (TMEM columns 0..63) against
            // B = [V; V] (the slot holds the e4m3 tile twice)
            constexpr int kPvSteps = kPlo ? 2 * kKSteps : kKSteps;
            auto issue_PV = [&](int t, int s, bool acc, bool kept) {
                if (kVdm && kept) {
                    const uint64_t vd = kvdesc + ((s * kTileBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kPvSteps; ++kk) {
                        const uint32_t off =
                            (kFp8 ? (kk >> 2) * kT + (kk & 3) * 32 : (kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                        if constexpr (kFp8) mma_ts_f8(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, vd + off, idS, (acc || kk > 0));
                        else mma_ts(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, vd + off, idS, (acc || kk > 0));
                    }
                    return;
                }
                const uint64_t vd = vdesc + ((s * kTileBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kPvSteps; ++kk) {
                    const uint64_t b = vd + ((kk * kKeysPerStep * 128) >> 4);
                    if constexpr (kFp8) mma_ts_f8(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, b, idPV, (acc || kk > 0));
                    else mma_ts(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, b, idPV, (acc || kk > 0));
                }
            };
            uint32_t it = 0;
            int kq = 0;
            for (int k = 0;; ++k) {
                const int b = k & 1;
                if (!mbar_wait(bar(BAR_MF + b), (k >> 1) & 1, abort_flag, a.status, a.wait_ns)) break;
                const int pos = meta[b].pos, n_items = meta[b].n_items;
                const int first_mean = meta[b].n_kept - meta[b].jb;   // local index of the first mean tile
                mbar_arrive(bar(BAR_ME + b));
                if (pos < 0) break;
                if (n_items == 0) continue;
                if (!mbar_wait(bar(BAR_Q), kq & 1, abort_flag, a.status, a.wait_ns)) break;
                if (!mbar_wait(bar(BAR_KF + (it & 1)), (it >> 1) & 1, abort_flag, a.status, a.wait_ns)) break;
                tc_fence_after();
                issue_S(0, it & 1, first_mean <= 0);
                tc_commit(bar(BAR_SF + 0));
                issue_S(1, it & 1, first_mean <= 0);
                tc_commit(bar(BAR_SF + 1));
                tc_commit(bar(BAR_KE + (it & 1)));
                if (n_items == 1) tc_commit(bar(BAR_QE));
                bool good = true;
                for (int j = 0; j < n_items; ++j, ++it) {
                    const int s = it & 1, ph = (it >> 1) & 1;
                    const int s1 = (it + 1) & 1, ph1 = ((it + 1) >> 1) & 1;
                    const bool more = j + 1 < n_items;
                    if (!mbar_wait(bar(BAR_VF + s), ph, abort_flag, a.status, a.wait_ns) ||
                        !mbar_wait(bar(BAR_PF + 0), it & 1, abort_flag, a.status, a.wait_ns)) {
                        good = false;
                        break;
                    }
                    tc_fence_after();
                    issue_PV(0, s, j > 0, j < first_mean);
                    if (more) {
                        if (!mbar_wait(bar(BAR_KF + s1), ph1, abort_flag, a.status, a.wait_ns)) {
                            good = false;
                            break;
                        }
                        tc_fence_after();
                        issue_S(0, s1, j + 1 >= first_mean);
                        tc_commit(bar(BAR_SF + 0));
                    } else {
                        tc_commit(bar(BAR_OF + 0));
                    }
                    if (!mbar_wait(bar(BAR_PF + 1), it & 1, abort_flag, a.status, a.wait_ns)) {
                        good = false;
                        break;
                    }
                    tc_fence_after();
                    issue_PV(1, s, j > 0, j < first_mean);
                    tc_commit(bar(BAR_VE + s));
                    if (more) {
                        issue_S(1, s1, j + 1 >= first_mean);
                        tc_commit(bar(BAR_SF + 1));
                        tc_commit(bar(BAR_KE + s1));
                        if (j + 2 == n_items) tc_commit(bar(BAR_QE));   // the unit's last S MMAs
                    } else {
                        tc_commit(bar(BAR_OF + 1));
                    }
                }
                if (!good) break;
                ++kq;
            }
            if (ld_shared_volatile(abort_flag)) {          // after an abort, every MMA issued is done
                tc_commit(bar(BAR_DR));                // before the CTA leaves
                mbar_wait_drain(bar(BAR_DR), 0);
            }
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ================= softmax warpgroups =================
        const int t = (warp - 4) / 4;                 // tile
        const int quarter = warp % 4;                 // TMEM lane quarter of this warp
        const int rowt = quarter * 32 + lane;         // row of the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t tS = lane_base + t * 256;
        const uint32_t tO = tS + 128;
        uint32_t it = 0;
        int kq = 0, nqc = 0;                          // nqc: units whose queries this role converted first
        for (int k = 0; !dead; ++k) {
            const int b = k & 1;
            const UnitMeta &M = meta[b];
            const bool gotm = mbar_wait(bar(BAR_MF + b), (k >> 1) & 1, abort_flag, a.status, a.wait_ns);
            if (!__all_sync(0xffffffffu, gotm)) break;
            if (M.pos < 0) break;
            const int n_items = M.n_items;
            const Unit U = decode_unit(bd, a, M.unit);
            const ReqDesc &rq = bd.req[U.r];
            const int I = U.I, n_kept = U.n_kept;
            const int qi = U.il * kBlock + rowt;          // query index inside the request
            const int head = U.hq0 + t;
            if (n_items == 0) {
                // a row (or part) with no term at all: O = 0, LSE = -inf
                if (qi < rq.lq) {
                    const long long tok = rq.q_off + qi;
                    if (a.n_split > 1) {
                        float *pdst = a.part_o + (((long long)U.split * bd.total_q + tok) * bd.h_q + head) * kHeadDim;
                        for (int c = 0; c < kHeadDim; c += 4) *reinterpret_cast<float4 *>(pdst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                        a.part_lse[((long long)U.split * bd.h_q + head) * bd.total_q + tok] = -INFINITY;
                    } else {
                        __nv_bfloat16 *dst = a.out + (tok * bd.h_q + head) * kHeadDim;
                        for (int c = 0; c < kHeadDim; c += 8) *reinterpret_cast<uint4 *>(dst + c) = make_uint4(0, 0, 0, 0);
                        if (a.lse) a.lse[(long long)head * bd.total_q + tok] = -INFINITY;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_ME + b));
                continue;
            }
            const int pos = rq.start + qi;                // absolute position
            // l: sum of the weights the MMA multiplies (normalises O); e4m3 also
            // keeps lt, the sum of the unrounded weights, for the LSE: weights
            // below e4m3's range (a long row's tail) flush to zero in P, and the
            // LSE (which split-KV merges by) must still count them
            float m = -INFINITY, l = 0.f, lt = 0.f;

            const int last_J = n_kept == 0 ? -1 : (sparse ? __ldg(a.col_idx + U.rp0 + n_kept - 1) : n_kept - 1);
            bool ok = true;
            // logit scale (log2 units): e4m3 codes carry the per-head scales
            const float csc = kFp8 ? a.scale_log2 * __ldg(a.q_scale + head) * __ldg(a.k_scale + U.h) : a.scale_log2;
            // the running max moves only when it grows by more than kTau (bf16
            // tolerates weights up to 2^8).  For e4m3 it always follows the max, so
            // the largest weight of a row is exactly 256 = e4m3(256 * 1) and only
            // the smaller weights carry e4m3 rounding.
            constexpr float kTau = kFp8 ? 0.f : 8.f;
            const int jb = M.jb;                          // this unit's part: terms jb ..
            // bf16 mean tiles run on fp16 queries (2^f per row) and fp16 key means
            // (2^e per tile); fqr = 2^-f undoes the row's scale.  A part that starts
            // with a mean tile converts its queries here, once they land, and one
            // thread then completes BAR_Q for the MMA thread
            float fqr = 1.f;
            if (!kFp8 && kMean && sparse && a.mean_corr && jb >= n_kept) {
                const bool gq = mbar_wait(bar(BAR_QL), nqc & 1, abort_flag, a.status, a.wait_ns);
                if (!__all_sync(0xffffffffu, gq)) break;
                fqr = q_to_f16(sbase + kSmemQ + t * kTileBytes, rowt);
                fence_proxy_async();                      // before the MMAs read the tile
                mbar_arrive(bar(BAR_QC));
                if (threadIdx.x == 128) {
                    const bool gc = mbar_wait(bar(BAR_QC), nqc & 1, abort_flag, a.status, a.wait_ns);
                    if (gc) mbar_arrive(bar(BAR_Q));
                }
                ++nqc;
            }
            for (int jl = 0; jl < n_items; ++jl, ++it) {
                const int j = jb + jl;
                const bool got = mbar_wait(bar(BAR_SF + t), it & 1, abort_flag, a.status, a.wait_ns);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }   // tcgen05.ld needs the whole warp
                tc_fence_after();
                uint32_t v[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, v[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence(v[c]);
                // raw logits; masked entries -inf.  The scale and the mean-token
                // bias are applied inside the exponent: p = 2^(s*c + bias - m).
                float x[128];
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[c][e]);
                float bias = 0.f;
                float cs = csc;                           // logit scale of this term (log2 units)
                // columns to keep, as four 32-bit words: the diagonal block keeps
                // keys up to the query's position; a mean tile c (blocks kMeanSpan*c
                // .. +kMeanSpan-1) keeps its skipped blocks J < I.  A skipped block
                // J < I is full (only the request's last block can be short, and it
                // is never before I), so its weight is n_J = 128: bias log2(128)
                uint32_t w[4] = {~0u, ~0u, ~0u, ~0u};
                bool masked = false;
                if (!kMean || j < n_kept) {
                    // kept blocks ascend and J <= I: only the last one can be the
                    // diagonal block, the one that needs the causal mask
                    const int k0 = j == n_kept - 1 ? last_J * kBlock : 0;
                    if (k0 + kBlock - 1 > pos) {
                        masked = true;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int n = pos - k0 - 32 * q + 1;          // keys of word q at or before pos
                            w[q] = n <= 0 ? 0u : (n >= 32 ? ~0u : ((1u << n) - 1u));
                        }
                    }
                } else {
                    masked = true;
                    const int c = M.corr[j - n_kept];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int J0 = c * kMeanSpan + 32 * q;
                        uint32_t valid = J0 >= I ? 0u : (I - J0 >= 32 ? 0xffffffffu : ((1u << (I - J0)) - 1u));
                        w[q] = valid ? (~M.bitmap[J0 >> 5] & valid) : 0u;   // 1 = skipped, before I
                    }
                    bias = 7.f;
                    if constexpr (!kFp8)                      // both fp16 scales undone (powers of two)
                        cs = csc * fqr * pow2f(-(int)__ldg(a.kexp + (long long)(rq.kb_base + c * kMeanSpan) * bd.h_kv + U.h));
                }
                if (masked) {
#pragma unroll
                    for (int e = 0; e < 128; ++e)
                        if (!((w[e >> 5] >> (e & 31)) & 1u)) x[e] = -INFINITY;
                }
                // row max in independent chains of three-input max, then a tree:
                // sixteen chains (at most four deep) for bf16; eight for e4m3,
                // whose exponent loop leaves fewer registers
                float mxr;
                if constexpr (!kFp8) {
                    float mx16[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) mx16[q] = max3f(x[3 * q], x[3 * q + 1], x[3 * q + 2]);
#pragma unroll
                    for (int e = 48; e < 128; e += 2)
                        mx16[((e - 48) >> 1) & 15] = max3f(mx16[((e - 48) >> 1) & 15], x[e], x[e + 1]);
                    mxr = max3f(max3f(max3f(mx16[0], mx16[1], mx16[2]), max3f(mx16[3], mx16[4], mx16[5]),
                                      max3f(mx16[6], mx16[7], mx16[8])),
                                max3f(mx16[9], mx16[10], mx16[11]),
                                max3f(max3f(mx16[12], mx16[13], mx16[14]), mx16[15], mx16[15]));
                } else {
                    float mx8[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) mx8[q] = x[q];
#pragma unroll
                    for (int e = 8; e < 128; e += 2) mx8[(e >> 1) & 7] = max3f(mx8[(e >> 1) & 7], x[e], x[e + 1]);
                    mxr = fmaxf(max3f(mx8[0], mx8[1], mx8[2]), max3f(max3f(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                }
                const float mx = mxr * cs + bias;                    // log2 units; -inf stays -inf
                // grow the running max only when it rises by more than 2^8 (rarely);
                // O is rescaled after P is written (x is dead by then), and the
                // TMEM round trip runs warp-wide
                const bool grow = mx > m + kTau;
                const bool any_grow = __any_sync(0xffffffffu, grow);
                const float f = grow ? fast_exp2(m - mx) : 1.f;   // 0 when m = -inf
                if (grow) {
                    l *= f;
                    if constexpr (kFp8 && (kLse || kPlo)) lt *= f;
                    m = mx;
                }
                const float off = bias - (m == -INFINITY ? 0.f : m);
                // exponents as paired FMAs: (s0, s1) * c + off.  P goes to TMEM
                // first; the denominator is summed from the packed registers after
                // the MMA has been told P is ready, off the critical path.
                const uint64_t cc = f2_pack(cs, cs);
                constexpr int kPk = kFp8 ? 32 : 64;   // packed words of P per row
                uint32_t pk[kPk];
                uint32_t pr[kPlo ? 32 : 1];           // kPlo: the residual term of P
                if constexpr (!kFp8) {
                    const uint64_t oo = f2_pack(off, off);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            float z0, z1;
                            f2_unpack(f2_fma(f2_pack(x[64 * half + 2 * e], x[64 * half + 2 * e + 1]), cc, oo), z0, z1);
                            pk[32 * half + e] = pack_bf16(fast_exp2(z0), fast_exp2(z1));
                        }
                        tmem_st32(tS + 32 * half, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32 * half));
                    }
                } else {
                    // e4m3 of 256 * p: four weights per TMEM column (and, with
                    // kLse, the sum of the unrounded weights)
                    const uint64_t oo = f2_pack(off + 8.f, off + 8.f);
                    auto exps = [&](auto with_sum) {
                        uint64_t ltp[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            float z0, z1, z2, z3;
                            f2_unpack(f2_fma(f2_pack(x[4 * e], x[4 * e + 1]), cc, oo), z0, z1);
                            f2_unpack(f2_fma(f2_pack(x[4 * e + 2], x[4 * e + 3]), cc, oo), z2, z3);
                            const float p0 = fast_exp2(z0), p1 = fast_exp2(z1), p2 = fast_exp2(z2), p3 = fast_exp2(z3);
                            if constexpr (decltype(with_sum)::value) {
                                ltp[0] = f2_add(ltp[0], f2_pack(p0, p1));
                                ltp[1] = f2_add(ltp[1], f2_pack(p2, p3));
                            }
                            const __nv_fp8x2_storage_t lo =
                                __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
                            const __nv_fp8x2_storage_t hi =
                                __nv_cvt_float2_to_fp8x2(make_float2(p2, p3), __NV_SATFINITE, __NV_E4M3);
                            pk[e] = (uint32_t)lo | ((uint32_t)hi << 16);
                            if constexpr (kPlo) {
                                const float2 d01 = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3)));
                                const float2 d23 = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
                                float r0, r1, r2, r3;
                                f2_unpack(f2_add(f2_pack(p0, p1), f2_pack(-d01.x, -d01.y)), r0, r1);
                                f2_unpack(f2_add(f2_pack(p2, p3), f2_pack(-d23.x, -d23.y)), r2, r3);
                                const __nv_fp8x2_storage_t rl =
                                    __nv_cvt_float2_to_fp8x2(make_float2(r0, r1), __NV_SATFINITE, __NV_E4M3);
                                const __nv_fp8x2_storage_t rh =
                                    __nv_cvt_float2_to_fp8x2(make_float2(r2, r3), __NV_SATFINITE, __NV_E4M3);
                                pr[e] = (uint32_t)rl | ((uint32_t)rh << 16);
                            }
                        }
                        tmem_st32(tS, *reinterpret_cast<const uint32_t(*)[32]>(pk));
                        if constexpr (kPlo) tmem_st32(tS + 32, *reinterpret_cast<const uint32_t(*)[32]>(pr));
                        if constexpr (decltype(with_sum)::value) {
                            float t0, t1, t2, t3;
                            f2_unpack(ltp[0], t0, t1);
                            f2_unpack(ltp[1], t2, t3);
                            lt += (t0 + t1) + (t2 + t3);
                        }
                    };
                    // kPlo: the denominator is the fp32 sum of the unrounded weights
                    // (the two terms carry ~2^-8 relative), taken here
                    exps(std::integral_constant<bool, kLse || kPlo>{});
                }
                if (any_grow && jl > 0) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait();
                        reg_fence(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st32(tO + c * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                // bf16: after the last kept block of a part with mean tiles, this
                // thread's query row goes to fp16 before P is handed over, so the
                // tile's next S (a mean tile) reads fp16 queries
                const bool conv = !kFp8 && kMean && sparse && a.mean_corr && j == n_kept - 1 && jl + 1 < n_items;
                if (!conv) mbar_arrive(bar(BAR_PF + t));
                // the denominator sums the same rounded weights the MMA multiplies,
                // so the weights of a row sum to exactly one
                float rs;
                if constexpr (!kFp8) {
                    uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        acc2[e & 1] = f2_add(acc2[e & 1], f2_pack(__uint_as_float(pk[e] << 16),
                                                                  __uint_as_float(pk[e] & 0xffff0000u)));
                    float r0, r1, r2, r3;
                    f2_unpack(acc2[0], r0, r1);
                    f2_unpack(acc2[1], r2, r3);
                    rs = (r0 + r1) + (r2 + r3);
                } else if constexpr (kPlo) {
                    rs = 0.f;                               // summed into lt with the exponentials
                } else {
                    // decoded e4m3 weights summed in half2 (<= 128 * 256 < 65504)
                    __half2 hs[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) hs[q] = __float2half2_rn(0.f);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const __nv_fp8x2_storage_t lo = (__nv_fp8x2_storage_t)(pk[e] & 0xffffu);
                        const __nv_fp8x2_storage_t hi = (__nv_fp8x2_storage_t)(pk[e] >> 16);
                        hs[e & 3] = __hadd2(hs[e & 3], __hadd2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3)),
                                                               __half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3))));
                    }
                    const float2 f0 = __half22float2(hs[0]), f1 = __half22float2(hs[1]);
                    const float2 f2 = __half22float2(hs[2]), f3 = __half22float2(hs[3]);
                    rs = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
                }
                l += rs;
                if (conv) {
                    fqr = q_to_f16(sbase + kSmemQ + t * kTileBytes, rowt);
                    fence_proxy_async();                  // before the MMAs read the tile
                    mbar_arrive(bar(BAR_PF + t));
                }
            }
            if (!ok) break;
            // epilogue: O / l -> bf16, LSE.  The unit's fields are decoded again
            // from the metadata (released only after this) rather than kept live
            // across the item loop.
            const Unit V = decode_unit(bd, a, M.unit);
            const ReqDesc &rv = bd.req[V.r];
            const int qv = V.il * kBlock + rowt;
            const int hv = V.hq0 + t;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_ME + b));
            const bool valid = qv < rv.lq;
            const bool fin = mbar_wait(bar(BAR_OF + t), kq & 1, abort_flag, a.status, a.wait_ns);
            if (!__all_sync(0xffffffffu, fin)) break;
            tc_fence_after();
            // O = (sum of weights * v codes) * v_scale / (sum of weights); for e4m3
            // both sums carry the factor 256, which cancels
            const float den = kPlo ? lt : l;               // kPlo: the unrounded weights' sum
            const float inv = den > 0.f ? (kFp8 ? __ldg(a.v_scale + V.h) : 1.f) / den : 0.f;
            const long long tok = rv.q_off + qv;
            const bool part = a.n_split > 1;            // split-KV: fp32 partial O of this part
            __nv_bfloat16 *dst = a.out + (tok * bd.h_q + hv) * kHeadDim;
            float *pdst = part ? a.part_o + (((long long)V.split * bd.total_q + tok) * bd.h_q + hv) * kHeadDim : nullptr;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_ld_wait();
                reg_fence(o);
                if (valid && !part) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + c * 32 + e) = w;
                    }
                } else if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(pdst + c * 32 + e) =
                            make_float4(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv,
                                        __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                }
            }
            // the next unit's first PV MMA overwrites O only after this warp
            // group's next P handshake, which follows these reads
            tc_fence_before();
            const float lsum = kFp8 && (kLse || kPlo) ? lt : l;
            const float lse_v =
                den > 0.f ? (m + __log2f(lsum) - (kFp8 ? 8.f : 0.f)) * 0.6931471805599453f : -INFINITY;
            if (valid && part) a.part_lse[((long long)V.split * bd.h_q + hv) * bd.total_q + tok] = lse_v;
            else if (valid && a.lse) a.lse[(long long)hv * bd.total_q + tok] = lse_v;
            ++kq;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}
// ---------------------------------------------------------------------------
// schedule: the order in which the persistent CTAs take units.  Units are
// grouped by (request, kv head), so the units in flight share one head's K and
// V (64 MB for a 128K request) and hit L2 instead of re-reading DRAM; groups
// go by decreasing row length (the requests with the longest rows first, kv
// heads in order), and inside a group rows go by decreasing work (kept blocks
// plus mean tiles), so the tail of the launch is short rows (the kept-count
// load balancing of the V2 popular article, "KV split").  One CTA per group:
// a counting sort of its rows by work.
// ---------------------------------------------------------------------------
constexpr int kSchedBins = 4096;
constexpr int kSchedThreads = 1024;

__global__ void __launch_bounds__(kSchedThreads)
sched_kernel(const __grid_constant__ BatchDesc bd, const int *__restrict__ row_ptr, int n_pairs, int n_split,
             int mean_span, int *__restrict__ work, int *__restrict__ next_unit) {
    __shared__ int hist[kSchedBins];
    __shared__ int warp_sum[kSchedThreads / 32];
    __shared__ int grp[3];                          // request, kv head, first position of the group
    const int tid = threadIdx.x, lane = tid % 32, wid = tid / 32;
    if (tid == 0) {
        if (blockIdx.x == 0) *next_unit = 0;
        int ord[FP_MAX_BATCH];
        for (int r = 0; r < bd.batch; ++r) {          // insertion sort: nkb descending, index ascending
            int k = r;
            while (k > 0 && bd.req[ord[k - 1]].nkb < bd.req[r].nkb) {
                ord[k] = ord[k - 1];
                --k;
            }
            ord[k] = r;
        }
        const int rank = blockIdx.x / bd.h_kv, h = blockIdx.x % bd.h_kv;
        int base = 0;
        const int per_row = n_pairs * n_split;          // units of one index row
        for (int k = 0; k < rank; ++k) base += bd.req[ord[k]].nqb * bd.h_kv * per_row;
        const int r = ord[rank];
        grp[0] = r;
        grp[1] = h;
        grp[2] = base + h * bd.req[r].nqb * per_row;
    }
    for (int k = tid; k < kSchedBins; k += kSchedThreads) hist[k] = 0;
    __syncthreads();
    const ReqDesc &rq = bd.req[grp[0]];
    const int h = grp[1], base = grp[2];
    auto cost = [&](int il) {
        const int row = rq.row_base + il * bd.h_kv + h;
        const int I = rq.start / kBlock + il;
        const int c = row_ptr ? row_ptr[row + 1] - row_ptr[row] + (mean_span ? (I + mean_span - 1) / mean_span : 0)
                              : I + 1;
        return kSchedBins - 1 - min(c, kSchedBins - 1);     // bin 0 = the most work
    };
    for (int il = tid; il < rq.nqb; il += kSchedThreads) atomicAdd(&hist[cost(il)], 1);
    __syncthreads();
    // exclusive scan of the bins: four consecutive bins per thread, then the block
    constexpr int kPer = kSchedBins / kSchedThreads;
    int v[kPer], run = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        v[k] = hist[tid * kPer + k];
        run += v[k];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int w = warp_sum[lane], wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        warp_sum[lane] = wi - w;                    // exclusive prefix of the warps
    }
    __syncthreads();
    int pre = warp_sum[wid] + incl - run;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        hist[tid * kPer + k] = pre;
        pre += v[k];
    }
    __syncthreads();
    for (int il = tid; il < rq.nqb; il += kSchedThreads) {
        const int slot = atomicAdd(&hist[cost(il)], 1);
        const int row = rq.row_base + il * bd.h_kv + h;
        const int per_row = n_pairs * n_split;
        for (int u = 0; u < per_row; ++u) work[base + slot * per_row + u] = row * per_row + u;
    }
}

// split-KV merge: O = sum_s e^{LSE_s - LSE} O_s, LSE = ln sum_s e^{LSE_s}, one warp
// per (query, head), four values of d per lane
__global__ void __launch_bounds__(256)
combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse, int n_split, long long total_q,
               int h_q, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse) {
    const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (w >= total_q * h_q) return;
    const long long tok = w / h_q;
    const int head = (int)(w % h_q);
    float mx = -INFINITY;
    for (int s = 0; s < n_split; ++s) mx = fmaxf(mx, __ldg(part_lse + ((long long)s * h_q + head) * total_q + tok));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (mx != -INFINITY) {
        for (int s = 0; s < n_split; ++s) {
            const float ls = __ldg(part_lse + ((long long)s * h_q + head) * total_q + tok);
            const float wgt = ls == -INFINITY ? 0.f : __expf(ls - mx);
            den += wgt;
            const float4 o = __ldg(reinterpret_cast<const float4 *>(part_o + (((long long)s * total_q + tok) * h_q + head) * kHeadDim) + lane);
            acc.x = fmaf(wgt, o.x, acc.x);
            acc.y = fmaf(wgt, o.y, acc.y);
            acc.z = fmaf(wgt, o.z, acc.z);
            acc.w = fmaf(wgt, o.w, acc.w);
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint2 pk;
    pk.x = pack_bf16(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(out + (tok * h_q + head) * kHeadDim + 4 * lane) = pk;
    if (lse && lane == 0) lse[(long long)head * total_q + tok] = den > 0.f ? mx + __logf(den) : -INFINITY;
}

// fp32 block means -> the operands of the bf16 mean tiles.  One CTA per mean
// tile (128 blocks of a request from its first block) and kv head: the key
// means, scaled by the power of two 2^e that puts the tile's largest magnitude
// in [2^14, 2^15), as fp16 (11 significant bits); e at kexp[tile's first
// block][h]; the value means as bf16 (they enter O linearly).  Rows past the
// last request's blocks (up to rows_pad) are zero, so the zero weights of
// their columns meet finite values.
// The scale exponents of the bf16 mean tiles sit in the workspace space of
// the (e4m3-only) second key term: total_kb * h_kv bytes.
static int8_t *mean_kexp(const AttnLaunch &L, const BatchDesc &bd) {
    const size_t term = ((size_t)mean_rows(bd) * bd.h_kv * kHeadDim * 2 + 255) / 256 * 256;
    return reinterpret_cast<int8_t *>(L.km16) + term;
}

constexpr int kMeanThreads = 1024;
__global__ void __launch_bounds__(kMeanThreads)
mean_tiles_f16_kernel(const __grid_constant__ BatchDesc bd, const float *__restrict__ km, const float *__restrict__ vm,
                      __half *__restrict__ ko, __nv_bfloat16 *__restrict__ vo, int8_t *__restrict__ kexp, int rows_pad) {
    int b = blockIdx.x, r = 0;
    for (; r < bd.batch; ++r) {
        const int nc = (bd.req[r].nkb + kBlock - 1) / kBlock;
        if (b < nc) break;
        b -= nc;
    }
    if (r == bd.batch) return;
    const ReqDesc &rq = bd.req[r];
    const int h = blockIdx.y;
    const int row0 = rq.kb_base + b * kBlock;
    const int nrow = min(kBlock, rq.nkb - b * kBlock);
    const bool last = r == bd.batch - 1;
    const int col = (threadIdx.x % 32) * 4;          // four dims
    const int rw = threadIdx.x / 32;                 // rows rw, rw + 32, ...
    float4 v[4], w[4];                               // key and value means of rows rw + 32 k
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int rr = rw + 32 * k;
        const long long o = ((long long)(row0 + rr) * bd.h_kv + h) * kHeadDim + col;
        v[k] = rr < nrow ? __ldg(reinterpret_cast<const float4 *>(km + o)) : make_float4(0.f, 0.f, 0.f, 0.f);
        w[k] = rr < nrow ? __ldg(reinterpret_cast<const float4 *>(vm + o)) : make_float4(0.f, 0.f, 0.f, 0.f);
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
    }
    __shared__ float red[kMeanThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int k = 1; k < kMeanThreads / 32; ++k) mx = fmaxf(mx, red[k]);
    const int e = fp16_scale_exp(__float_as_uint(mx));
    const float sf = pow2f(e);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int rr = rw + 32 * k;
        if (rr >= nrow && !(last && row0 + rr < rows_pad)) continue;
        const long long o = ((long long)(row0 + rr) * bd.h_kv + h) * kHeadDim + col;
        const __half2 k01 = __floats2half2_rn(v[k].x * sf, v[k].y * sf), k23 = __floats2half2_rn(v[k].z * sf, v[k].w * sf);
        *reinterpret_cast<uint2 *>(ko + o) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&k01), *reinterpret_cast<const uint32_t *>(&k23));
        *reinterpret_cast<uint2 *>(vo + o) = make_uint2(pack_bf16(w[k].x, w[k].y), pack_bf16(w[k].z, w[k].w));
    }
    if (threadIdx.x == 0) kexp[(long long)row0 * bd.h_kv + h] = (int8_t)e;
}

// fp32 block means -> e4m3 codes with the per-head K / V scales (block means
// never exceed the largest |value| the scale maps to 448); [n, n_pad) is zeroed.
// The key means get two terms, hi at ao[k] and lo = e4m3(x - hi) at
// ao[n_pad + k] (about 8 significant bits together): a mean token's logit
// enters the exponent, and one e4m3 term (2^-4 relative) moved the LSE of
// long sharp rows by ~0.1.  The value means keep one term (they enter O
// linearly).
__global__ void to_e4m3_kernel(const float *__restrict__ a, const float *__restrict__ b, const float *__restrict__ sa,
                               const float *__restrict__ sb, uint8_t *__restrict__ ao, uint8_t *__restrict__ bo,
                               long long n, long long n_pad, int h_kv) {
    for (long long k = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 2; k < n_pad;
         k += (long long)gridDim.x * blockDim.x * 2) {
        const int h = (int)((k / kHeadDim) % h_kv);
        const float ia = 1.f / __ldg(sa + h), ib = 1.f / __ldg(sb + h);
        const float2 va = k < n ? make_float2(a[k] * ia, a[k + 1] * ia) : make_float2(0.f, 0.f);
        const float2 vb = k < n ? make_float2(b[k] * ib, b[k + 1] * ib) : make_float2(0.f, 0.f);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(va, __NV_SATFINITE, __NV_E4M3);
        const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
        *reinterpret_cast<__nv_fp8x2_storage_t *>(ao + k) = hi;
        *reinterpret_cast<__nv_fp8x2_storage_t *>(ao + n_pad + k) =
            __nv_cvt_float2_to_fp8x2(make_float2(va.x - hf.x, va.y - hf.y), __NV_SATFINITE, __NV_E4M3);
        *reinterpret_cast<__nv_fp8x2_storage_t *>(bo + k) = __nv_cvt_float2_to_fp8x2(vb, __NV_SATFINITE, __NV_E4M3);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
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

static bool debug_on() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("FPREFILL_DEBUG");
        v = (e && *e && *e != '0') ? 1 : 0;
    }
    return v == 1;
}

static int fail(const char *what, int code) {
    if (debug_on()) fprintf(stderr, "[fprefill] %s failed (%d)\n", what, code);
    return FP_ERR_CUDA;
}

// 3-D map over [n2][n1][128] elements (bf16, or bytes for e4m3) with strides
// (in elements) s1, s2; box (one 128-byte row of d, 1, box2), 128-byte
// swizzle, zero fill out of bounds.
static bool make_map(CUtensorMap *m, const void *base, long long n1, long long n2, long long s1, long long s2,
                     int box2, bool fp8 = false, bool f16 = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        fail("cuTensorMapEncodeTiled lookup", 0);
        return false;
    }
    const int esz = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)n1, (cuuint64_t)n2};
    cuuint64_t strides[2] = {(cuuint64_t)(s1 * esz), (cuuint64_t)(s2 * esz)};
    cuuint32_t box[3] = {(cuuint32_t)(128 / esz), 1, (cuuint32_t)box2};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : (f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16), 3,
                    const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && debug_on())
        fprintf(stderr, "[fprefill] tensor map dims (128,%lld,%lld) strides (%lld,%lld) box2 %d: CUresult %d\n",
                n1, n2, s1 * esz, s2 * esz, box2, (int)r);
    return r == CUDA_SUCCESS;
}

// 3-D map over a dim-major value cache [num_pages][h_kv * 128][page_size]:
// box (128 bytes of keys, the 128 d rows of one head, one page), 128-byte
// swizzle, zero fill out of bounds (a page index past the pool reads zeros).
static bool make_map_dm(CUtensorMap *m, const void *base, int h_kv, int page_size, int num_pages, bool fp8) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        fail("cuTensorMapEncodeTiled lookup", 0);
        return false;
    }
    const int esz = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)page_size, (cuuint64_t)h_kv * kHeadDim, (cuuint64_t)num_pages};
    cuuint64_t strides[2] = {(cuuint64_t)page_size * esz, (cuuint64_t)h_kv * kHeadDim * page_size * esz};
    cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)kHeadDim, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && debug_on())
        fprintf(stderr, "[fprefill] dim-major V map (%d,%d,%d): CUresult %d\n", page_size, h_kv * kHeadDim, num_pages,
                (int)r);
    return r == CUDA_SUCCESS;
}

int attn_smem_bytes() { return kSmemAttn; }

// The failure path of the bounded waits, without a fault: one thread waits on
// an mbarrier that nothing arrives on, through the same wait the kernels use,
// and records FP_ERR_TIMEOUT when the limit runs out.
__global__ void wait_timeout_kernel(int *status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
        mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
    }
}
cudaError_t launch_wait_timeout(int *status, unsigned long long limit_ns, cudaStream_t st) {
    wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit_ns);
    return cudaGetLastError();
}

// returns 0 on success, otherwise an fp_status
int launch_attn(const AttnLaunch &L, cudaStream_t st) {
    const BatchDesc &bd = *L.bd;
    const int n_pairs = bd.g / 2;
    const bool sparse = L.row_ptr != nullptr;
    const int n_split = L.n_split > 1 ? L.n_split : 1;
    const int units = bd.total_rows * n_pairs * n_split;
    if (units == 0) return FP_OK;
    const int rpb = L.page_size < kBlock ? L.page_size : kBlock;
    CUtensorMap tmQ, tmK, tmV, tmKm, tmVm;
    const long long total_q = bd.total_q;
    const long long tokens = (long long)L.num_pages * L.page_size;
    const bool f8 = L.fp8;
    if (!make_map(&tmQ, L.q, bd.h_q, total_q, L.q_stride_head, L.q_stride_tok, kBlock, f8)) return fail("Q map", 0);
    if (!make_map(&tmK, L.k_cache, bd.h_kv, tokens, kHeadDim, (long long)bd.h_kv * kHeadDim, rpb, f8))
        return fail("K map", 0);
    if (L.v_dim_major ? !make_map_dm(&tmV, L.v_cache, bd.h_kv, L.page_size, L.num_pages, f8)
                      : !make_map(&tmV, L.v_cache, bd.h_kv, tokens, kHeadDim, (long long)bd.h_kv * kHeadDim, rpb, f8))
        return fail("V map", 0);
    const bool use_means = sparse && L.mean_corr;
    cudaError_t e;
    if (use_means) {
        // rows past the last block (padding up to one full 128-row box) are zero
        const long long n = (long long)bd.total_kb * bd.h_kv * kHeadDim;
        const long long n_pad = (long long)mean_rows(bd) * bd.h_kv * kHeadDim;
        if (f8) {
            to_e4m3_kernel<<<1024, 256, 0, st>>>(L.k_mean, L.v_mean, L.k_scale, L.v_scale, (uint8_t *)L.km16,
                                                 (uint8_t *)L.vm16, n, n_pad, bd.h_kv);
        } else {
            int tiles = 0;
            for (int r = 0; r < bd.batch; ++r) tiles += (bd.req[r].nkb + kBlock - 1) / kBlock;
            if (tiles > 0)
                mean_tiles_f16_kernel<<<dim3(tiles, bd.h_kv), kMeanThreads, 0, st>>>(
                    bd, L.k_mean, L.v_mean, reinterpret_cast<__half *>(L.km16), L.vm16, mean_kexp(L, bd), mean_rows(bd));
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return fail("mean conversion launch", (int)e);
        // e4m3: the key means' hi rows [0, mean_rows), lo rows [mean_rows, 2 mean_rows);
        // bf16: one fp16 term.  Both load 128-row boxes.
        if (!make_map(&tmKm, L.km16, bd.h_kv, (f8 ? 2LL : 1LL) * mean_rows(bd), kHeadDim, (long long)bd.h_kv * kHeadDim,
                      kBlock, f8, !f8))
            return fail("mean K map", 0);
        if (!make_map(&tmVm, L.vm16, bd.h_kv, mean_rows(bd), kHeadDim, (long long)bd.h_kv * kHeadDim, kBlock, f8))
            return fail("mean V map", 0);
    } else {
        tmKm = tmK;     // never read
        tmVm = tmV;
    }
    int *next_unit = L.work + units;
    const int mean_span = use_means ? kBlock : 0;
    sched_kernel<<<bd.batch * bd.h_kv, kSchedThreads, 0, st>>>(bd, L.row_ptr, n_pairs, n_split, mean_span, L.work,
                                                              next_unit);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail("schedule launch", (int)e);
    AttnArgs a;
    a.row_ptr = L.row_ptr;
    a.col_idx = L.col_idx;
    a.work = L.work;
    a.next_unit = next_unit;
    a.n_units = units;
    a.block_table = L.block_table;
    a.max_pages = L.max_pages;
    a.page_size = L.page_size;
    a.num_pages = L.num_pages;
    a.n_pairs = n_pairs;
    a.n_split = n_split;
    a.part_o = L.part_o;
    a.part_lse = L.part_lse;
    a.mean_corr = use_means ? 1 : 0;
    a.mean_rows = mean_rows(bd);
    a.kexp = use_means && !f8 ? mean_kexp(L, bd) : nullptr;
    a.scale_log2 = L.softmax_scale * 1.4426950408889634f;
    a.q_scale = L.q_scale;
    a.k_scale = L.k_scale;
    a.v_scale = L.v_scale;
    a.out = (__nv_bfloat16 *)L.out;
    a.lse = L.lse;
    a.status = L.status;
    a.wait_ns = L.wait_ns;
    const bool want_lse = L.lse != nullptr || n_split > 1;
    const bool plo = f8 && L.p_terms == 2;
    auto kern = L.v_dim_major
                    ? (f8 ? (plo ? (want_lse ? attn_kernel<true, true, true, true> : attn_kernel<true, false, true, true>)
                                 : (want_lse ? attn_kernel<true, true, true> : attn_kernel<true, false, true>))
                          : (use_means ? attn_kernel<false, false, true> : attn_kernel<false, false, true, false, false>))
                    : (f8 ? (plo ? (want_lse ? attn_kernel<true, true, false, true> : attn_kernel<true, false, false, true>)
                                 : (want_lse ? attn_kernel<true, true, false> : attn_kernel<true, false, false>))
                          : (use_means ? attn_kernel<false, false, false> : attn_kernel<false, false, false, false, false>));
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAttn)) != cudaSuccess)
        return fail("attention smem attribute", (int)e);
    // persistent: one CTA per SM (the shared memory admits one), never more than units
    int dev = 0, n_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return fail("SM count", (int)e);
    const int grid = units < n_sm ? units : n_sm;
    kern<<<grid, kAttnThreads, kSmemAttn, st>>>(bd, tmQ, tmK, tmV, tmKm, tmVm, a);
    if ((e = cudaGetLastError()) != cudaSuccess) {
        if (debug_on()) fprintf(stderr, "[fprefill] attention launch: %s\n", cudaGetErrorString(e));
        return fail("attention launch", (int)e);
    }
    if (n_split > 1) {
        const long long warps = (long long)bd.total_q * bd.h_q;
        const long long blocks = (warps * 32 + 255) / 256;
        combine_kernel<<<(unsigned)blocks, 256, 0, st>>>(L.part_o, L.part_lse, n_split, bd.total_q, bd.h_q,
                                                         (__nv_bfloat16 *)L.out, L.lse);
        if ((e = cudaGetLastError()) != cudaSuccess) return fail("split-KV merge launch", (int)e);
    }
    return FP_OK;
}

}  // namespace fp
