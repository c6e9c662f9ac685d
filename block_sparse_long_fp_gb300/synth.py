"""Seeded synthetic inputs for block-sparse causal prefill attention.

This module only draws random numbers and lays them out in memory (paged KV
cache, block table, varlen descriptors).  It contains none of the method's
arithmetic (no pooling, scoring, thresholding or attention), so both the CUDA
path and the float64 oracle can take their inputs from it.

Recipe (FlashPrefill V1 "3.1 instantaneous pattern discovery" motivates the
block-coherent structure; the sink/needle structure follows the sink / local /
sparse-block patterns described in the FlashPrefill V2 paper reading, section
1.2):

* per head, independently for Q and K:  x_t = 0.6 * u[t // 128] + 0.8 * n_t,
  u, n ~ N(0, I_d)  (positions t are absolute token positions);
* one random unit vector s per kv head, shared by its g query heads; keys with
  t < 256 get +3 s, every query gets +1 s;
* "needles": for a kv head, a key block j in [2, nkb-5] takes u^K_j = 2 u^Q_i of
  one random query head of the group and a later query block i >= j + 4;
* V ~ N(0, I_d);
* optional ``logit_scale`` c multiplies every query (a sharper model).

Values are rounded to bf16 (round to nearest even) or, for the FP8 variant, to
e4m3 with one scale per head (amax / 448).  Seeds: ``1000*config + 10*request
+ kind`` with kind 0=Q, 1=K, 2=V, 3=shared (s, needles), 4=page order.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

BLOCK = 128          # block length of the generator's coherent structure
SINK_BOOST_TOKENS = 256

_POISON_BF16 = np.uint16(0x4280)   # 64.0: fills token slots past a request's end
_POISON_E4M3 = np.uint8(0x7E)      # 448.0 before scaling


@dataclass
class Spec:
    name: str
    requests: list            # list of (lq, start_pos); lk = start_pos + lq
    h_q: int
    h_kv: int
    d: int = 128
    page_size: int = 64
    layout: str = "shuffled"  # contiguous | shuffled | interleaved
    dtype: str = "bf16"       # bf16 | e4m3
    n_needles: int = 4
    logit_scale: float = 1.0
    config_id: int = 0

    @property
    def batch(self):
        return len(self.requests)

    @property
    def total_q(self):
        return sum(lq for lq, _ in self.requests)

    @property
    def total_k(self):
        return sum(lq + s for lq, s in self.requests)


@dataclass
class Case:
    spec: Spec
    q: np.ndarray             # [total_q, h_q, d] uint16 (bf16 bits) or uint8 (e4m3)
    k_cache: np.ndarray       # [num_pages, page_size, h_kv, d]
    v_cache: np.ndarray
    q_scale: np.ndarray       # float32 [h_q]  (ones for bf16)
    k_scale: np.ndarray       # float32 [h_kv]
    v_scale: np.ndarray
    block_table: np.ndarray   # int32 [batch, max_pages]; -1 = unused
    cu_seqlens_q: np.ndarray  # int32 [batch + 1]
    seqlens_k: np.ndarray     # int32 [batch]
    q_start_pos: np.ndarray   # int32 [batch]
    needles: list = field(default_factory=list)


def seed_of(config_id: int, request: int, kind: int) -> int:
    return 1000 * config_id + 10 * request + kind


# ----------------------------------------------------------------------------
# the workloads of the pages (restated as concrete shapes)
# ----------------------------------------------------------------------------

def config_spec(n: int, **over) -> Spec:
    """Workload n of the benchmark family (1: tiny; 2: Llama-3.1-8B layer at
    32K; 3: Qwen3-30B-A3B layer at 128K; 4: varlen continuous batch with a
    chunked prefill; 5: 256K)."""
    if n == 1:
        s = Spec("tiny-2k-g4", [(2048, 0)], 4, 1, page_size=64, layout="contiguous",
                 n_needles=2, config_id=1)
    elif n == 2:
        s = Spec("llama8b-32k", [(32768, 0)], 32, 8, page_size=64, layout="shuffled",
                 n_needles=4, config_id=2)
    elif n == 3:
        s = Spec("qwen30b-128k", [(131072, 0)], 32, 4, page_size=64, layout="shuffled",
                 n_needles=4, config_id=3)
    elif n == 4:
        reqs = [(2048, 0), (4096, 0), (8192, 40960), (16384, 0), (32768, 0), (65536, 0)]
        s = Spec("varlen-6req-chunk", reqs, 32, 8, page_size=64, layout="interleaved",
                 n_needles=4, config_id=4)
    elif n == 5:
        s = Spec("qwen30b-256k", [(262144, 0)], 32, 4, page_size=64, layout="shuffled",
                 n_needles=4, config_id=5)
    else:
        raise ValueError(f"no workload {n}")
    for k, v in over.items():
        setattr(s, k, v)
    return s


# ----------------------------------------------------------------------------
# rounding helpers (input formats only)
# ----------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 (already scaled into [-448, 448]) -> e4m3fn codes via torch's
    round-to-nearest-even conversion."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.clamp_(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


# ----------------------------------------------------------------------------
# generation
# ----------------------------------------------------------------------------

def _page_assignment(spec: Spec, n_pages_req):
    """Physical page id of every logical page, per request."""
    total = int(sum(n_pages_req))
    if spec.layout == "contiguous":
        ids, base = [], 0
        for n in n_pages_req:
            ids.append(np.arange(base, base + n, dtype=np.int32))
            base += n
        return ids, total
    if spec.layout == "interleaved":
        ids = [[] for _ in n_pages_req]
        nxt = 0
        for k in range(max(n_pages_req)):
            for r, n in enumerate(n_pages_req):
                if k < n:
                    ids[r].append(nxt)
                    nxt += 1
        return [np.asarray(x, dtype=np.int32) for x in ids], total
    if spec.layout == "shuffled":
        rng = np.random.Generator(np.random.Philox(seed_of(spec.config_id, 0, 4)))
        perm = rng.permutation(total).astype(np.int32)
        ids, base = [], 0
        for n in n_pages_req:
            ids.append(perm[base:base + n])
            base += n
        return ids, total
    raise ValueError(spec.layout)


def make_case(spec: Spec, threads: int | None = None) -> Case:
    B = BLOCK
    d, hq, hkv = spec.d, spec.h_q, spec.h_kv
    if hq % hkv:
        raise ValueError("h_q must be a multiple of h_kv")
    g = hq // hkv
    ps = spec.page_size
    nthreads = threads or _threads()

    lqs = [lq for lq, _ in spec.requests]
    starts = [s for _, s in spec.requests]
    lks = [lq + s for lq, s in spec.requests]
    n_pages_req = [-(-lk // ps) for lk in lks]
    page_ids, num_pages = _page_assignment(spec, n_pages_req)
    max_pages = max(n_pages_req)
    block_table = np.full((spec.batch, max_pages), -1, dtype=np.int32)
    for r, ids in enumerate(page_ids):
        block_table[r, :len(ids)] = ids

    cu = np.zeros(spec.batch + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lqs)
    total_q = int(cu[-1])

    # float32 staging, rounded per head in worker threads
    q32 = np.empty((total_q, hq, d), dtype=np.float32)
    k32 = np.empty((num_pages * ps, hkv, d), dtype=np.float32)
    v32 = np.empty((num_pages * ps, hkv, d), dtype=np.float32)
    k32[:] = 64.0
    v32[:] = 64.0
    needles = []

    pool = _cf.ThreadPoolExecutor(max_workers=nthreads)
    try:
        for r in range(spec.batch):
            lq, start, lk = lqs[r], starts[r], lks[r]
            nkb = -(-lk // B)
            qb0, qb1 = start // B, (lk - 1) // B       # absolute query blocks present
            shared = np.random.Generator(np.random.Philox(seed_of(spec.config_id, r, 3)))
            svec = shared.standard_normal((hkv, d))
            svec /= np.linalg.norm(svec, axis=1, keepdims=True)
            q_ss = np.random.SeedSequence(seed_of(spec.config_id, r, 0)).spawn(hq)
            k_ss = np.random.SeedSequence(seed_of(spec.config_id, r, 1)).spawn(hkv)
            v_ss = np.random.SeedSequence(seed_of(spec.config_id, r, 2)).spawn(hkv)
            pos_q = np.arange(start, lk)
            pos_k = np.arange(lk)
            qrows = slice(int(cu[r]), int(cu[r + 1]))
            # token slot of every key position in the paged pool
            pg = page_ids[r][pos_k // ps].astype(np.int64)
            slot = pg * ps + (pos_k % ps)

            uq = {}

            def gen_q(h):
                rng = np.random.Generator(np.random.Philox(q_ss[h]))
                u = rng.standard_normal((nkb, d))
                n = rng.standard_normal((lq, d))
                x = 0.6 * u[pos_q // B] + 0.8 * n + svec[h // g]
                q32[qrows, h, :] = x * spec.logit_scale
                return h, u

            for h, u in pool.map(gen_q, range(hq)):
                uq[h] = u

            # needles: key block j gets 2x the u of a later query block i of one
            # query head of the group (i outside the local window: i >= j + 4)
            uk_over = {}
            for h in range(hkv):
                for _ in range(spec.n_needles):
                    lo_i = max(qb0, 6)
                    if lo_i > qb1:
                        break
                    i = int(shared.integers(lo_i, qb1 + 1))
                    hi_j = min(i - 4, nkb - 5)
                    if hi_j < 2:
                        continue
                    j = int(shared.integers(2, hi_j + 1))
                    hsel = h * g + int(shared.integers(0, g))
                    uk_over[(h, j)] = 2.0 * uq[hsel][i]
                    needles.append(dict(request=r, kv_head=h, key_block=j,
                                        query_block=i, q_head=hsel))

            def gen_k(h):
                rng = np.random.Generator(np.random.Philox(k_ss[h]))
                u = rng.standard_normal((nkb, d))
                for (hh, j), val in uk_over.items():
                    if hh == h:
                        u[j] = val
                n = rng.standard_normal((lk, d))
                x = 0.6 * u[pos_k // B] + 0.8 * n
                x[:SINK_BOOST_TOKENS] += 3.0 * svec[h]
                k32[slot, h, :] = x

            def gen_v(h):
                rng = np.random.Generator(np.random.Philox(v_ss[h]))
                v32[slot, h, :] = rng.standard_normal((lk, d))

            list(pool.map(gen_k, range(hkv)))
            list(pool.map(gen_v, range(hkv)))
    finally:
        pool.shutdown()

    if spec.dtype == "bf16":
        qc = _round_bf16_threaded(q32, nthreads)
        kc = _round_bf16_threaded(k32, nthreads)
        vc = _round_bf16_threaded(v32, nthreads)
        kc = kc.reshape(num_pages, ps, hkv, d)
        vc = vc.reshape(num_pages, ps, hkv, d)
        one = lambda n: np.ones(n, dtype=np.float32)
        qs, ks, vs = one(hq), one(hkv), one(hkv)
    elif spec.dtype == "e4m3":
        qc, qs = _quant_e4m3_per_head(q32, valid=None)
        valid = _valid_slots(block_table, lks, ps, num_pages)
        kc, ks = _quant_e4m3_per_head(k32, valid)
        vc, vs = _quant_e4m3_per_head(v32, valid)
        kc = kc.reshape(num_pages, ps, hkv, d)
        vc = vc.reshape(num_pages, ps, hkv, d)
    else:
        raise ValueError(spec.dtype)

    return Case(spec, qc, kc, vc, qs, ks, vs, block_table, cu,
                np.asarray(lks, dtype=np.int32), np.asarray(starts, dtype=np.int32),
                needles)


def _round_bf16_threaded(x: np.ndarray, nthreads: int) -> np.ndarray:
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    n = flat.size
    step = max(1 << 20, -(-n // (4 * nthreads)))
    chunks = [(i, min(n, i + step)) for i in range(0, n, step)]

    def work(c):
        a, b = c
        out[a:b] = to_bf16_bits(flat[a:b])

    with _cf.ThreadPoolExecutor(max_workers=nthreads) as ex:
        list(ex.map(work, chunks))
    return out.reshape(x.shape)


def _valid_slots(block_table, lks, ps, num_pages):
    valid = np.zeros(num_pages * ps, dtype=bool)
    for r, lk in enumerate(lks):
        pos = np.arange(lk)
        valid[block_table[r, pos // ps].astype(np.int64) * ps + pos % ps] = True
    return valid


def _quant_e4m3_per_head(x: np.ndarray, valid):
    """x: [tokens, heads, d] float32 -> (codes uint8, scale float32[heads]).
    Scale = amax over the head's real tokens / 448."""
    heads = x.shape[1]
    scales = np.empty(heads, dtype=np.float32)
    codes = np.empty(x.shape, dtype=np.uint8)
    for h in range(heads):
        xh = x[:, h, :]
        src = xh if valid is None else xh[valid]
        amax = float(np.abs(src).max()) if src.size else 1.0
        sc = np.float32(amax / 448.0 if amax > 0 else 1.0)
        scales[h] = sc
        y = xh / sc
        if valid is not None:
            y = y.copy()
            y[~valid] = 448.0
        codes[:, h, :] = to_e4m3_codes(y)
    return codes, scales


# ----------------------------------------------------------------------------
# random block-keep patterns (for testing the attention stage on its own)
# ----------------------------------------------------------------------------

def random_keep_lists(case: Case, density: float, seed: int, block: int = BLOCK):
    """Per (request, query block, kv head) row, an ascending list of kept key
    blocks: the row's own (diagonal) block plus each earlier block with
    probability ``density``.  Rows are ordered (request, query block, kv head)."""
    rng = np.random.Generator(np.random.Philox(seed))
    rows = []
    for r, (lq, start) in enumerate(case.spec.requests):
        nqb = -(-lq // block)
        i0 = start // block
        for i in range(nqb):
            ia = i0 + i
            for _h in range(case.spec.h_kv):
                pick = np.nonzero(rng.random(ia) < density)[0]
                rows.append(np.concatenate([pick, [ia]]).astype(np.int32))
    return rows
