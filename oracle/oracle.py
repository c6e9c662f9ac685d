"""Python side of the float64 oracle (test infrastructure only).

The arithmetic lives in ``oracle.c`` (compiled here with gcc, OpenMP); this
module decodes the input formats to float64, gathers paged KV into contiguous
positions, lays out the score map and CSR exactly as the library's header
documents them, and calls the C routines.  It never imports the CUDA library.

Parity status of each function (what pins it; see tests/test_oracle_pins.py):
  pool         pinned: numpy mean; constant-block and linearity checks.
  score_rows   pinned: hand-derived closed form (tests/golden/score_tiny.json),
               per-query shift invariance, head/query permutation invariance,
               row maximum exactly 1.
  score_rows_head_union   pinned: g = 1 reduces it to score_rows, head-order
               invariance, each head's own normalised row bounded by it, max 1.
  select_row   pinned: brute-force rule check, sink/local/causal invariants;
               top-k / top-p: count, dominance, tie order, minimal mass, limits.
  attn_rows    pinned: alpha=0 equals direct dense causal softmax; exact mean
               correction for constant-key blocks; token-level brute force
               with appended "mean tokens" at L <= 512; V-linearity.
  Block-score values at full size with realistic inputs have no printed
  worked example: beyond the pins above they are "parity unpinned".
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, OpenMP)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(src):
        return _LIB
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        L = ctypes.c_long
        I = ctypes.c_int
        D = ctypes.c_double
        _lib.oracle_pool.argtypes = [P, L, I, I, I, P]
        _lib.oracle_score_rows.argtypes = [P, L, L, I, I, I, I, D, P, L, P, L, P, P]
        _lib.oracle_select_row.argtypes = [P, L, D, I, I, I, P, P]
        _lib.oracle_select_row_rule.argtypes = [P, L, I, D, I, D, I, I, I, P, P]
        _lib.oracle_attn_rows.argtypes = [P, L, L, I, I, I, I, D, P, P, L, P, P, L, P, I,
                                          P, P, L, P, P]
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int):
    """Number of OpenMP threads the oracle uses (call before the first use)."""
    os.environ["OMP_NUM_THREADS"] = str(int(n))


# ----------------------------------------------------------------------------
# input decoding (formats only)
# ----------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """e4m3fn: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is
    subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities."""
    c = codes.astype(np.int64)
    sgn = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return sgn * val


def decode(case_arr: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return decode_bf16(case_arr)
    if dtype == "e4m3":
        return decode_e4m3(case_arr)
    raise ValueError(dtype)


def request_q(case, r: int) -> np.ndarray:
    """Query rows of request r as float64 [lq, hq, d] (scale applied)."""
    a, b = int(case.cu_seqlens_q[r]), int(case.cu_seqlens_q[r + 1])
    x = decode(case.q[a:b], case.spec.dtype)
    return x * case.q_scale.astype(np.float64)[None, :, None]


def request_kv(case, r: int):
    """Gather request r's K and V from the paged pool (physical slot =
    page_table[t // page] * page + t % page) as float64 [lk, hkv, d]."""
    lk = int(case.seqlens_k[r])
    ps = case.k_cache.shape[1]
    t = np.arange(lk)
    pages = case.block_table[r, t // ps].astype(np.int64)
    kc = case.k_cache[pages, t % ps]
    vc = case.v_cache[pages, t % ps]
    k = decode(kc, case.spec.dtype) * case.k_scale.astype(np.float64)[None, :, None]
    v = decode(vc, case.spec.dtype) * case.v_scale.astype(np.float64)[None, :, None]
    return k, v


# ----------------------------------------------------------------------------
# the method's steps
# ----------------------------------------------------------------------------

def pool(x: np.ndarray, B: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    lk, h, d = x.shape
    nkb = -(-lk // B)
    out = np.empty((nkb, h, d), dtype=np.float64)
    _load().oracle_pool(_p(x), lk, h, d, B, _p(out))
    return out


def score_rows(q, start, hkv, B, scale, kbar, rows):
    """Score rows (i_local*hkv + h) of one request; returns a list of arrays
    (row of query block I = start//B + i_local has I+1 entries)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    kbar = np.ascontiguousarray(kbar, dtype=np.float64)
    lq, hq, d = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    lens = np.array([start // B + r // hkv + 1 for r in rows], dtype=np.int64)
    off = np.zeros(len(rows), dtype=np.int64)
    if len(rows):
        off[1:] = np.cumsum(lens)[:-1]
    out = np.empty(int(lens.sum()), dtype=np.float64)
    _load().oracle_score_rows(_p(q), lq, start, hq, hkv, d, B, scale, _p(kbar), kbar.shape[0],
                              _p(rows), len(rows), _p(off), _p(out))
    return [out[o:o + n] for o, n in zip(off, lens)]


def score_rows_head_union(q, start, hkv, B, scale, kbar, rows):
    """The union-of-heads reading of the score rows (V1 summary 3.1 applied to
    each query head alone): for row (i_local, h), each query head h' of the
    group scores the block with its own B queries and its row is normalised to
    a maximum of 1; the row is the maximum over the group's heads."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    lq, hq, d = q.shape
    g = hq // hkv
    out = []
    for row in rows:
        il, h = divmod(int(row), hkv)
        per_head = [score_rows(q[:, hh:hh + 1, :], start, 1, B, scale, kbar[:, h:h + 1, :], [il])[0]
                    for hh in range(h * g, (h + 1) * g)]
        out.append(np.max(np.stack(per_head), axis=0))
    return out


def select_row(score_row: np.ndarray, I: int, alpha: float, B: int, sink: int, local: int, rule: int = 0,
               top_k: int = 0, top_p: float = 0.0):
    """keep / flag masks of one score row: rule 0 the max threshold, 1 top-k,
    2 top-p (the last two as ablations)."""
    s = np.ascontiguousarray(score_row, dtype=np.float64)
    keep = np.zeros(I + 1, dtype=np.uint8)
    flag = np.zeros(I + 1, dtype=np.uint8)
    if rule == 0:
        _load().oracle_select_row(_p(s), I, alpha, B, sink, local, _p(keep), _p(flag))
    else:
        _load().oracle_select_row_rule(_p(s), I, rule, alpha, top_k, top_p, B, sink, local, _p(keep), _p(flag))
    return keep.astype(bool), flag.astype(bool)


def attn_rows(q, start, k, v, kbar, vbar, B, scale, keep, mean_corr, qi, qh):
    """O and LSE for query rows (qi[k] local index, qh[k] head).  keep:
    uint8 [nqb, hkv, nkb] or None (dense causal)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    kbar = np.ascontiguousarray(kbar, dtype=np.float64)
    vbar = np.ascontiguousarray(vbar, dtype=np.float64)
    lq, hq, d = q.shape
    hkv = k.shape[1]
    qi = np.ascontiguousarray(qi, dtype=np.int64)
    qh = np.ascontiguousarray(qh, dtype=np.int32)
    n = len(qi)
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    kp = None
    if keep is not None:
        keep = np.ascontiguousarray(keep, dtype=np.uint8)
        kp = _p(keep)
    _load().oracle_attn_rows(_p(q), lq, start, hq, hkv, d, B, scale, _p(k), _p(v), k.shape[0],
                             _p(kbar), _p(vbar), kbar.shape[0], kp, int(bool(mean_corr)),
                             _p(qi), _p(qh), n, _p(o), _p(lse))
    return o, lse


# ----------------------------------------------------------------------------
# layouts shared with the library's documented interface (formats, restated)
# ----------------------------------------------------------------------------

def score_row_offsets(requests, hkv: int, B: int):
    """Offsets of every score row in the flat score map, rows ordered
    (request, query block, kv head); row (I) has I+1 entries.  Returns
    (list of per-request offset arrays [nqb, hkv], total length)."""
    offs, pos = [], 0
    for lq, start in requests:
        nqb = -(-lq // B)
        i0 = start // B
        o = np.zeros((nqb, hkv), dtype=np.int64)
        for i in range(nqb):
            for h in range(hkv):
                o[i, h] = pos
                pos += i0 + i + 1
        offs.append(o)
    return offs, pos


def csr_from_keep(keep_rows):
    """keep_rows: list of boolean arrays in row order -> (row_ptr, col_idx)."""
    counts = np.array([int(np.count_nonzero(k)) for k in keep_rows], dtype=np.int64)
    row_ptr = np.zeros(len(keep_rows) + 1, dtype=np.int32)
    row_ptr[1:] = np.cumsum(counts)
    col_idx = np.concatenate([np.nonzero(k)[0] for k in keep_rows]).astype(np.int32) \
        if keep_rows else np.zeros(0, dtype=np.int32)
    return row_ptr, col_idx


def discover_and_select(case, B=128, sink=256, local=512, alpha=0.1, scale=None,
                        requests_subset=None, row_subset=None, rule=0, top_k=0, top_p=0.0, head_union=False):
    """Steps 1-3 for every request (or a subset): block means, score rows,
    keep / flag masks.  Returns a dict with per-request results."""
    spec = case.spec
    d, hkv = spec.d, spec.h_kv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    res = []
    reqs = range(spec.batch) if requests_subset is None else requests_subset
    for r in reqs:
        lq, start = spec.requests[r]
        q = request_q(case, r)
        k, v = request_kv(case, r)
        kbar, vbar = pool(k, B), pool(v, B)
        nqb = -(-lq // B)
        rows = np.arange(nqb * hkv) if row_subset is None else np.asarray(row_subset(r, nqb, hkv))
        srows = (score_rows_head_union if head_union else score_rows)(q, start, hkv, B, scale, kbar, rows)
        keep = np.zeros((nqb, hkv, kbar.shape[0]), dtype=np.uint8)
        flag = np.zeros((nqb, hkv, kbar.shape[0]), dtype=np.uint8)
        have = np.zeros((nqb, hkv), dtype=bool)
        for row, s in zip(rows, srows):
            i, h = divmod(int(row), hkv)
            I = start // B + i
            kp, fl = select_row(s, I, alpha, B, sink, local, rule, top_k, top_p)
            keep[i, h, :I + 1] = kp
            flag[i, h, :I + 1] = fl
            have[i, h] = True
        res.append(dict(request=r, q=q, k=k, v=v, kbar=kbar, vbar=vbar, rows=rows,
                        score=srows, keep=keep, flag=flag, have=have, start=start))
    return res
