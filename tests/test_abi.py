"""The C ABI without a GPU: the library loads, exports every declared entry
point, and its host-side logic (sizes, layouts, argument checks) is right.
No call here reaches a kernel launch."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fp():
    from block_sparse_long_fp_gb300 import build, fprefill
    build.build()
    return fprefill


def declared_functions():
    txt = open(os.path.join(ROOT, "include", "fprefill.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(fp_[a-z_]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(fp):
    names = declared_functions()
    assert len(names) >= 15
    L = fp.lib()
    for n in names:
        assert hasattr(L, n), n


def problem(fp, reqs, h_q=8, h_kv=2, page=64, extra_pages=0):
    cu = np.zeros(len(reqs) + 1, np.int32)
    cu[1:] = np.cumsum([lq for lq, _ in reqs])
    lk = np.array([lq + s for lq, s in reqs], np.int32)
    st = np.array([s for _, s in reqs], np.int32)
    pr = fp.FpProblem()
    pr.batch, pr.h_q, pr.h_kv, pr.d, pr.dtype = len(reqs), h_q, h_kv, 128, fp.FP_BF16
    pr.cu_seqlens_q, pr.seqlens_k, pr.q_start_pos = cu.ctypes.data, lk.ctypes.data, st.ctypes.data
    pr.q = 256
    pr.q_stride_tok, pr.q_stride_head = h_q * 128, 128
    pr.k_cache = pr.v_cache = 512
    pr.page_size = page
    pr.num_pages = int(sum(-(-x // page) for x in lk)) + extra_pages
    pr.block_table = 1024
    pr.max_pages_per_seq = int(max(-(-x // page) for x in lk))
    return pr, (cu, lk, st)


def test_sizes_match_the_documented_layout(fp, oracle_mod):
    reqs = [(300, 0), (1000, 0), (256, 512), (1, 128)]
    pr, keep = problem(fp, reqs)
    prm = fp.default_params()
    L = fp.lib()
    rows = sum(-(-lq // 128) for lq, _ in reqs) * 2
    assert L.fp_num_rows(ctypes.byref(pr), ctypes.byref(prm)) == rows
    assert L.fp_num_key_blocks(ctypes.byref(pr), ctypes.byref(prm)) == sum(-(-(lq + s) // 128) for lq, s in reqs)
    _, total = oracle_mod.score_row_offsets(reqs, 2, 128)
    assert L.fp_score_size(ctypes.byref(pr), ctypes.byref(prm)) == total
    assert L.fp_total_q(ctypes.byref(pr)) == 1557
    assert L.fp_attn_workspace_size(ctypes.byref(pr), ctypes.byref(prm)) >= 256 + rows * 4


def test_score_offsets_follow_the_documented_layout(fp, oracle_mod):
    """fp_score_offsets (host only) against the oracle's own restatement of
    the score-map layout, on a varlen batch with chunks and a one-token request."""
    reqs = [(300, 0), (1000, 0), (256, 512), (1, 128), (640, 0)]
    pr, keep = problem(fp, reqs, h_q=8, h_kv=2)
    prm = fp.default_params()
    L = fp.lib()
    rows = int(L.fp_num_rows(ctypes.byref(pr), ctypes.byref(prm)))
    offs = np.full(rows + 1, -7, np.int64)
    assert L.fp_score_offsets(ctypes.byref(pr), ctypes.byref(prm), offs.ctypes.data, offs.size) == rows + 1
    ref, total = oracle_mod.score_row_offsets(reqs, 2, 128)
    assert np.array_equal(offs[:-1], np.concatenate([o.reshape(-1) for o in ref]))
    assert offs[-1] == total == L.fp_score_size(ctypes.byref(pr), ctypes.byref(prm))
    # too small an array, or a null one, is refused without writing
    small = np.full(rows, -7, np.int64)
    assert L.fp_score_offsets(ctypes.byref(pr), ctypes.byref(prm), small.ctypes.data, small.size) == -1
    assert np.all(small == -7)
    assert L.fp_score_offsets(ctypes.byref(pr), ctypes.byref(prm), None, rows + 1) == -1


def test_default_params_are_the_pages_configuration(fp):
    p = fp.default_params()
    assert (p.block, p.sink_tokens, p.local_tokens, p.mean_correction) == (128, 256, 512, 1)
    assert abs(p.alpha - 0.1) < 1e-7 and p.softmax_scale == 0.0
    assert p.p_terms == 1                       # the pages' single e4m3 term of P


def test_p_terms_out_of_range_is_refused(fp):
    pr, keep = problem(fp, [(300, 0), (256, 512)])
    L = fp.lib()
    for bad in (-1, 3):
        prm = fp.default_params(p_terms=bad)
        assert L.fp_num_rows(ctypes.byref(pr), ctypes.byref(prm)) == -1
        assert L.fp_attn_workspace_size(ctypes.byref(pr), ctypes.byref(prm)) == 0


@pytest.mark.parametrize("mutate,code", [
    (lambda pr, a: setattr(pr, "d", 64), 2),                     # d != 128 unsupported
    (lambda pr, a: setattr(pr, "h_q", 7), 1),                    # h_q not a multiple of h_kv
    (lambda pr, a: a[1].__setitem__(0, 999), 1),                 # seqlens_k != start + lq
    (lambda pr, a: a[2].__setitem__(0, 64), 1),                  # start not a multiple of 128
    (lambda pr, a: setattr(pr, "page_size", 48), 2),             # page size neither divides nor is a multiple
    (lambda pr, a: setattr(pr, "max_pages_per_seq", 1), 1),      # block table too narrow
    (lambda pr, a: setattr(pr, "k_cache", 520), 1),              # misaligned cache pointer
    (lambda pr, a: setattr(pr, "q_stride_head", 100), 1),        # stride not 16-byte multiple
    (lambda pr, a: setattr(pr, "batch", 0), 1),
    (lambda pr, a: setattr(pr, "batch", 129), 2),
])
def test_argument_errors_are_returned_before_any_launch(fp, mutate, code):
    pr, arrs = problem(fp, [(300, 0), (200, 0)])
    mutate(pr, arrs)
    prm = fp.default_params()
    L = fp.lib()
    dummy = ctypes.c_void_p(4096)
    s = L.fp_discover(ctypes.byref(pr), ctypes.byref(prm), dummy, dummy, dummy, dummy, 1 << 20, None)
    assert s == code
    s = L.fp_dense_attn(ctypes.byref(pr), ctypes.byref(prm), dummy, None, dummy, 1 << 30, None)
    assert s == code


def test_workspace_and_capacity_checks(fp):
    pr, keep = problem(fp, [(300, 0)])
    prm = fp.default_params()
    L = fp.lib()
    d = ctypes.c_void_p(4096)
    assert L.fp_discover(ctypes.byref(pr), ctypes.byref(prm), d, d, d, d, 16, None) == fp.FP_ERR_WORKSPACE
    assert L.fp_dense_attn(ctypes.byref(pr), ctypes.byref(prm), d, None, d, 16, None) == fp.FP_ERR_WORKSPACE
    size = L.fp_score_size(ctypes.byref(pr), ctypes.byref(prm))
    assert L.fp_select(ctypes.byref(pr), ctypes.byref(prm), d, d, d, size - 1, d, None, d, 1 << 20,
                       None) == fp.FP_ERR_INVALID
    prm.block = 64
    assert L.fp_dense_attn(ctypes.byref(pr), ctypes.byref(prm), d, None, d, 1 << 30, None) == fp.FP_ERR_UNSUPPORTED


def test_odd_group_and_fp8_attention_are_reported_unsupported(fp):
    pr, keep = problem(fp, [(300, 0)], h_q=6, h_kv=2)
    prm = fp.default_params()
    L = fp.lib()
    d = ctypes.c_void_p(4096)
    assert L.fp_dense_attn(ctypes.byref(pr), ctypes.byref(prm), d, None, d, 1 << 30, None) == fp.FP_ERR_UNSUPPORTED


def test_value_cache_layout_is_checked_on_the_host(fp):
    prm = fp.default_params()
    L = fp.lib()
    d = ctypes.c_void_p(4096)
    pr, keep = problem(fp, [(300, 0)], page=64)
    pr.v_layout = 2
    assert L.fp_dense_attn(ctypes.byref(pr), ctypes.byref(prm), d, None, d, 1 << 30, None) == fp.FP_ERR_INVALID
    pr, keep = problem(fp, [(300, 0)], page=32)
    pr.v_layout = fp.FP_V_DIM_MAJOR            # bf16 needs pages of a multiple of 64 tokens
    assert L.fp_dense_attn(ctypes.byref(pr), ctypes.byref(prm), d, None, d, 1 << 30, None) == fp.FP_ERR_UNSUPPORTED
    pr, keep = problem(fp, [(300, 0)], page=64)
    pr.dtype = fp.FP_E4M3                      # e4m3 needs a multiple of 128
    pr.q_scale = pr.k_scale = pr.v_scale = 4096
    pr.v_layout = fp.FP_V_DIM_MAJOR
    assert L.fp_dense_attn(ctypes.byref(pr), ctypes.byref(prm), d, None, d, 1 << 30, None) == fp.FP_ERR_UNSUPPORTED


def test_wait_timeout_check_refuses_bad_arguments_on_the_host(fp):
    L = fp.lib()
    d = ctypes.c_void_p(4096)
    assert L.fp_check_wait_timeout(None, 1000, None) == fp.FP_ERR_INVALID
    assert L.fp_check_wait_timeout(d, 0, None) == fp.FP_ERR_INVALID
    assert L.fp_check_wait_timeout(d, 10_000_000_001, None) == fp.FP_ERR_INVALID


def test_status_strings(fp):
    for s in range(7):
        assert fp.status_string(s) and fp.status_string(s) != "unknown status"
