"""Split-KV sizing on the host (no GPU): the attention workspace holds the
fp32 partial outputs and LSEs of every part, the automatic choice splits only
problems with too few work units, and out-of-range requests are refused."""
import ctypes

import numpy as np
import pytest


def _problem(fp, requests, h_q, h_kv):
    lq = [q for q, _ in requests]
    cu = np.zeros(len(requests) + 1, np.int32)
    cu[1:] = np.cumsum(lq)
    st = np.array([s for _, s in requests], np.int32)
    lk = st + np.array(lq, np.int32)
    pr = fp.FpProblem()
    pr.batch, pr.h_q, pr.h_kv, pr.d, pr.dtype = len(requests), h_q, h_kv, 128, fp.FP_BF16
    pr.cu_seqlens_q, pr.seqlens_k, pr.q_start_pos = cu.ctypes.data, lk.ctypes.data, st.ctypes.data
    pr.q = 256
    pr.q_stride_tok, pr.q_stride_head = h_q * 128, 128
    pr.k_cache = pr.v_cache = 512
    pr.page_size = 64
    pr.num_pages = int(lk.sum() // 64 + len(requests))
    pr.block_table = 1024
    pr.max_pages_per_seq = int(lk.max() // 64 + 1)
    return pr, (cu, st, lk), int(cu[-1])


@pytest.fixture(scope="module")
def fp():
    from block_sparse_long_fp_gb300 import build, fprefill
    build.build()
    return fprefill


def _ws(fp, pr, splits):
    prm = fp.default_params(kv_splits=splits)
    return int(fp.lib().fp_attn_workspace_size(ctypes.byref(pr), ctypes.byref(prm)))


def test_workspace_holds_the_partials_of_every_part(fp):
    pr, keep, total_q = _problem(fp, [(1536, 0), (700, 256)], 8, 2)
    one, three = _ws(fp, pr, 1), _ws(fp, pr, 3)
    assert one > 0 and three > one
    # fp32 partial O [3, total_q, 8, 128] and LSE [3, 8, total_q], each rounded up to 256 bytes
    assert three - one >= 3 * total_q * 8 * 128 * 4 + 3 * 8 * total_q * 4


def _splits(fp, pr, splits):
    prm = fp.default_params(kv_splits=splits)
    return int(fp.lib().fp_attn_kv_splits(ctypes.byref(pr), ctypes.byref(prm)))


def test_automatic_choice_splits_only_short_work_lists(fp):
    # a 512-query chunk at the end of a 32K context: 4 blocks x 2 kv heads x 2 pairs = 16
    # units; 9 parts make 144 units, one wave on 152 SMs (1/9 of a unit time)
    chunk, keep, _ = _problem(fp, [(512, 32768)], 8, 2)
    assert _splits(fp, chunk, 0) == 9
    assert _splits(fp, chunk, 1) == 1 and _splits(fp, chunk, 7) == 7
    assert _ws(fp, chunk, 0) > _ws(fp, chunk, 1)
    # the 128K layer has 16384 units: never split automatically
    big, keep2, _ = _problem(fp, [(131072, 0)], 32, 4)
    assert _splits(fp, big, 0) == 1
    assert _ws(fp, big, 0) == _ws(fp, big, 1)
    # 25 blocks x 4 kv heads x 4 pairs = 400 units: 3 waves, the last with 96 units;
    # three parts make 1200 units in 8 waves of a third (2.67 unit times instead of 3)
    mid, keep4, _ = _problem(fp, [(128 * 25, 32768)], 32, 4)
    assert _splits(fp, mid, 0) == 3
    # short rows are not worth splitting (fewer than ~16 terms per part)
    small, keep3, _ = _problem(fp, [(640, 0)], 4, 1)
    assert _ws(fp, small, 0) == _ws(fp, small, 1)


def test_split_count_out_of_range_is_refused(fp):
    pr, keep, _ = _problem(fp, [(1536, 0)], 8, 2)
    assert _ws(fp, pr, 32) > 0
    assert _ws(fp, pr, 33) == 0
    assert _ws(fp, pr, -1) == 0
    assert _splits(fp, pr, 33) == -1
