"""fp_sparse_attn_noalloc: the sparse-attention entry point for callers that
cannot allocate device memory (a plugin whose host framework owns all device
memory, a serving loop held to a fixed memory budget).  It must give the
result of fp_sparse_attn -- which takes a caller-allocated workspace -- from
the library's built-in scratch array, call after call.

This file is collected last on purpose: its GPU test uses the library's
process-wide scratch array, and if it fails, a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

from block_sparse_long_fp_gb300 import synth

MAX_ABS, MEAN_ABS = 2e-2, 2e-3      # the bf16 tolerance the parity tests use


def _problem_too_big_for_the_scratch(fp):
    """A 256K request with 8 kv heads: the bf16 block means alone fill 8 MiB."""
    L = 262144
    cu = np.array([0, L], np.int32)
    lk = np.array([L], np.int32)
    st = np.array([0], np.int32)
    pr = fp.FpProblem()
    pr.batch, pr.h_q, pr.h_kv, pr.d, pr.dtype = 1, 16, 8, 128, fp.FP_BF16
    pr.cu_seqlens_q, pr.seqlens_k, pr.q_start_pos = cu.ctypes.data, lk.ctypes.data, st.ctypes.data
    pr.q = 256
    pr.q_stride_tok, pr.q_stride_head = 16 * 128, 128
    pr.k_cache = pr.v_cache = 512
    pr.page_size, pr.num_pages = 64, L // 64
    pr.block_table = 1024
    pr.max_pages_per_seq = L // 64
    return pr, (cu, lk, st)


def test_noalloc_rejects_problems_beyond_its_scratch():
    """The size check happens before the GPU is touched (runs without one)."""
    from block_sparse_long_fp_gb300 import build, fprefill
    build.build()
    pr, keep = _problem_too_big_for_the_scratch(fprefill)
    prm = fprefill.default_params()
    L = fprefill.lib()
    need = L.fp_attn_workspace_size(ctypes.byref(pr), ctypes.byref(prm))
    limit = 8 << 20
    assert need > limit
    d = ctypes.c_void_p(4096)
    s = L.fp_sparse_attn_noalloc(ctypes.byref(pr), ctypes.byref(prm), d, d, d, d, d, None, None, None)
    assert s == fprefill.FP_ERR_WORKSPACE
    # an argument error is reported as such, not as a size problem
    pr.h_q = 15
    s = L.fp_sparse_attn_noalloc(ctypes.byref(pr), ctypes.byref(prm), d, d, d, d, d, None, None, None)
    assert s == fprefill.FP_ERR_INVALID


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_fp_gb300 import build, fprefill
    build.build()
    specs = [
        synth.Spec("noalloc-a", [(1536, 0), (700, 256)], 8, 2, page_size=32, layout="shuffled",
                   n_needles=2, logit_scale=8.0, config_id=81),
        synth.Spec("noalloc-b", [(3000, 0)], 4, 1, page_size=64, layout="interleaved",
                   n_needles=2, logit_scale=8.0, config_id=82),
    ]
    for call, spec in enumerate(specs):         # two calls in a row, different problems
        case = synth.make_case(spec)
        layer = fprefill.layer_from_case(case)
        k_mean, v_mean, score = layer.discover()
        row_ptr, col_idx, _ = layer.select(score)
        ref, ref_lse = layer.sparse_attn(row_ptr, col_idx, k_mean, v_mean)
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device=ref.device)
        layer.sparse_attn_noalloc(row_ptr, col_idx, k_mean, v_mean, out, lse, status)
        torch.cuda.synchronize()
        assert int(status.item()) == fprefill.FP_OK, f"call {call}: device status {int(status.item())}"
        err = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all(), f"call {call}"
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, f"call {call}"
        assert (lse - ref_lse).abs().max().item() <= 2e-2, f"call {call}"


@pytest.mark.gpu
def test_noalloc_reports_a_device_error_and_the_next_call_starts_clean():
    """The scratch array keeps the last call's contents, status word included.
    A call whose index holds a block past the diagonal records
    FP_ERR_DEVICE_BOUNDS, which status_dev_opt must report; the next call,
    on a good index, must start from a clear status (FP_OK) and give
    fp_sparse_attn's result."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_fp_gb300 import build, fprefill
    build.build()
    spec = synth.Spec("noalloc-err", [(512, 0), (300, 128)], 4, 2, page_size=64, layout="shuffled",
                      n_needles=1, logit_scale=6.0, config_id=83)
    case = synth.make_case(spec)
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, _ = layer.select(score)
    ref, ref_lse = layer.sparse_attn(row_ptr, col_idx, k_mean, v_mean)
    torch.cuda.synchronize()
    assert layer.device_status() == fprefill.FP_OK
    bad = col_idx.clone()
    rp = row_ptr.cpu().numpy()
    bad[int(rp[2 * spec.h_kv])] = 3             # row (I = 2, kv head 0): a block after its diagonal
    out = torch.empty_like(ref)
    lse = torch.empty_like(ref_lse)
    status = torch.full((1,), -1, dtype=torch.int32, device=ref.device)
    layer.sparse_attn_noalloc(row_ptr, bad, k_mean, v_mean, out, lse, status)
    torch.cuda.synchronize()
    assert int(status.item()) == fprefill.FP_ERR_DEVICE_BOUNDS
    status.fill_(-1)
    out.fill_(float("nan"))
    layer.sparse_attn_noalloc(row_ptr, col_idx, k_mean, v_mean, out, lse, status)
    torch.cuda.synchronize()
    assert int(status.item()) == fprefill.FP_OK
    err = (out.float() - ref.float()).abs()
    assert torch.isfinite(out.float()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    assert (lse - ref_lse).abs().max().item() <= 2e-2
