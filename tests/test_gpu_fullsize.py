"""Parity at the benchmark's full sizes, in the configuration bench.py times:
the same seeded workloads (128K layer in bf16 and e4m3, the sparse regime,
the varlen batch with a chunked prefill, 256K), the same C-ABI calls and
tensor layouts.  The oracle computes sampled score rows, their index rows and
sampled output rows one by one (only the sampled query blocks are decoded)."""
import math

import numpy as np
import pytest

from block_sparse_long_fp_gb300 import synth
from parity_util import BF16_MAX_ABS, BF16_MEAN_ABS, FP8_LSE_ABS, FP8_MAX_ABS, SCORE_ABS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_fp_gb300 import build
    build.build()


def sampled_parity(spec, alpha=0.1, mean_corr=True, rows_per_request=3, queries_per_row=24, max_abs=BF16_MAX_ABS,
                   mean_abs=BF16_MEAN_ABS, lse_abs=2e-2, seed=0):
    import torch
    import oracle
    from block_sparse_long_fp_gb300 import fprefill
    case = synth.make_case(spec)
    prm = fprefill.default_params(alpha=alpha, mean_correction=int(mean_corr))
    layer = fprefill.layer_from_case(case, params=prm)
    # one pass of the path, the three calls of the benchmark step
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    out, lse = layer.sparse_attn(row_ptr, col_idx, k_mean, v_mean)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    score_h = score.cpu().numpy()
    rp, ci = row_ptr.cpu().numpy(), col_idx.cpu().numpy()
    km, vm = k_mean.cpu().numpy(), v_mean.cpu().numpy()
    hkv, g = spec.h_kv, spec.h_q // spec.h_kv
    scale = 1 / math.sqrt(spec.d)
    offs, _ = oracle.score_row_offsets(spec.requests, hkv, 128)
    rng = np.random.default_rng(seed)
    errs, lerrs, kept_total, causal_total = [], [], 0, 0
    row_base = kb_base = 0
    for r, (lq, start) in enumerate(spec.requests):
        nqb = -(-lq // 128)
        k, v = oracle.request_kv(case, r)
        kbar, vbar = oracle.pool(k, 128), oracle.pool(v, 128)
        nkb = kbar.shape[0]
        np.testing.assert_allclose(km[kb_base:kb_base + nkb], kbar, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(vm[kb_base:kb_base + nkb], vbar, rtol=1e-5, atol=1e-6)
        rows = {(nqb - 1, hkv - 1), (0, 0)}
        while len(rows) < min(rows_per_request, nqb * hkv):
            rows.add((int(rng.integers(0, nqb)), int(rng.integers(0, hkv))))
        for i, h in sorted(rows):
            I = start // 128 + i
            q0 = int(case.cu_seqlens_q[r]) + i * 128
            q1 = int(case.cu_seqlens_q[r]) + min(lq, (i + 1) * 128)
            qblk = oracle.decode(case.q[q0:q1], spec.dtype) * case.q_scale.astype(np.float64)[None, :, None]
            s_ref = oracle.score_rows(qblk, start + i * 128, hkv, 128, scale, kbar, [h])[0]
            o = offs[r][i, h]
            assert np.abs(score_h[o:o + I + 1] - s_ref).max() <= SCORE_ABS, (r, i, h)
            keep_ref, flag = oracle.select_row(s_ref, I, alpha, 128, 256, 512)
            grow = row_base + i * hkv + h
            cols = ci[rp[grow]:rp[grow + 1]]
            assert np.all(np.diff(cols) > 0)
            kept = np.zeros(I + 1, bool)
            kept[cols] = True
            assert not np.any((kept != keep_ref) & ~flag), (r, i, h)
            kept_total += int(keep_ref.sum())
            causal_total += I + 1
            # the attention on the blocks the GPU kept (they equal the oracle's
            # outside the flagged near-threshold band, checked just above)
            keep = np.zeros((1, hkv, nkb), np.uint8)
            keep[0, h, :I + 1] = kept
            nrow = q1 - q0
            qi = rng.integers(0, nrow, queries_per_row)
            qi[0] = nrow - 1
            qh = h * g + rng.integers(0, g, queries_per_row)
            o_ref, l_ref = oracle.attn_rows(qblk, start + i * 128, k, v, kbar, vbar, 128, scale, keep, mean_corr,
                                            qi, qh)
            tok = torch.as_tensor(q0 + qi, device=out.device)
            hd = torch.as_tensor(qh, device=out.device)
            got = out[tok, hd].float().cpu().numpy()
            gl = lse[hd, tok].cpu().numpy()
            errs.append(np.abs(got - o_ref).ravel())
            lerrs.append(np.abs(gl - l_ref))
        row_base += nqb * hkv
        kb_base += nkb
    e, le = np.concatenate(errs), np.concatenate(lerrs)
    assert np.isfinite(e).all()
    assert e.max() <= max_abs, (e.max(), e.mean())
    assert e.mean() <= mean_abs, e.mean()
    assert le.max() <= lse_abs, le.max()
    return dict(density=kept_total / causal_total, emax=float(e.max()))


def test_qwen30b_128k_bf16():
    """The benchmark's headline layer: 128K, 32/4 heads, shuffled 64-token pages."""
    sampled_parity(synth.config_spec(3))


def test_qwen30b_128k_bf16_sparse_regime():
    """The same layer with queries scaled by 16 (the bench's sparse variant)."""
    r = sampled_parity(synth.config_spec(3, logit_scale=16.0))
    assert r["density"] < 0.3


def test_qwen30b_128k_e4m3():
    sampled_parity(synth.config_spec(3, dtype="e4m3"), max_abs=FP8_MAX_ABS, mean_abs=6e-3, lse_abs=FP8_LSE_ABS)


def test_varlen_batch_with_chunk():
    """Six requests in one interleaved page pool, one an 8192-query chunk at 40960."""
    sampled_parity(synth.config_spec(4), rows_per_request=2)


def test_256k_bf16():
    sampled_parity(synth.config_spec(5), rows_per_request=2, queries_per_row=16)
