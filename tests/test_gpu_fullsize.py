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


def sample_rows(spec, case, r, score_h, offs, rng, n_random, n_near=8, alpha=0.1):
    """Score rows (query block i, kv head h) of request r to check: the first
    and the last, every needle row of the generator, up to n_near rows whose
    scores (as the GPU computed them; used only to choose rows) have an entry
    within 1e-3 relative of the threshold, and random rows up to n_random."""
    lq, start = spec.requests[r]
    nqb, hkv = -(-lq // 128), spec.h_kv
    rows = {(nqb - 1, hkv - 1), (0, 0)}
    for nd in case.needles:
        i = nd["query_block"] - start // 128
        if nd["request"] == r and 0 <= i < nqb:
            rows.add((i, nd["kv_head"]))
    near = []
    for i in rng.permutation(nqb):
        for h in range(hkv):
            o = offs[r][i, h]
            sc = score_h[o:o + start // 128 + i + 1]
            if np.any(np.abs(sc - alpha) <= 1e-3 * alpha):
                near.append((int(i), h))
        if len(near) >= n_near:
            break
    rows.update(near[:n_near])
    while len(rows) < min(n_random, nqb * hkv):
        rows.add((int(rng.integers(0, nqb)), int(rng.integers(0, hkv))))
    return sorted(rows)


def sampled_parity(spec, alpha=0.1, mean_corr=(True,), rows_per_request=32, queries_per_row=64,
                   max_abs=BF16_MAX_ABS, mean_abs=BF16_MEAN_ABS, lse_abs=2e-2, seed=0, p_terms=1):
    """The three calls of the benchmark step on the full workload, then, on
    sampled rows: pooled means of every block, score rows, their index rows
    (exact outside the flagged band) and sampled output rows of the
    attention, for each mean-correction setting in `mean_corr` (the same
    index serves both)."""
    import torch
    import oracle
    from block_sparse_long_fp_gb300 import fprefill
    case = synth.make_case(spec)
    prm = fprefill.default_params(alpha=alpha, p_terms=p_terms)
    layer = fprefill.layer_from_case(case, params=prm)
    # one pass of the path, the three calls of the benchmark step
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    outs = {}
    for mc in mean_corr:
        layer.params.mean_correction = int(mc)
        outs[mc] = layer.sparse_attn(row_ptr, col_idx, k_mean, v_mean)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    score_h = score.cpu().numpy()
    rp, ci = row_ptr.cpu().numpy(), col_idx.cpu().numpy()
    km, vm = k_mean.cpu().numpy(), v_mean.cpu().numpy()
    hkv, g = spec.h_kv, spec.h_q // spec.h_kv
    scale = 1 / math.sqrt(spec.d)
    offs, _ = oracle.score_row_offsets(spec.requests, hkv, 128)
    rng = np.random.default_rng(seed)
    errs = {mc: [] for mc in mean_corr}
    lerrs = {mc: [] for mc in mean_corr}
    kept_total = causal_total = n_rows = 0
    row_base = kb_base = 0
    for r, (lq, start) in enumerate(spec.requests):
        nqb = -(-lq // 128)
        k, v = oracle.request_kv(case, r)
        kbar, vbar = oracle.pool(k, 128), oracle.pool(v, 128)
        nkb = kbar.shape[0]
        np.testing.assert_allclose(km[kb_base:kb_base + nkb], kbar, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(vm[kb_base:kb_base + nkb], vbar, rtol=1e-5, atol=1e-6)
        for i, h in sample_rows(spec, case, r, score_h, offs, rng, rows_per_request, alpha=alpha):
            n_rows += 1
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
            tok = torch.as_tensor(q0 + qi, device=score.device)
            hd = torch.as_tensor(qh, device=score.device)
            for mc in mean_corr:
                o_ref, l_ref = oracle.attn_rows(qblk, start + i * 128, k, v, kbar, vbar, 128, scale, keep, mc,
                                                qi, qh)
                out, lse = outs[mc]
                got = out[tok, hd].float().cpu().numpy()
                gl = lse[hd, tok].cpu().numpy()
                errs[mc].append(np.abs(got - o_ref).ravel())
                lerrs[mc].append(np.abs(gl - l_ref))
        row_base += nqb * hkv
        kb_base += nkb
    res = dict(density=kept_total / causal_total, rows=n_rows)
    for mc in mean_corr:
        e, le = np.concatenate(errs[mc]), np.concatenate(lerrs[mc])
        assert np.isfinite(e).all()
        assert e.max() <= max_abs, (mc, e.max(), e.mean())
        assert e.mean() <= mean_abs, (mc, e.mean())
        assert le.max() <= lse_abs, (mc, le.max())
        res[f"emax_mc{int(mc)}"] = float(e.max())
    return res


def test_qwen30b_128k_bf16():
    """The benchmark's headline layer: 128K, 32/4 heads, shuffled 64-token pages."""
    r = sampled_parity(synth.config_spec(3))
    assert r["rows"] >= 32


def test_qwen30b_128k_bf16_sparse_regime():
    """The same layer with queries scaled by 16 (the bench's sparse variant),
    with the mean correction on and off."""
    r = sampled_parity(synth.config_spec(3, logit_scale=16.0), mean_corr=(True, False))
    assert r["density"] < 0.3 and r["rows"] >= 32


def test_qwen30b_128k_e4m3():
    sampled_parity(synth.config_spec(3, dtype="e4m3"), max_abs=FP8_MAX_ABS, mean_abs=6e-3, lse_abs=FP8_LSE_ABS)


def test_qwen30b_128k_e4m3_two_term_p():
    """The 128K e4m3 layer with queries x 16 and P in two e4m3 terms."""
    sampled_parity(synth.config_spec(3, dtype="e4m3", logit_scale=16.0), max_abs=FP8_MAX_ABS, mean_abs=6e-3,
                   lse_abs=FP8_LSE_ABS, rows_per_request=16, p_terms=2)


def test_qwen30b_128k_e4m3_sparse_regime():
    """e4m3 with queries x 16 (through the per-head query scales): the
    configuration of the bench's FP8 sparse number, at the FP8 bound."""
    r = sampled_parity(synth.config_spec(3, dtype="e4m3", logit_scale=16.0), max_abs=FP8_MAX_ABS, mean_abs=6e-3,
                       lse_abs=FP8_LSE_ABS)
    assert r["density"] < 0.3


def test_llama8b_32k_mean_correction_on_and_off():
    """Workload 2 (32K, 32/8 heads, shuffled 64-token pages) as specified and
    with queries x 16, the attention with the mean correction on and off."""
    sampled_parity(synth.config_spec(2), mean_corr=(True, False), rows_per_request=16, queries_per_row=32)
    sampled_parity(synth.config_spec(2, logit_scale=16.0), mean_corr=(True, False), rows_per_request=32)


def test_varlen_batch_with_chunk():
    """Six requests in one interleaved page pool, one an 8192-query chunk at 40960."""
    sampled_parity(synth.config_spec(4), rows_per_request=4, queries_per_row=32)


def test_256k_bf16():
    sampled_parity(synth.config_spec(5), rows_per_request=8, queries_per_row=32)
