"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it with the float64 oracle on the same seeded inputs."""
import math

import numpy as np

# tolerances of the output (against float64): bf16 path max-abs 2e-2, mean-abs 2e-3
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
FP8_MAX_ABS = 6e-2
# LSE of the e4m3 path: it is taken from fp32 sums of the unrounded weights (the e4m3
# rounding of P enters only O), so it carries fp32 error like the bf16 path
FP8_LSE_ABS = 2e-2
SCORE_ABS = 2e-6          # scores lie in (0, 1]; fp32 evaluation error is ~1e-7


def gpu_stage_outputs(case, alpha=0.1, mean_corr=True, dense=False, kv_splits=0, select=None, attention=True,
                      v_layout=0):
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    prm = fprefill.default_params(alpha=alpha, mean_correction=int(mean_corr), kv_splits=kv_splits, **(select or {}))
    layer = fprefill.layer_from_case(case, params=prm, v_layout=v_layout)
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    if not attention:
        out = lse = None
    elif dense:
        out, lse = layer.dense_attn()
    else:
        out, lse = layer.sparse_attn(row_ptr, col_idx, k_mean, v_mean)
    torch.cuda.synchronize()
    st = layer.device_status()
    return dict(layer=layer, k_mean=k_mean.cpu().numpy(), v_mean=v_mean.cpu().numpy(),
                score=score.cpu().numpy(), row_ptr=row_ptr.cpu().numpy(),
                col_idx=col_idx.cpu().numpy(), nnz=int(nnz.item()),
                out=None if out is None else out.float().cpu().numpy(),
                lse=None if lse is None else lse.cpu().numpy(), status=st)


def check_pool(case, g, ref):
    kb = 0
    for r, res in enumerate(ref):
        nkb = res["kbar"].shape[0]
        np.testing.assert_allclose(g["k_mean"][kb:kb + nkb], res["kbar"], rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(g["v_mean"][kb:kb + nkb], res["vbar"], rtol=1e-5, atol=1e-6)
        kb += nkb


def score_offsets(case):
    import oracle
    offs, total = oracle.score_row_offsets(case.spec.requests, case.spec.h_kv, 128)
    return offs, total


def check_scores_and_index(case, g, ref):
    """Scores within SCORE_ABS (when g["score"] is not None); the CSR equals
    the oracle's keep mask except at flagged (near-threshold) blocks.  Returns
    the number of flagged flips."""
    offs, total = score_offsets(case)
    hkv = case.spec.h_kv
    flips = 0
    row_base = 0
    for r, res in enumerate(ref):
        start = res["start"]
        for row, s_ref in zip(res["rows"], res["score"]):
            i, h = divmod(int(row), hkv)
            I = start // 128 + i
            o = offs[r][i, h]
            if g["score"] is not None:
                s_gpu = g["score"][o:o + I + 1]
                err = np.abs(s_gpu - s_ref).max()
                assert err <= SCORE_ABS, (r, i, h, err)
            grow = row_base + int(row)
            cols = g["col_idx"][g["row_ptr"][grow]:g["row_ptr"][grow + 1]]
            assert np.all(np.diff(cols) > 0), "CSR row not ascending"
            kept = np.zeros(I + 1, bool)
            kept[cols] = True
            want = res["keep"][i, h, :I + 1].astype(bool)
            diff = kept != want
            assert not np.any(diff & ~res["flag"][i, h, :I + 1].astype(bool)), (r, i, h, np.nonzero(diff))
            flips += int(diff.sum())
        row_base += -(-case.spec.requests[r][0] // 128) * hkv
    return flips


def keep_from_csr(case, g):
    """The GPU's index (row_ptr / col_idx) as per-request keep masks
    [nqb, h_kv, nkb], the layout the oracle's attention takes."""
    hkv = case.spec.h_kv
    out, row = [], 0
    for lq, start in case.spec.requests:
        nqb = -(-lq // 128)
        nkb = -(-(start + lq) // 128)
        keep = np.zeros((nqb, hkv, nkb), np.uint8)
        for i in range(nqb):
            for h in range(hkv):
                keep[i, h, g["col_idx"][g["row_ptr"][row]:g["row_ptr"][row + 1]]] = 1
                row += 1
        out.append(keep)
    return out


def oracle_outputs(case, ref, mean_corr, dense=False, rows_per_request=None, seed=0, keeps=None):
    """Oracle O/LSE for every query row (or a sample of them).  keeps: per
    request keep masks to use instead of the oracle's own selection (the
    GPU's index, once check_scores_and_index has accepted it: a block whose
    score sits in the flagged band at the threshold may go either way, and the
    attention is then compared on the same set of blocks)."""
    import oracle
    rng = np.random.default_rng(seed)
    outs = []
    for r, res in enumerate(ref):
        lq = case.spec.requests[r][0]
        hq = case.spec.h_q
        if rows_per_request is None:
            qi = np.repeat(np.arange(lq), hq)
            qh = np.tile(np.arange(hq), lq)
        else:
            n = rows_per_request
            qi = np.concatenate([rng.integers(0, lq, n), [0, lq - 1], np.arange(min(lq, 130))])
            qh = rng.integers(0, hq, len(qi))
        keep = None if dense else (res["keep"] if keeps is None else keeps[r])
        o, lse = oracle.attn_rows(res["q"], res["start"], res["k"], res["v"], res["kbar"], res["vbar"], 128,
                                  1 / math.sqrt(case.spec.d), keep, mean_corr and not dense, qi, qh)
        outs.append((qi, qh, o, lse))
    return outs


def check_outputs(case, g, oref, max_abs=BF16_MAX_ABS, mean_abs=BF16_MEAN_ABS, lse_abs=2e-2):
    errs, lerrs = [], []
    for r, (qi, qh, o, lse) in enumerate(oref):
        q0 = int(case.cu_seqlens_q[r])
        got = g["out"][q0 + qi, qh]
        errs.append(np.abs(got - o).ravel())
        lerrs.append(np.abs(g["lse"][qh, q0 + qi] - lse))
    e = np.concatenate(errs)
    le = np.concatenate(lerrs)
    assert np.isfinite(e).all()
    assert e.max() <= max_abs, (e.max(), e.mean())
    assert e.mean() <= mean_abs, e.mean()
    assert le.max() <= lse_abs, le.max()
    return float(e.max()), float(e.mean())


def density(case, ref):
    kept = tot = 0
    for r, res in enumerate(ref):
        lq, start = case.spec.requests[r]
        for i in range(-(-lq // 128)):
            I = start // 128 + i
            kept += int(res["keep"][i, :, :I + 1].sum())
            tot += (I + 1) * case.spec.h_kv
    return kept / max(1, tot)
