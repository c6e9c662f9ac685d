"""CUDA path (through the C ABI) against the float64 oracle, stage by stage:
pooled means, block scores, keep masks / CSR (bit-exact outside the flagged
near-threshold band), and the attention output (max-abs 2e-2, mean-abs 2e-3
for bf16)."""
import numpy as np
import pytest

from block_sparse_long_fp_gb300 import synth
from parity_util import (check_outputs, check_pool, check_scores_and_index, density, gpu_stage_outputs,
                         keep_from_csr, oracle_outputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_fp_gb300 import build
    build.build()


def full_parity(spec, alpha=0.1, mean_corr=True, rows_per_request=None, max_abs=None, mean_abs=None,
                lse_abs=2e-2, select=None, v_layout=0, case_fn=None):
    """select: {select_rule, top_k, top_p} for the top-k / top-p ablations;
    v_layout: the value cache's layout on the GPU (the oracle reads the same values);
    case_fn: changes the generated case before both sides see it."""
    import oracle
    from parity_util import BF16_MAX_ABS, BF16_MEAN_ABS
    case = synth.make_case(spec)
    if case_fn is not None:
        case_fn(case)
    sel = select or {}
    ref = oracle.discover_and_select(case, alpha=alpha, rule=sel.get("select_rule", 0), top_k=sel.get("top_k", 0),
                                     top_p=sel.get("top_p", 0.0), head_union=sel.get("score_mode", 0) == 1)
    g = gpu_stage_outputs(case, alpha=alpha, mean_corr=mean_corr, select=select, v_layout=v_layout)
    assert g["status"] == 0
    check_pool(case, g, ref)
    flips = check_scores_and_index(case, g, ref)
    # the attention on the index the GPU selected (identical to the oracle's
    # outside the flagged near-threshold band, which the check above allows)
    oref = oracle_outputs(case, ref, mean_corr, rows_per_request=rows_per_request, keeps=keep_from_csr(case, g))
    emax, emean = check_outputs(case, g, oref, max_abs=max_abs or BF16_MAX_ABS, mean_abs=mean_abs or BF16_MEAN_ABS,
                                lse_abs=lse_abs)
    return dict(density=density(case, ref), flips=flips, emax=emax, emean=emean)


@pytest.mark.parametrize("mean_corr", [True, False])
def test_tiny_workload(mean_corr):
    """2K tokens, 4 query heads on 1 kv head, contiguous KV (workload 1)."""
    full_parity(synth.config_spec(1), mean_corr=mean_corr)


@pytest.mark.parametrize("mean_corr", [True, False])
def test_sharp_logits_skip_blocks(mean_corr):
    """8K tokens, queries scaled by 8: about half of the blocks fall below
    alpha * max, so skipping and the mean-correction tiles are exercised."""
    spec = synth.Spec("sharp-8k", [(8192, 0)], 4, 1, page_size=64, layout="shuffled", n_needles=2,
                      logit_scale=8.0, config_id=1)
    r = full_parity(spec, mean_corr=mean_corr, rows_per_request=3000)
    assert r["density"] < 0.7


@pytest.mark.parametrize("page,layout", [(16, "shuffled"), (64, "interleaved"), (128, "shuffled"),
                                         (256, "contiguous")])
def test_varlen_chunked_ragged(page, layout):
    """Several requests in one paged pool: ragged lengths, a one-token
    request and chunks whose queries start at positions 512 and 128."""
    spec = synth.Spec("varlen-small", [(300, 0), (1000, 0), (256, 512), (1, 128), (640, 0)], 8, 2,
                      page_size=page, layout=layout, n_needles=2, logit_scale=6.0, config_id=60 + page)
    full_parity(spec)


def test_random_index_attention_only():
    """fp_sparse_attn alone on a random CSR (diagonal + each earlier block
    with probability 0.3), compared with the oracle on the same index."""
    import math
    import torch
    import oracle
    from block_sparse_long_fp_gb300 import fprefill
    spec = synth.Spec("rand-csr", [(1536, 0), (700, 256)], 8, 2, page_size=32, layout="shuffled",
                      n_needles=1, config_id=71)
    case = synth.make_case(spec)
    rows = synth.random_keep_lists(case, 0.3, seed=5)
    row_ptr = np.zeros(len(rows) + 1, np.int32)
    row_ptr[1:] = np.cumsum([len(x) for x in rows])
    col_idx = np.concatenate(rows).astype(np.int32)
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, _ = layer.discover()
    rp = torch.from_numpy(row_ptr).cuda()
    ci = torch.from_numpy(col_idx).cuda()
    out, lse = layer.sparse_attn(rp, ci, k_mean, v_mean)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    g = dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy())
    k = 0
    oref = []
    for r, (lq, start) in enumerate(spec.requests):
        q = oracle.request_q(case, r)
        kk, vv = oracle.request_kv(case, r)
        kbar, vbar = oracle.pool(kk, 128), oracle.pool(vv, 128)
        nqb = -(-lq // 128)
        keep = np.zeros((nqb, spec.h_kv, kbar.shape[0]), np.uint8)
        for i in range(nqb):
            for h in range(spec.h_kv):
                keep[i, h, rows[k]] = 1
                k += 1
        qi = np.repeat(np.arange(lq), spec.h_q)
        qh = np.tile(np.arange(spec.h_q), lq)
        o, l = oracle.attn_rows(q, start, kk, vv, kbar, vbar, 128, 1 / math.sqrt(128), keep, True, qi, qh)
        oref.append((qi, qh, o, l))
    check_outputs(case, g, oref)


@pytest.mark.parametrize("mean_corr,kv_splits", [(True, 0), (False, 0), (True, 3), (False, 5)])
def test_empty_rows_and_rows_without_their_diagonal_block(mean_corr, kv_splits):
    """A CSR where every third row is empty and every fifth drops its own
    (diagonal) block.  With the correction an empty row past block 0 is made
    of mean tokens only; a row with no term at all gives O = 0, LSE = -inf."""
    import math
    import torch
    import oracle
    from block_sparse_long_fp_gb300 import fprefill
    spec = synth.Spec("empty-rows", [(1536, 0), (700, 256), (128, 0)], 8, 2, page_size=32, layout="shuffled",
                      n_needles=1, config_id=74)
    case = synth.make_case(spec)
    rows = synth.random_keep_lists(case, 0.3, seed=7)
    for k in range(len(rows)):
        if k % 3 == 0:
            rows[k] = rows[k][:0]
        elif k % 5 == 0:
            rows[k] = rows[k][:-1]
    row_ptr = np.zeros(len(rows) + 1, np.int32)
    row_ptr[1:] = np.cumsum([len(x) for x in rows])
    col_idx = np.concatenate(rows).astype(np.int32)
    layer = fprefill.layer_from_case(case, params=fprefill.default_params(mean_correction=int(mean_corr),
                                                                          kv_splits=kv_splits))
    k_mean, v_mean, _ = layer.discover()
    out, lse = layer.sparse_attn(torch.from_numpy(row_ptr).cuda(), torch.from_numpy(col_idx).cuda(), k_mean,
                                 v_mean)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    got_o, got_l = out.float().cpu().numpy(), lse.cpu().numpy()
    k = 0
    n_void = 0
    for r, (lq, start) in enumerate(spec.requests):
        q = oracle.request_q(case, r)
        kk, vv = oracle.request_kv(case, r)
        kbar, vbar = oracle.pool(kk, 128), oracle.pool(vv, 128)
        nqb = -(-lq // 128)
        keep = np.zeros((nqb, spec.h_kv, kbar.shape[0]), np.uint8)
        for i in range(nqb):
            for h in range(spec.h_kv):
                keep[i, h, rows[k]] = 1
                k += 1
        qi = np.repeat(np.arange(lq), spec.h_q)
        qh = np.tile(np.arange(spec.h_q), lq)
        o, l = oracle.attn_rows(q, start, kk, vv, kbar, vbar, 128, 1 / math.sqrt(128), keep, mean_corr, qi, qh)
        q0 = int(case.cu_seqlens_q[r])
        go, gl = got_o[q0 + qi, qh], got_l[qh, q0 + qi]
        void = np.isneginf(l)
        n_void += int(void.sum())
        assert np.array_equal(np.isneginf(gl), void), r
        assert np.all(go[void] == 0.0), r
        err = np.abs(go[~void] - o[~void])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (r, err.max(), err.mean())
        assert np.abs(gl[~void] - l[~void]).max() <= 2e-2, r
    assert n_void > 0


@pytest.mark.parametrize("kv_splits,v_layout", [(0, 0), (4, 0), (0, 1)])
def test_dense_path_equals_causal_softmax(kv_splits, v_layout):
    import oracle
    spec = synth.Spec("dense", [(1000, 0), (384, 256)], 4, 2, page_size=64, layout="shuffled",
                      n_needles=1, config_id=72)
    case = synth.make_case(spec)
    ref = oracle.discover_and_select(case)
    g = gpu_stage_outputs(case, dense=True, kv_splits=kv_splits, v_layout=v_layout)
    assert g["status"] == 0
    oref = oracle_outputs(case, ref, mean_corr=False, dense=True)
    check_outputs(case, g, oref)


@pytest.mark.parametrize("dtype,logit_scale", [("bf16", 8.0), ("e4m3", 6.0)])
def test_split_kv_chunk_at_the_end_of_a_long_context(dtype, logit_scale):
    """A 512-query chunked-prefill step at position 32768: 16 work units for
    152 SMs, so each row's key list is split (automatically) and merged by LSE."""
    import ctypes
    from block_sparse_long_fp_gb300 import fprefill
    from parity_util import FP8_LSE_ABS, FP8_MAX_ABS
    spec = synth.Spec("chunk-at-32k", [(512, 32768)], 8, 2, page_size=64, layout="shuffled", n_needles=2,
                      logit_scale=logit_scale, dtype=dtype, config_id=75)
    case = synth.make_case(spec)
    layer = fprefill.layer_from_case(case)
    one = fprefill.default_params(kv_splits=1)
    L = fprefill.lib()
    assert layer.ws_bytes > L.fp_attn_workspace_size(ctypes.byref(layer.problem), ctypes.byref(one))
    fp8 = dtype == "e4m3"
    full_parity(spec, rows_per_request=700, max_abs=FP8_MAX_ABS if fp8 else None, mean_abs=6e-3 if fp8 else None,
                lse_abs=FP8_LSE_ABS if fp8 else 2e-2)


@pytest.mark.parametrize("select,mean_corr", [(dict(select_rule=1, top_k=1), True), (dict(select_rule=1, top_k=1), False),
                                              (dict(select_rule=1, top_k=8), True),
                                              (dict(select_rule=2, top_p=0.5), True),
                                              (dict(select_rule=2, top_p=0.9), True)])
def test_topk_topp_selection_ablations(select, mean_corr):
    """The top-k and top-p rules (ablations of the max threshold): the GPU's
    index equals the oracle's outside the flagged boundary band, and the
    attention on it matches.  With one kept block per row (k = 1) a row is
    nearly all mean tokens: the mean tiles' keys enter the MMA in fp16 (11
    significant bits, against fp16 queries), so their logits err by 2^-12
    relative, not the 2^-9 of one bf16 term."""
    spec = synth.Spec("sharp-8k", [(8192, 0)], 4, 1, page_size=64, layout="shuffled", n_needles=2,
                      logit_scale=8.0, config_id=1)
    full_parity(spec, rows_per_request=1500, select=select, mean_corr=mean_corr)


@pytest.mark.parametrize("select", [dict(select_rule=1, top_k=3), dict(select_rule=2, top_p=0.7)])
def test_topk_topp_on_a_ragged_varlen_batch(select):
    spec = synth.Spec("varlen-small", [(300, 0), (1000, 0), (256, 512), (1, 128), (640, 0)], 8, 2,
                      page_size=32, layout="interleaved", n_needles=2, logit_scale=6.0, config_id=92)
    full_parity(spec, select=select)


@pytest.mark.parametrize("name,select", [("varlen", None), ("sharp", None), ("e4m3", None),
                                         ("sharp", dict(select_rule=1, top_k=4))])
def test_discover_select_equals_the_separate_stages(name, select):
    """fp_discover_select gives bit for bit what fp_discover + fp_select give:
    the same means, score map and index (fused with the threshold rule; the
    separate kernels behind one call for the other rules).  Its own outputs
    are also checked against the oracle: the means, the optional score map,
    and the index of both forms of the call (with and without the score map)
    outside the flagged near-threshold band."""
    import torch
    import oracle
    from block_sparse_long_fp_gb300 import fprefill
    specs = {
        "varlen": synth.Spec("varlen-small", [(300, 0), (1000, 0), (256, 512), (1, 128), (640, 0)], 8, 2,
                             page_size=32, layout="interleaved", n_needles=2, logit_scale=6.0, config_id=93),
        "sharp": synth.Spec("sharp-8k", [(8192, 0)], 4, 1, page_size=64, layout="shuffled", n_needles=2,
                            logit_scale=8.0, config_id=1),
        "e4m3": synth.Spec("e4m3-chunk", [(1024, 2048), (700, 0)], 8, 2, page_size=64, layout="shuffled",
                           n_needles=2, logit_scale=6.0, dtype="e4m3", config_id=94),
    }
    case = synth.make_case(specs[name])
    sel = select or {}
    layer = fprefill.layer_from_case(case, params=fprefill.default_params(**sel))
    km, vm, sc = layer.discover()
    rp, ci, nz = layer.select(sc)
    score = torch.full_like(sc, float("nan"))
    km2, vm2, rp2, ci2, nz2 = layer.discover_select(score=score)
    km3, vm3, rp3, ci3, nz3 = layer.discover_select()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    n = int(nz.item())
    assert int(nz2.item()) == n and int(nz3.item()) == n
    assert torch.equal(km, km2) and torch.equal(vm, vm2)
    assert torch.equal(sc, score)
    assert torch.equal(rp, rp2) and torch.equal(rp, rp3)
    assert torch.equal(ci[:n], ci2[:n]) and torch.equal(ci[:n], ci3[:n])
    # the fused call's own outputs against the float64 oracle
    ref = oracle.discover_and_select(case, rule=sel.get("select_rule", 0), top_k=sel.get("top_k", 0),
                                     top_p=sel.get("top_p", 0.0))
    fused = dict(k_mean=km3.cpu().numpy(), v_mean=vm3.cpu().numpy(), score=None, row_ptr=rp3.cpu().numpy(),
                 col_idx=ci3.cpu().numpy())
    check_pool(case, fused, ref)
    check_scores_and_index(case, fused, ref)
    with_map = dict(k_mean=km2.cpu().numpy(), v_mean=vm2.cpu().numpy(), score=score.cpu().numpy(),
                    row_ptr=rp2.cpu().numpy(), col_idx=ci2.cpu().numpy())
    check_pool(case, with_map, ref)
    check_scores_and_index(case, with_map, ref)


@pytest.mark.parametrize("name", ["varlen", "sharp", "e4m3"])
def test_union_of_heads_scores_selection_and_attention(name):
    """FP_SCORE_HEAD_UNION (each query head scored alone, the row keeps the
    maximum over the group): scores within 2e-6, the index exact outside the
    flagged band, the attention on it within the bounds."""
    from parity_util import FP8_LSE_ABS, FP8_MAX_ABS
    specs = {
        "varlen": synth.Spec("varlen-small", [(300, 0), (1000, 0), (256, 512), (1, 128), (640, 0)], 8, 2,
                             page_size=32, layout="interleaved", n_needles=2, logit_scale=6.0, config_id=95),
        "sharp": synth.Spec("sharp-8k", [(8192, 0)], 4, 1, page_size=64, layout="shuffled", n_needles=2,
                            logit_scale=8.0, config_id=1),
        "e4m3": synth.Spec("e4m3-chunk", [(1024, 2048), (700, 0)], 8, 2, page_size=64, layout="shuffled",
                           n_needles=2, logit_scale=6.0, dtype="e4m3", config_id=96),
    }
    fp8 = name == "e4m3"
    r = full_parity(specs[name], rows_per_request=1500, select=dict(score_mode=1),
                    max_abs=FP8_MAX_ABS if fp8 else None, mean_abs=6e-3 if fp8 else None,
                    lse_abs=FP8_LSE_ABS if fp8 else 2e-2)
    if name == "sharp":
        packed = full_parity(specs[name], rows_per_request=200)
        assert r["density"] >= packed["density"]   # every head's own blocks: a larger union


def test_union_of_heads_with_an_odd_group():
    """Three query heads per kv head (the last pair has one head): scores and
    index only (the attention kernel takes head pairs)."""
    import oracle
    spec = synth.Spec("odd-group", [(700, 0), (300, 256)], 6, 2, page_size=64, layout="shuffled", n_needles=1,
                      logit_scale=6.0, config_id=97)
    case = synth.make_case(spec)
    ref = oracle.discover_and_select(case, head_union=True)
    g = gpu_stage_outputs(case, select=dict(score_mode=1), attention=False)
    assert g["status"] == 0
    check_scores_and_index(case, g, ref)


def test_page_table_entry_out_of_range_sets_status():
    """A corrupted page-table entry is caught by the kernels' bounds checks:
    the status word reports it and the run completes."""
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    spec = synth.Spec("bad-page", [(512, 0)], 4, 2, page_size=64, layout="contiguous", config_id=73)
    case = synth.make_case(spec)
    case.block_table[0, 3] = case.k_cache.shape[0] + 5
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, score = layer.discover()
    layer.dense_attn()
    torch.cuda.synchronize()
    assert layer.device_status() == fprefill.FP_ERR_DEVICE_BOUNDS


def test_index_entry_out_of_range_sets_status():
    """Index entries outside [0, I] (a negative block, a block after the
    diagonal) are caught before any page-table read: the status word reports
    them and the run completes."""
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    spec = synth.Spec("bad-index", [(512, 0)], 4, 2, page_size=64, layout="contiguous", config_id=74)
    case = synth.make_case(spec)
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    rp = row_ptr.cpu().numpy()
    ci = col_idx.clone()
    ci[int(rp[0])] = -1                        # row (I = 0, h = 0)
    ci[int(rp[2 * spec.h_kv + 1])] = 3         # row (I = 2, h = 1): its first entry becomes J = 3 > I
    layer.sparse_attn(row_ptr, ci, k_mean, v_mean)
    torch.cuda.synchronize()
    assert layer.device_status() == fprefill.FP_ERR_DEVICE_BOUNDS


def test_a_wait_that_runs_out_reports_timeout_and_the_context_stays_usable():
    """The bounded wait the kernels use gives up on a barrier that nothing
    completes: FP_ERR_TIMEOUT lands in the status word, no fault, and the
    same workspace then serves a normal attention call with the same result
    as before."""
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    spec = synth.Spec("timeout", [(700, 0), (300, 256)], 8, 2, page_size=64, layout="shuffled", n_needles=1,
                      logit_scale=6.0, config_id=75)
    case = synth.make_case(spec)
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    out, lse = layer.sparse_attn(row_ptr, col_idx, k_mean, v_mean)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    ref_out, ref_lse = out.clone(), lse.clone()
    layer.check_wait_timeout(2_000_000)               # 2 ms on a barrier nothing arrives on
    torch.cuda.synchronize()
    assert layer.device_status() == fprefill.FP_ERR_TIMEOUT
    layer.reset_status()
    out2, lse2 = layer.sparse_attn(row_ptr, col_idx, k_mean, v_mean)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert torch.equal(out2, ref_out) and torch.equal(lse2, ref_lse)


def test_fp8_discover_and_select():
    """e4m3 inputs with per-head scales: block means of the dequantised
    values, fp32 scores and the index against the oracle on the same codes."""
    import oracle
    spec = synth.Spec("fp8-disc", [(2048, 0), (700, 256)], 8, 2, page_size=64, layout="shuffled",
                      dtype="e4m3", n_needles=2, logit_scale=6.0, config_id=74)
    case = synth.make_case(spec)
    ref = oracle.discover_and_select(case)
    from block_sparse_long_fp_gb300 import fprefill
    import torch
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    g = dict(k_mean=k_mean.cpu().numpy(), v_mean=v_mean.cpu().numpy(), score=score.cpu().numpy(),
             row_ptr=row_ptr.cpu().numpy(), col_idx=col_idx.cpu().numpy())
    check_pool(case, g, ref)
    check_scores_and_index(case, g, ref)


@pytest.mark.parametrize("logit_scale", [1.0, 6.0])
def test_fp8_attention_workload_generator(logit_scale):
    """e4m3 at the workloads' own generator (scale 1) and sharper logits."""
    from parity_util import FP8_LSE_ABS, FP8_MAX_ABS
    spec = synth.Spec("fp8-gen", [(4096, 0)], 8, 2, page_size=64, layout="shuffled", dtype="e4m3",
                      n_needles=2, logit_scale=logit_scale, config_id=76)
    full_parity(spec, rows_per_request=3000, max_abs=FP8_MAX_ABS, mean_abs=6e-3, lse_abs=FP8_LSE_ABS)


@pytest.mark.parametrize("mean_corr,p_terms", [(True, 2), (False, 2), (True, 1), (False, 1)])
def test_fp8_attention_sharp_varlen(mean_corr, p_terms):
    """e4m3 Q/K/V with per-head scales through the whole path (kind::f8f6f4
    MMAs), varlen with a chunk, blocks really skipped.

    Queries scaled by 6 make two to four keys dominate each row.  With P as
    the pages' single e4m3 term of 256 p (p_terms 1) the row's largest
    weight is exact but the next ones carry up to 1/16 relative rounding,
    which no longer averages out: the measured worst element is 0.062, so
    that form is held to max-abs 0.1.  With the residual term (p_terms 2,
    a second PV pass) the weights carry about 1/256 and the FP8 bound
    max-abs 6e-2 holds."""
    from parity_util import FP8_LSE_ABS, FP8_MAX_ABS
    spec = synth.Spec("fp8-attn", [(2048, 0), (700, 256), (3000, 0)], 8, 2, page_size=64, layout="shuffled",
                      dtype="e4m3", n_needles=2, logit_scale=6.0, config_id=75)
    r = full_parity(spec, mean_corr=mean_corr, rows_per_request=2000, max_abs=FP8_MAX_ABS if p_terms == 2 else 0.1,
                    mean_abs=6e-3, lse_abs=FP8_LSE_ABS, select=dict(p_terms=p_terms))
    assert r["density"] < 0.95


@pytest.mark.parametrize("dtype,page", [("bf16", 64), ("bf16", 256), ("e4m3", 128), ("e4m3", 256)])
def test_dim_major_value_cache(dtype, page):
    """The value cache stored dim-major, [num_pages, h_kv, d, page_size] with
    each page's keys contiguous (the column-stored values of the V2 popular
    article's FP8 passage).  Pooling reads it in place; the attention takes a
    kept block's V tile as a K-major operand (mean tiles keep their own
    token-major copies).  The whole path against the oracle, which reads the
    same values token-major, on a ragged varlen batch with a chunk and skipped
    blocks."""
    from parity_util import FP8_LSE_ABS, FP8_MAX_ABS
    spec = synth.Spec("v-dim-major", [(2048, 0), (3000, 0), (256, 512)], 8, 2, page_size=page, layout="shuffled",
                      dtype=dtype, n_needles=2, logit_scale=6.0, config_id=76)
    if dtype == "bf16":
        r = full_parity(spec, v_layout=1, rows_per_request=2000)
    else:
        # queries x 6 make rows sharp: P in two e4m3 terms (see the test above)
        r = full_parity(spec, v_layout=1, rows_per_request=2000, max_abs=FP8_MAX_ABS, mean_abs=6e-3,
                        lse_abs=FP8_LSE_ABS, select=dict(p_terms=2))
    assert r["density"] < 0.95


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_long_rows_on_the_tensor_cores_with_shared_column_sums(dtype):
    """A 3300-block request (422,400 tokens): past 3120 blocks the tensor-core
    score kernel keeps one column-sum array per head slot, added to with
    shared-memory atomics.  Sampled score rows (within 2e-6) and their index
    rows (exact outside the flagged band) against the oracle."""
    import oracle
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    L = 3300 * 128
    spec = synth.Spec("long-rows-tc", [(L, 0)], 8, 1, page_size=128, layout="shuffled", dtype=dtype,
                      n_needles=2, logit_scale=4.0, config_id=78)
    case = synth.make_case(spec)
    rows = np.array([0, 5, 1023, 1024, 2048, 3120, 3299])
    ref = oracle.discover_and_select(case, row_subset=lambda r, nqb, hkv: rows)
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    g = dict(k_mean=k_mean.cpu().numpy(), v_mean=v_mean.cpu().numpy(), score=score.cpu().numpy(),
             row_ptr=row_ptr.cpu().numpy(), col_idx=col_idx.cpu().numpy())
    check_pool(case, g, ref)
    check_scores_and_index(case, g, ref)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_rows_past_the_tensor_core_limit_use_the_fp32_score_kernel(dtype):
    """A 1,612,800-token request (12600 key blocks) is past the tensor-core
    score kernel's shared-memory limit (12480 blocks, with one column-sum array
    per head slot past 3120): its scores come from the fp32 CUDA-core kernel.
    Sampled score rows and their index rows against the oracle."""
    import oracle
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    L = 12600 * 128
    spec = synth.Spec("long-rows", [(L, 0)], 2, 1, page_size=128, layout="shuffled", dtype=dtype,
                      n_needles=2, logit_scale=4.0, config_id=77)
    case = synth.make_case(spec)
    rows = np.array([0, 5, 700, 4096, 12599])
    ref = oracle.discover_and_select(case, row_subset=lambda r, nqb, hkv: rows)
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    g = dict(k_mean=k_mean.cpu().numpy(), v_mean=v_mean.cpu().numpy(), score=score.cpu().numpy(),
             row_ptr=row_ptr.cpu().numpy(), col_idx=col_idx.cpu().numpy())
    check_pool(case, g, ref)
    check_scores_and_index(case, g, ref)


@pytest.mark.parametrize("nkb", [1072, 1073])
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_rows_at_the_limit_of_the_staged_query_tiles(nkb, dtype):
    """Rows of up to 1072 blocks stage their query tiles in shared memory (the
    launch then takes all 227 KB); 1073 reads them from global memory.  Two
    head pairs, so the phases overlap; sampled score and index rows against
    the oracle on both sides of the limit."""
    import oracle
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    spec = synth.Spec("staged-limit", [(nkb * 128, 0)], 4, 1, page_size=128, layout="shuffled", dtype=dtype,
                      n_needles=2, logit_scale=4.0, config_id=79)
    case = synth.make_case(spec)
    rows = np.array([0, 1, 127, 128, 700, nkb - 2, nkb - 1])
    ref = oracle.discover_and_select(case, row_subset=lambda r, nqb, hkv: rows)
    layer = fprefill.layer_from_case(case)
    k_mean, v_mean, score = layer.discover()
    row_ptr, col_idx, nnz = layer.select(score)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    g = dict(k_mean=k_mean.cpu().numpy(), v_mean=v_mean.cpu().numpy(), score=score.cpu().numpy(),
             row_ptr=row_ptr.cpu().numpy(), col_idx=col_idx.cpu().numpy())
    check_pool(case, g, ref)
    check_scores_and_index(case, g, ref)


def _bf16_times_pow2(bits, e):
    """bf16 bit patterns times 2^e, exactly: the exponent field moves by e
    (zeros stay zero; every normal value stays normal)."""
    b = bits.astype(np.int32)
    ex = (b >> 7) & 0xff
    ok = (ex > 0) & (ex < 255)
    ne = ex + e
    assert np.all((ne[ok] > 0) & (ne[ok] < 255))
    return np.where(ok, (b & ~(0xff << 7)) | (ne << 7), b).astype(np.uint16)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_queries_and_keys_far_from_unit_scale(dtype):
    """Queries times 2^-13 and keys times 2^13 (bf16 values, or the e4m3
    per-head scales): every logit equals the unscaled case's, but the key
    means reach past fp16's largest value and most query entries fall below
    its normal range.  The score MMAs and the bf16 mean tiles take fp16
    operands scaled by powers of two (per 128-block tile of key means, per
    query row), so scores, index and outputs meet the same bounds."""
    from parity_util import FP8_LSE_ABS, FP8_MAX_ABS
    spec = synth.Spec("scaled-8k", [(8192, 0)], 4, 1, page_size=64, layout="shuffled", dtype=dtype, n_needles=2,
                      logit_scale=6.0, config_id=5)

    def scale(case):
        if dtype == "bf16":
            case.q = _bf16_times_pow2(case.q, -13)
            case.k_cache = _bf16_times_pow2(case.k_cache, 13)
        else:
            case.q_scale = (case.q_scale * 2.0 ** -13).astype(np.float32)
            case.k_scale = (case.k_scale * 2.0 ** 13).astype(np.float32)

    fp8 = dtype == "e4m3"
    r = full_parity(spec, rows_per_request=3000, case_fn=scale, max_abs=FP8_MAX_ABS if fp8 else None,
                    mean_abs=6e-3 if fp8 else None, lse_abs=FP8_LSE_ABS if fp8 else 2e-2,
                    select=dict(p_terms=2) if fp8 else None)
    assert r["density"] < 0.8
