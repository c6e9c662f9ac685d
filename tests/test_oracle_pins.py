"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test states the fact it checks.  None of them re-types the oracle's own
formula: the references are either closed forms derived by hand
(tests/golden), textbook dense softmax attention, invariants of the
definitions, or a token-level brute force in a different formulation
("mean tokens" appended to the key set).
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dense_causal_softmax(q, k, v, start, scale):
    """Textbook causal softmax attention, whole matrix at once.
    q [lq,hq,d], k/v [lk,hkv,d]; query i sits at position start+i."""
    lq, hq, d = q.shape
    lk, hkv, _ = k.shape
    g = hq // hkv
    o = np.empty((lq, hq, d))
    lse = np.empty((lq, hq))
    pos = start + np.arange(lq)
    mask = np.arange(lk)[None, :] <= pos[:, None]
    for h in range(hq):
        s = scale * q[:, h, :] @ k[:, h // g, :].T
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        den = w.sum(axis=1, keepdims=True)
        o[:, h, :] = (w @ v[:, h // g, :]) / den
        lse[:, h] = (m + np.log(den))[:, 0]
    return o, lse


def rand_qkv(rng, lq, start, hq, hkv, d, scale_q=1.0):
    lk = start + lq
    q = rng.standard_normal((lq, hq, d)) * scale_q
    k = rng.standard_normal((lk, hkv, d))
    v = rng.standard_normal((lk, hkv, d))
    return q, k, v


def all_rows(oracle, q, k, v, start, B, scale, keep, mean_corr):
    lq, hq, d = q.shape
    qi = np.repeat(np.arange(lq), hq)
    qh = np.tile(np.arange(hq), lq)
    kbar, vbar = oracle.pool(k, B), oracle.pool(v, B)
    o, lse = oracle.attn_rows(q, start, k, v, kbar, vbar, B, scale, keep, mean_corr, qi, qh)
    return o.reshape(lq, hq, d), lse.reshape(lq, hq)


# ----------------------------------------------------------------------------
# pooling
# ----------------------------------------------------------------------------

def test_pool_is_block_mean_with_ragged_tail(oracle_mod):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((77, 3, 5))
    got = oracle_mod.pool(x, 16)
    assert got.shape == (5, 3, 5)
    for J in range(5):
        np.testing.assert_allclose(got[J], x[J * 16:(J + 1) * 16].mean(axis=0), rtol=0, atol=1e-14)
    # the last block has 77 - 64 = 13 tokens: its mean of a constant is that constant
    c = np.full((77, 1, 2), 3.25)
    assert np.all(oracle_mod.pool(c, 16) == 3.25)


# ----------------------------------------------------------------------------
# block scores
# ----------------------------------------------------------------------------

def test_score_matches_hand_derived_golden(oracle_mod):
    gdat = json.load(open(os.path.join(GOLDEN, "score_tiny.json")))
    B = gdat["B"]
    k = np.array(gdat["k"], dtype=float)[:, None, :]
    q = np.stack([np.array(gdat["q_head0"], float), np.array(gdat["q_head1"], float)], axis=1)
    kbar = oracle_mod.pool(k, B)
    np.testing.assert_array_equal(kbar[:, 0, :], np.array(gdat["kbar"], float))
    rows = oracle_mod.score_rows(q, 0, 1, B, gdat["scale"], kbar, [0, 1])
    np.testing.assert_allclose(rows[0], gdat["score_row_I0"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(rows[1], gdat["score_row_I1"], rtol=1e-14, atol=0)


def test_score_rows_peak_at_exactly_one(oracle_mod):
    rng = np.random.default_rng(1)
    q, k, _ = rand_qkv(rng, 256, 0, 4, 2, 16, scale_q=3.0)
    kbar = oracle_mod.pool(k, 32)
    rows = oracle_mod.score_rows(q, 0, 2, 32, 0.25, kbar, np.arange(16))
    for s in rows:
        assert s.max() == 1.0
        assert np.all(s > 0) and np.all(s <= 1.0)


def numpy_scores(q, kbar, start, hkv, B, scale):
    """Independent vectorised formulation: one logsumexp-style matrix per row."""
    lq, hq, d = q.shape
    g = hq // hkv
    out = {}
    for il in range(-(-lq // B)):
        I = start // B + il
        for h in range(hkv):
            qs = q[il * B:(il + 1) * B, h * g:(h + 1) * g, :].transpose(1, 0, 2).reshape(-1, d)
            s = scale * qs @ kbar[:I + 1, h, :].T              # [rows, I+1]
            p = np.exp(s - s.max(axis=1, keepdims=True))
            col = p.sum(axis=0)
            out[(il, h)] = col / col.max()
    return out


def test_score_matches_vectorised_formulation(oracle_mod):
    rng = np.random.default_rng(2)
    start, B = 64, 32
    q, k, _ = rand_qkv(rng, 200, start, 6, 2, 8, scale_q=2.0)
    kbar = oracle_mod.pool(k, B)
    ref = numpy_scores(q, kbar, start, 2, B, 0.3)
    nqb = -(-200 // B)
    rows = oracle_mod.score_rows(q, start, 2, B, 0.3, kbar, np.arange(nqb * 2))
    for r, s in enumerate(rows):
        np.testing.assert_allclose(s, ref[divmod(r, 2)], rtol=1e-12, atol=0)


def test_score_invariant_to_common_key_shift(oracle_mod):
    """Adding one vector c to every key shifts each query's logits by the
    same amount q.c for all J; the per-query max normalisation cancels it."""
    rng = np.random.default_rng(3)
    q, k, _ = rand_qkv(rng, 128, 0, 4, 1, 8, scale_q=2.0)
    c = rng.standard_normal(8) * 3
    kb1 = oracle_mod.pool(k, 16)
    kb2 = oracle_mod.pool(k + c, 16)
    r1 = oracle_mod.score_rows(q, 0, 1, 16, 0.5, kb1, np.arange(8))
    r2 = oracle_mod.score_rows(q, 0, 1, 16, 0.5, kb2, np.arange(8))
    for a, b in zip(r1, r2):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=0)
    # a shift that differs per query block is NOT cancelled in general (control)
    k3 = k.copy()
    k3[:16] += c
    kb3 = oracle_mod.pool(k3, 16)
    r3 = oracle_mod.score_rows(q, 0, 1, 16, 0.5, kb3, np.arange(8))
    assert max(np.abs(a - b).max() for a, b in zip(r1, r3)) > 1e-3


def test_score_invariant_to_query_and_head_permutation(oracle_mod):
    rng = np.random.default_rng(4)
    q, k, _ = rand_qkv(rng, 64, 0, 4, 1, 8, scale_q=2.0)
    kbar = oracle_mod.pool(k, 16)
    base = oracle_mod.score_rows(q, 0, 1, 16, 0.5, kbar, [3])[0]
    q2 = q.copy()
    q2[48:64] = q2[48:64][rng.permutation(16)]
    q2[48:64] = q2[48:64][:, [2, 0, 3, 1]]
    got = oracle_mod.score_rows(q2, 0, 1, 16, 0.5, kbar, [3])[0]
    np.testing.assert_allclose(got, base, rtol=1e-13)


def test_head_union_scores(oracle_mod):
    """The union-of-heads score reading: with one head per group it is the
    packed score; it does not depend on the order of the group's heads; every
    head's own normalised row lies under it and touches it at its maximum;
    each row peaks at exactly 1."""
    rng = np.random.default_rng(14)
    B, start, hkv, g, d = 16, 32, 2, 3, 8
    q = rng.normal(size=(70, hkv * g, d))
    k = rng.normal(size=(start + 70, hkv, d))
    kbar = oracle_mod.pool(k, B)
    nqb = -(-70 // B)
    rows = list(range(nqb * hkv))
    union = oracle_mod.score_rows_head_union(q, start, hkv, B, 0.3, kbar, rows)
    # g = 1: the packed score of the single head
    for hh in range(hkv * g):
        h = hh // g
        one = oracle_mod.score_rows_head_union(q[:, hh:hh + 1], start, 1, B, 0.3, kbar[:, h:h + 1], range(nqb))
        packed = oracle_mod.score_rows(q[:, hh:hh + 1], start, 1, B, 0.3, kbar[:, h:h + 1], range(nqb))
        for a_, b_ in zip(one, packed):
            np.testing.assert_array_equal(a_, b_)
    perm = np.concatenate([h * g + rng.permutation(g) for h in range(hkv)])
    union_p = oracle_mod.score_rows_head_union(q[:, perm], start, hkv, B, 0.3, kbar, rows)
    for r, (u, up) in enumerate(zip(union, union_p)):
        np.testing.assert_array_equal(u, up)
        assert u.max() == 1.0
        il, h = divmod(r, hkv)
        for hh in range(h * g, (h + 1) * g):
            own = oracle_mod.score_rows(q[:, hh:hh + 1], start, 1, B, 0.3, kbar[:, h:h + 1], [il])[0]
            assert np.all(own <= u) and u[np.argmax(own)] == 1.0


# ----------------------------------------------------------------------------
# selection
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("alpha", [0.0, 0.1, 0.5, 1.0])
def test_select_rule_and_invariants(oracle_mod, alpha):
    rng = np.random.default_rng(5)
    B, sink, local = 128, 256, 512
    for I in [0, 1, 3, 4, 9, 40]:
        s = rng.random(I + 1) ** 4
        s /= s.max()
        keep, flag = oracle_mod.select_row(s, I, alpha, B, sink, local)
        for J in range(I + 1):
            want = s[J] >= alpha or J < 2 or J >= I - 3
            assert keep[J] == want, (I, J)
        # sink, local and the diagonal are always present; nothing beyond I
        assert keep[:min(2, I + 1)].all() and keep[max(0, I - 3):].all()
        assert len(keep) == I + 1


def test_select_threshold_is_inclusive_and_flags_band(oracle_mod):
    s = np.array([1.0, 0.5, 0.1, 0.1 * (1 - 5e-5), 0.1 * (1 - 2e-4), 0.05, 0.3, 0.2, 0.2, 0.2])
    keep, flag = oracle_mod.select_row(s, 9, 0.1, 128, 0, 0)
    # local=0 -> no local blocks; sink=0 -> none; only J >= I - 0 + 1 = 10 (none)
    assert list(keep) == [True, True, True, False, False, False, True, True, True, True]
    assert list(flag) == [False, False, True, True, False, False, False, False, False, False]


@pytest.mark.parametrize("k", [1, 3, 7, 40, 55])
def test_topk_keeps_the_k_highest_lowest_index_first(oracle_mod, k):
    """Top-k (V1 summary 4.4 ablation), no forced blocks: exactly min(k, n)
    blocks; every kept score >= every dropped one; among equal scores at the
    boundary the kept ones have the lower indices."""
    rng = np.random.default_rng(11)
    for I in [0, 5, 40]:
        s = np.round(rng.random(I + 1), 1) + 0.05      # many ties on a 0.1 grid
        keep, flag = oracle_mod.select_row(s, I, 0.1, 128, 0, 0, rule=1, top_k=k)
        n = I + 1
        assert keep.sum() == min(k, n)
        if keep.all():
            continue
        assert s[keep].min() >= s[~keep].max()
        t = s[keep].min()
        tied = np.nonzero(s == t)[0]
        kept_tied, dropped_tied = tied[keep[tied]], tied[~keep[tied]]
        if len(dropped_tied):
            assert kept_tied.max() < dropped_tied.min()
        assert flag[tied].all()                          # the boundary value is flagged


@pytest.mark.parametrize("p", [1e-6, 0.3, 0.6, 0.9, 1.0])
def test_topp_keeps_the_smallest_top_set_holding_p_of_the_mass(oracle_mod, p):
    """Top-p (V1 summary 4.4 ablation), no forced blocks: the kept set holds
    at least p of the row's mass, dropping its lowest value (with its ties)
    falls short, and every kept score >= every dropped one."""
    rng = np.random.default_rng(12)
    for I in [0, 6, 60]:
        s = rng.random(I + 1) ** 3 + 1e-3
        keep, flag = oracle_mod.select_row(s, I, 0.1, 128, 0, 0, rule=2, top_p=p)
        total = s.sum()
        assert s[keep].sum() >= p * total * (1 - 1e-12)
        t = s[keep].min()
        assert s[s > t].sum() < p * total
        if not keep.all():
            assert t >= s[~keep].max()
        if p == 1.0:
            assert keep.all()
        if p == 1e-6:
            assert keep.sum() == np.sum(s == s.max())


def test_topk_topp_keep_sink_and_local_blocks(oracle_mod):
    rng = np.random.default_rng(13)
    I = 30
    s = rng.random(I + 1)
    for rule, kw in ((1, dict(top_k=2)), (2, dict(top_p=0.2))):
        keep, _ = oracle_mod.select_row(s, I, 0.1, 128, 256, 512, rule=rule, **kw)
        alone, _ = oracle_mod.select_row(s, I, 0.1, 128, 0, 0, rule=rule, **kw)
        forced = np.zeros(I + 1, bool)
        forced[:2] = True
        forced[I - 3:] = True
        assert np.array_equal(keep, alone | forced)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def test_alpha_zero_equals_dense_causal_softmax(oracle_mod):
    rng = np.random.default_rng(6)
    B, start, scale = 32, 0, 1 / math.sqrt(16)
    q, k, v = rand_qkv(rng, 200, start, 4, 2, 16)
    nqb, nkb = -(-200 // B), -(-200 // B)
    keep = np.zeros((nqb, 2, nkb), np.uint8)
    for i in range(nqb):
        keep[i, :, :i + 1] = 1
    o, lse = all_rows(oracle_mod, q, k, v, start, B, scale, keep, True)
    ro, rl = dense_causal_softmax(q, k, v, start, scale)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)
    o2, l2 = all_rows(oracle_mod, q, k, v, start, B, scale, None, False)
    np.testing.assert_allclose(o2, ro, rtol=0, atol=1e-12)


def test_dense_with_chunk_offset(oracle_mod):
    rng = np.random.default_rng(7)
    B, start, scale = 32, 96, 0.2
    q, k, v = rand_qkv(rng, 70, start, 2, 1, 8)
    o, lse = all_rows(oracle_mod, q, k, v, start, B, scale, None, True)
    ro, rl = dense_causal_softmax(q, k, v, start, scale)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)


def test_mean_correction_exact_for_constant_key_blocks(oracle_mod):
    """If all keys of each skipped block are equal, e^{q.kbar} = e^{q.k} for
    every token and n * vbar = sum v: the corrected result is exact."""
    rng = np.random.default_rng(8)
    B, L, scale = 32, 256, 0.3
    nb = L // B
    kb = rng.standard_normal((nb, 1, 8)) * 2
    k = np.repeat(kb, B, axis=0)
    q = rng.standard_normal((L, 2, 8))
    v = rng.standard_normal((L, 1, 8))
    keep = np.zeros((nb, 1, nb), np.uint8)
    for i in range(nb):
        keep[i, 0, i] = 1                 # only the diagonal is computed exactly
        if i >= 3:
            keep[i, 0, 1] = 1
    o, lse = all_rows(oracle_mod, q, k, v, 0, B, scale, keep, True)
    ro, rl = dense_causal_softmax(q, k, v, 0, scale)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)
    # without correction it is not exact (control)
    o3, _ = all_rows(oracle_mod, q, k, v, 0, B, scale, keep, False)
    assert np.abs(o3 - ro).max() > 1e-2


def bruteforce_mean_tokens(q, k, v, start, B, scale, keep, mean_corr):
    """Token-level brute force: the key set of a query is every token of its
    kept blocks (causal) plus, for each skipped earlier block, one "mean
    token" (np.mean of the block's keys/values) carrying log(n) as a bias."""
    lq, hq, d = q.shape
    lk, hkv, _ = k.shape
    g = hq // hkv
    o = np.zeros((lq, hq, d))
    for i in range(lq):
        p = start + i
        I = p // B
        il = I - start // B
        for h in range(hq):
            hk = h // g
            keys, vals, bias = [], [], []
            for J in range(I + 1):
                blk = slice(J * B, min((J + 1) * B, lk))
                if keep[il, hk, J]:
                    for t in range(J * B, min((J + 1) * B, p + 1)):
                        keys.append(k[t, hk]); vals.append(v[t, hk]); bias.append(0.0)
                elif mean_corr and J < I:
                    n = min(B, lk - J * B)
                    keys.append(k[blk, hk].mean(axis=0)); vals.append(v[blk, hk].mean(axis=0))
                    bias.append(math.log(n))
            logits = scale * np.array(keys) @ q[i, h] + np.array(bias)
            w = np.exp(logits - logits.max())
            o[i, h] = w @ np.array(vals) / w.sum()
    return o


@pytest.mark.parametrize("mean_corr", [True, False])
def test_token_level_bruteforce_small(oracle_mod, mean_corr):
    """L <= 512 with B=32, sink=32, local=64 so that blocks really are skipped."""
    rng = np.random.default_rng(9)
    B, sink, local, alpha, scale = 32, 32, 64, 0.3, 1 / math.sqrt(16)
    L, hq, hkv, d = 320, 4, 2, 16
    q, k, v = rand_qkv(rng, L, 0, hq, hkv, d, scale_q=0.5)
    u = rng.standard_normal((L // B, hkv, d))
    k += np.repeat(u, B, axis=0)                     # block-coherent keys
    for i in range(L // B):                          # each query block aims at one key block
        j = rng.integers(0, i + 1)
        q[i * B:(i + 1) * B] += 0.5 * np.repeat(u[j], hq // hkv, axis=0)[None]
    kbar = oracle_mod.pool(k, B)
    nqb = L // B
    rows = oracle_mod.score_rows(q, 0, hkv, B, scale, kbar, np.arange(nqb * hkv))
    keep = np.zeros((nqb, hkv, nqb), np.uint8)
    for r, s in enumerate(rows):
        i, h = divmod(r, hkv)
        keep[i, h, :i + 1] = oracle_mod.select_row(s, i, alpha, B, sink, local)[0]
    assert keep.sum() < 0.9 * hkv * nqb * (nqb + 1) / 2    # something is skipped
    o, _ = all_rows(oracle_mod, q, k, v, 0, B, scale, keep, mean_corr)
    ref = bruteforce_mean_tokens(q, k, v, 0, B, scale, keep, mean_corr)
    np.testing.assert_allclose(o, ref, atol=1e-12)


def test_output_linear_in_values(oracle_mod):
    """Softmax weights (including the mean tokens) sum to one: O(aV + c) =
    a O(V) + c."""
    rng = np.random.default_rng(10)
    B, L = 32, 160
    q, k, v = rand_qkv(rng, L, 0, 2, 1, 8, scale_q=3.0)
    keep = np.zeros((5, 1, 5), np.uint8)
    for i in range(5):
        keep[i, 0, i] = 1
        keep[i, 0, 0] = 1
    o1, l1 = all_rows(oracle_mod, q, k, v, 0, B, 0.4, keep, True)
    c = rng.standard_normal(8)
    o2, l2 = all_rows(oracle_mod, q, k, 2.5 * v + c, 0, B, 0.4, keep, True)
    np.testing.assert_allclose(o2, 2.5 * o1 + c, atol=1e-12)
    np.testing.assert_allclose(l2, l1, atol=1e-13)


def test_mean_correction_off_all_kept_equals_dense(oracle_mod):
    rng = np.random.default_rng(11)
    q, k, v = rand_qkv(rng, 96, 0, 2, 2, 8)
    nb = 3
    keep = np.zeros((nb, 2, nb), np.uint8)
    for i in range(nb):
        keep[i, :, :i + 1] = 1
    a, _ = all_rows(oracle_mod, q, k, v, 0, 32, 0.3, keep, True)
    b, _ = all_rows(oracle_mod, q, k, v, 0, 32, 0.3, keep, False)
    np.testing.assert_array_equal(a, b)


# ----------------------------------------------------------------------------
# formats and layouts
# ----------------------------------------------------------------------------

def test_e4m3_decoding_matches_known_codes_and_torch(oracle_mod):
    codes = np.array([0x00, 0x01, 0x08, 0x38, 0x40, 0x7E, 0xB8, 0xFE, 0x7F], np.uint8)
    got = oracle_mod.decode_e4m3(codes)
    want = [0.0, 2.0 ** -9, 2.0 ** -6, 1.0, 2.0, 448.0, -1.0, -448.0]
    np.testing.assert_array_equal(got[:8], want)
    assert np.isnan(got[8])
    torch = pytest.importorskip("torch")
    allc = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(allc).view(torch.float8_e4m3fn).float().double().numpy()
    mine = oracle_mod.decode_e4m3(allc)
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])
    assert np.all(np.isnan(mine[~ok]))


def test_page_permutation_leaves_gathered_kv_unchanged(oracle_mod):
    from block_sparse_long_fp_gb300 import synth
    a = synth.make_case(synth.Spec("t", [(300, 0)], 2, 1, page_size=16, layout="contiguous",
                                   n_needles=1, config_id=91), threads=2)
    b = synth.make_case(synth.Spec("t", [(300, 0)], 2, 1, page_size=16, layout="shuffled",
                                   n_needles=1, config_id=91), threads=2)
    assert not np.array_equal(a.block_table, b.block_table)
    ka, va = oracle_mod.request_kv(a, 0)
    kb, vb = oracle_mod.request_kv(b, 0)
    np.testing.assert_array_equal(ka, kb)
    np.testing.assert_array_equal(va, vb)


def test_dense_mask_and_csr_sizes_closed_form():
    """Index sizes quoted by the V2 popular article (CSR index section): a
    dense per-(query block, key block, query head) byte mask at 128K with 32
    query heads is 1024 * 1024 * 32 B = 32 MiB, whatever the density."""
    nb = 131072 // 128
    assert nb * nb * 32 == 32 * 2 ** 20
    # our per-kv-head int32 CSR at 5% of the causal pairs, 4 kv heads
    pairs = nb * (nb + 1) // 2 * 4
    csr = int(0.05 * pairs) * 4 + (nb * 4 + 1) * 4
    assert csr < 32 * 2 ** 20 / 50


def test_skipped_diagonal_is_not_mean_corrected(oracle_mod):
    """Only skipped blocks strictly before the query block get a mean term:
    the diagonal block is partly in the future of its queries, so its mean
    would leak future keys."""
    rng = np.random.default_rng(12)
    B, L, scale = 16, 96, 0.35
    q, k, v = rand_qkv(rng, L, 0, 2, 1, 8, scale_q=1.5)
    nb = L // B
    keep = (rng.random((nb, 1, nb)) < 0.5).astype(np.uint8)
    keep[:, :, 0] = 1
    for i in range(nb):
        keep[i, 0, i + 1:] = 0
    keep[3, 0, 3] = 0                                 # a skipped diagonal
    o, _ = all_rows(oracle_mod, q, k, v, 0, B, scale, keep, True)
    ref = bruteforce_mean_tokens(q, k, v, 0, B, scale, keep, True)
    np.testing.assert_allclose(o, ref, atol=1e-12)
