"""The seeded input generator: shapes, paging, determinism, formats."""
import numpy as np
import pytest

from block_sparse_long_fp_gb300 import synth


def small(layout="shuffled", dtype="bf16", reqs=((300, 0), (200, 128)), ps=16):
    return synth.Spec("t", list(reqs), 4, 2, d=128, page_size=ps, layout=layout, dtype=dtype,
                      n_needles=2, config_id=90)


@pytest.mark.parametrize("layout", ["contiguous", "shuffled", "interleaved"])
def test_layout_and_descriptors(layout):
    c = synth.make_case(small(layout), threads=2)
    assert c.q.shape == (500, 4, 128) and c.q.dtype == np.uint16
    assert list(c.cu_seqlens_q) == [0, 300, 500]
    assert list(c.seqlens_k) == [300, 328]
    assert list(c.q_start_pos) == [0, 128]
    npg = [-(-300 // 16), -(-328 // 16)]
    assert c.k_cache.shape == (sum(npg), 16, 2, 128)
    used = np.concatenate([c.block_table[r, :npg[r]] for r in range(2)])
    assert sorted(used.tolist()) == list(range(sum(npg)))        # a permutation of the pool
    assert np.all(c.block_table[0, npg[0]:] == -1)


def test_deterministic():
    a = synth.make_case(small(), threads=1)
    b = synth.make_case(small(), threads=3)
    np.testing.assert_array_equal(a.q, b.q)
    np.testing.assert_array_equal(a.k_cache, b.k_cache)
    np.testing.assert_array_equal(a.block_table, b.block_table)


def test_e4m3_scales_cover_range():
    c = synth.make_case(small(dtype="e4m3"), threads=2)
    assert c.q.dtype == np.uint8 and c.k_cache.dtype == np.uint8
    assert c.q_scale.shape == (4,) and c.k_scale.shape == (2,)
    import torch
    qf = torch.from_numpy(c.q).view(torch.float8_e4m3fn).float().numpy()
    assert np.isfinite(qf).all() and np.abs(qf).max() == 448.0


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-3], np.float32)
    b = synth.to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(b)
    np.testing.assert_array_equal(back[:4], [1.0, 1.0, 1.0 + 2 ** -6, -2.5])
    assert abs(back[4] - 1e-3) <= 1e-3 * 2 ** -8


def test_workload_specs():
    s3 = synth.config_spec(3)
    assert (s3.total_q, s3.h_q, s3.h_kv, s3.page_size) == (131072, 32, 4, 64)
    s4 = synth.config_spec(4)
    assert s4.total_q == 129024 and s4.total_k == 169984
    assert (8192, 40960) in s4.requests
