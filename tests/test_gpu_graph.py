"""The stages captured in a CUDA graph and replayed on new inputs: each replay
gives what a direct call on the same inputs gives."""
import numpy as np
import pytest

from block_sparse_long_fp_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_fp_gb300 import build
    build.build()


def test_select_replayed_from_a_graph_matches_direct_calls():
    """fp_select scans the kept counts with a decoupled look-back whose states
    outlive the call; a replay must not read the states of the replay before.
    Two score maps with different kept counts alternate in the captured
    buffer, and every replay's CSR equals a direct call's, bit for bit."""
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    spec = synth.Spec("graph-select", [(16384, 0), (6000, 2048)], 16, 8, page_size=64, layout="shuffled",
                      dtype="bf16", n_needles=2, logit_scale=4.0, config_id=91)
    layer = fprefill.layer_from_case(synth.make_case(spec))
    _, _, score = layer.discover()
    maps = [score.clone(), score.clamp_min(0).sqrt(), score.clone()]   # the square root keeps more blocks
    buf = maps[0].clone()
    row_ptr, col_idx, nnz = layer.select(buf)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.select(buf, row_ptr, col_idx, nnz)
    counts = []
    for m in maps + maps:
        buf.copy_(m)
        graph.replay()
        torch.cuda.synchronize()
        rp, ci, nz = layer.select(m)
        torch.cuda.synchronize()
        n = int(nz.item())
        counts.append(n)
        assert int(nnz.item()) == n
        assert torch.equal(row_ptr, rp)
        assert torch.equal(col_idx[:n], ci[:n])
    assert len(set(counts)) == 2
    assert layer.device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_layer_replayed_from_a_graph_matches_direct_calls(dtype):
    """fp_discover, fp_select and fp_sparse_attn captured once into a CUDA
    graph (buffers fixed), then replayed after the queries change in place:
    each replay's index and output equal those of direct calls on the same
    queries, bit for bit."""
    import torch
    from block_sparse_long_fp_gb300 import fprefill
    spec = synth.Spec("graph-layer", [(8192, 0), (3000, 1024)], 8, 2, page_size=64, layout="shuffled",
                      dtype=dtype, n_needles=2, logit_scale=6.0, config_id=93)
    layer = fprefill.layer_from_case(synth.make_case(spec))
    q = layer.q_scale if dtype == "e4m3" else layer.q      # e4m3: the per-head query scales

    def direct():
        km, vm, sc = layer.discover()
        rp, ci, nz = layer.select(sc)
        out, _ = layer.sparse_attn(rp, ci, km, vm, want_lse=False)
        torch.cuda.synchronize()
        return rp.clone(), ci[:int(nz.item())].clone(), out.clone()

    km, vm, sc = layer.discover()                          # the buffers the graph keeps
    rp, ci, nz = layer.select(sc)
    out, _ = layer.sparse_attn(rp, ci, km, vm, want_lse=False)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.discover(km, vm, sc)
        layer.select(sc, rp, ci, nz)
        layer.sparse_attn(rp, ci, km, vm, out=out, want_lse=False)
    densities = []
    for factor in (1.0, 2.0, 0.25):
        q.mul_(factor)
        graph.replay()
        torch.cuda.synchronize()
        g_rp, g_ci, g_out = rp.clone(), ci[:int(nz.item())].clone(), out.clone()
        d_rp, d_ci, d_out = direct()
        assert torch.equal(g_rp, d_rp)
        assert torch.equal(g_ci, d_ci)
        assert torch.equal(g_out, d_out)
        densities.append(int(nz.item()))
    assert len(set(densities)) > 1
    assert layer.device_status() == 0
