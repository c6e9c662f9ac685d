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
