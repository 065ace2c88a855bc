"""The bench's two ways of running one decode step compute the same outputs:
the CUDA graph of the per-layer calls it times, and the end-to-end path (the
C-ABI entry point called once per layer, with the decode queries copied from
pinned host memory every step)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_e2e_path_matches_graph_step():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    import workloads
    from sparse_kv_decode_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    D = bench.Decode(workloads.by_name("tiny"), dev)
    D.prefill((0,))
    g = bench.capture(lambda: D.sparse_step(0))
    g.replay()
    torch.cuda.synchronize()
    ref = [D.o_sp.clone(), D.l_sp.clone()]
    D.o_sp.zero_()
    D.l_sp.zero_()
    e2e = bench.run_e2e(D, 0, 2, 1)
    torch.cuda.synchronize()
    assert torch.equal(ref[0], D.o_sp) and torch.equal(ref[1], D.l_sp)
    assert e2e["h2d_bytes_per_step"] == D.L * D.B * D.Hq * D.d * 2
    assert e2e["d2h_bytes_per_step"] == D.L * D.B * D.Hq * (D.d * 2 + 4)
    for ws in D.workspaces():
        assert D.sk.workspace_status(ws) == 0
