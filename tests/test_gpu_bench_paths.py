"""The bench's two ways of running one step compute the same outputs: the
per-phase CUDA graphs it times, and the end-to-end path (per-layer calls
through the public API, with the inputs copied from host memory on a copy
stream while the previous layer computes)."""
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
    path = bench.Path(workloads.by_name("tiny"), 0, dev)
    path.capture()
    path.step()
    torch.cuda.synchronize()
    outs = (path.o_sp, path.l_sp, path.o_de, path.l_de)
    ref = [t.clone() for t in outs]
    for t in outs:
        t.zero_()
    e2e = bench.run_e2e(path, 2, 1)
    torch.cuda.synchronize()
    for a, b in zip(ref, outs):
        assert torch.equal(a, b)
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
