"""The update phase captured in a CUDA graph.

muon_update_units launches only kernels on the caller's stream (cluster
launches included) and allocates nothing, so a caller can capture a whole
fused update once and replay it: no per-kernel launch cost, which is what
bounds small workloads.  Two replays must leave exactly the state two eager
calls leave (momentum carries over between them), and the device error
word must stay clear."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(hm):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _state(s):
    return {f: s.fetch(f).numpy().copy() for f in ("w", "m", "q", "s")}


@pytest.mark.parametrize("name,step", [("tiny", False), ("mixed", False), ("tiny", True), ("mixed", True)])
def test_fused_update_replayed_from_a_cuda_graph_equals_eager(hm, dev, name, step):
    from head_muon_mxfp8_gb300.session import MuonSession, muon_hparams
    stages = hm.HM_STAGE_STEP if step else hm.HM_STAGE_ALL_FUSED
    cfg = workloads.get(name)
    data = workloads.generate(cfg, seed=17)
    hp = muon_hparams(cfg.muon)

    eager = MuonSession.from_config(cfg, device=dev)
    eager.load("w", data["w"])
    eager.load("g", data["g"])
    eager.load("m", np.zeros_like(data["w"]))
    for _ in range(2):
        eager.run(hp, stages)
    torch.cuda.synchronize()
    want = _state(eager)
    eager.close()

    s = MuonSession.from_config(cfg, device=dev)
    side = torch.cuda.Stream(device=dev)
    # one eager call on the capture stream first: first-use setup (kernel
    # attributes, the f2 step table) happens outside the capture
    s.load("m", np.zeros_like(data["w"]))
    s.run(hp, stages, side)
    torch.cuda.synchronize()
    s.load("w", data["w"])
    s.load("g", data["g"])
    s.load("m", np.zeros_like(data["w"]))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    before = hm.hm_kernel_launches()
    with torch.cuda.graph(graph, stream=side):
        s.run(hp, stages, side)
    captured = hm.hm_kernel_launches() - before
    assert captured > 0
    torch.cuda.synchronize()
    # capture records work without running it: the state is still the input
    assert np.array_equal(s.fetch("m").numpy(), np.zeros_like(data["w"]))
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert hm.hm_device_error() == 0
    got = _state(s)
    for f in want:
        assert np.array_equal(got[f], want[f]), f
    assert all(s.canary_intact().values())
    s.close()
