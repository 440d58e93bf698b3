"""GPU parity of the emulated outer reduce-scatter (FP32, BF16 and BF16-SR
node partials, accumulate on / off) against the oracle, bit-exact, written
into ragged rank segments."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import gradient as OG  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(hm):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.mark.parametrize("name,P,L", [("tiny_ragged", 8, 4), ("mixed", 4, 1), ("mixed", 6, 3)])
@pytest.mark.parametrize("mode", ["fp32", "bf16", "bf16_sr"])
def test_reduce_scatter_grad(hm, dev, name, P, L, mode):
    from head_muon_mxfp8_gb300.session import MuonSession
    cfg = workloads.get(name)
    n = cfg.numel
    parts = workloads.gaussian((P, n), 1e-3, seed=31)
    g0 = workloads.gaussian(n, 1e-3, seed=32)
    code = {"fp32": hm.HM_RS_FP32, "bf16": hm.HM_RS_BF16, "bf16_sr": hm.HM_RS_BF16_SR}[mode]
    seed, offset = 0x123456789ABC, 77
    s = MuonSession.from_config(cfg, device=dev)
    pt = torch.from_numpy(parts).to(dev)
    for accumulate in (False, True):
        s.load("g", g0)
        hm.reduce_scatter_grad(s.chain, pt.data_ptr(), P, L, s.g.data_ptr(), code, accumulate, seed, offset)
        torch.cuda.synchronize()
        got = s.fetch("g").numpy()
        want = OG.reduce_scatter(parts, L, mode, seed=seed, offset=offset)
        if accumulate:
            want = (g0 + want).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert s.canary_intact()["g"]
    s.close()


def test_reduce_scatter_rejects_partial_nodes(hm, dev):
    import ctypes as C
    ch = hm.shard_chain(1024, 2, 1, 1)
    buf = torch.zeros(4096, device=dev)
    st = hm.lib().reduce_scatter_grad(C.c_void_p(ch), C.c_void_p(buf.data_ptr()), 3, 2, C.c_void_p(buf.data_ptr()),
                                      0, 0, 0, 0, None)
    assert st == hm.HM_ERR_GEOMETRY
    hm.chain_destroy(ch)
