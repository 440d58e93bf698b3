"""newton_schulz_noalloc: one unit's Newton-Schulz with no device allocation,
for callers that cannot call cudaMalloc (a stream capture in progress, an
allocator that already owns all device memory, a latency-critical path).

Its output must match the existing path (the Newton-Schulz stage of
muon_update_units) on the same unit, within the Newton-Schulz tolerance the
other tests use, on two calls in a row; the second call must leave the
device's free memory unchanged (the first call on a device may load the
library module that holds the built-in scratch).  Collected last so that a
run stopping at the first failure has already run every other test."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402

from muon_parity import NS_TOL  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(hm):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _existing_path(hm, dev, rows, cols, seed):
    """u and v of one unit through muon_update_units (f0 then Newton-Schulz)."""
    from head_muon_mxfp8_gb300.session import MuonSession, muon_hparams
    cfg = workloads.scaled_muon("one_unit", [(rows, cols, None)], so=2, sw=1, sg=1)
    g = workloads.gaussian(rows * cols, 1e-3, seed)
    s = MuonSession.from_config(cfg, device=dev)
    s.load("g", g)
    s.load("m", np.zeros_like(g))
    s.load("w", np.zeros_like(g))
    hp = muon_hparams(cfg.muon)
    s.run(hp, hm.HM_STAGE_F0 | hm.HM_STAGE_GATHER | hm.HM_STAGE_NS)
    torch.cuda.synchronize()
    u = s.fetch("u")
    v = s.unit_v(0).numpy()
    s.close()
    return u, v, hp


def test_noalloc_matches_existing_entry_point_two_calls(hm, dev):
    # a 128 x 4096 head, then a transposed 1024 x 96 unit (padded Gram size)
    for call, (rows, cols, seed) in enumerate([(128, 4096, 31), (1024, 96, 32)]):
        u, v_ref, hp = _existing_path(hm, dev, rows, cols, seed)
        u_dev = u.to(dev).contiguous()
        v_out = torch.full((rows * cols,), float("nan"), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info(dev)[0]
        hm.newton_schulz_noalloc(u_dev.data_ptr(), rows, cols, v_out.data_ptr(), hp)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info(dev)[0]
        assert hm.hm_device_error() == 0
        v = v_out.cpu().numpy().astype(np.float64)
        err = np.linalg.norm(v - v_ref) / np.linalg.norm(v_ref)
        assert err <= NS_TOL, f"call {call}: rel err {err:.3e}"
        if call == 1:
            assert free_after == free_before


def test_noalloc_rejects_sizes_beyond_its_scratch(hm, dev):
    from head_muon_mxfp8_gb300.session import muon_hparams
    hp = muon_hparams(workloads.MuonHparams())
    L = hm.lib()
    import ctypes as C
    buf = torch.zeros(1 << 20, dtype=torch.float32, device=dev)
    p = C.c_void_p(buf.data_ptr())
    assert L.newton_schulz_noalloc(p, 129, 256, p, C.byref(hp), None) == hm.HM_ERR_WORKSPACE
    assert L.newton_schulz_noalloc(p, 64, 8193 + 7, p, C.byref(hp), None) == hm.HM_ERR_WORKSPACE
    assert L.newton_schulz_noalloc(p, 3, 5, p, C.byref(hp), None) == hm.HM_ERR_ALIGN
