"""newton_schulz_noalloc: one unit's Newton-Schulz with no device allocation,
for callers that cannot call cudaMalloc -- code inside a framework whose
caching allocator already owns all device memory, or a latency-critical path
that must not take the allocation lock or the synchronisation an allocation
can bring.

Each call's v is checked against the fp32 oracle (the Newton-Schulz
tolerance of the other tests) and, bit for bit, against the existing entry
point (muon_update_units' Newton-Schulz stage, which runs the same kernels)
on the same u.  The calls run back
to back in decreasing size, so a later, smaller unit meets whatever the
built-in scratch array kept from a larger one; every call after the first
must leave the device's free memory unchanged.  Collected last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import muon as OM  # noqa: E402

from muon_parity import NS_TOL  # noqa: E402

pytestmark = pytest.mark.gpu


# decreasing size: the largest accepted shapes first (both orientations), then
# a transposed unit with a padded Gram size, a head, a unit whose rows (72) and
# cols (1000) are multiples of neither 32 nor 64, and a small head
CASES = [(8192, 128, 51), (128, 8192, 52), (1024, 96, 53), (128, 4096, 54), (72, 1000, 55), (64, 256, 56)]


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


def test_noalloc_matches_oracle_and_existing_entry_point(hm, dev):
    inputs = [(rows, cols) + _existing_path(hm, dev, rows, cols, seed) for rows, cols, seed in CASES]
    for call, (rows, cols, u, v_ref, hp) in enumerate(inputs):
        u_dev = u.to(dev).contiguous()
        v_out = torch.full((rows * cols,), float("nan"), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info(dev)[0]
        hm.newton_schulz_noalloc(u_dev.data_ptr(), rows, cols, v_out.data_ptr(), hp)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info(dev)[0]
        assert hm.hm_device_error() == 0
        v = v_out.cpu().numpy().astype(np.float64)
        assert np.isfinite(v).all(), f"call {call} ({rows}x{cols}): v not fully written"
        # against the fp32 oracle, run on the same bf16 u
        u32 = OM.bf16_bits_to_f32(u.numpy().view(np.uint16)).reshape(rows, cols)
        ref = OM.newton_schulz(u32, hp.ns_steps, hp.ns_a, hp.ns_b, hp.ns_c, hp.eps).ravel()
        err = np.linalg.norm(v - ref) / np.linalg.norm(ref)
        assert err <= NS_TOL, f"call {call} ({rows}x{cols}): rel err vs oracle {err:.3e}"
        # against the existing entry point: the same kernels on the same u, bit for bit
        assert np.array_equal(v.astype(np.float32).view(np.uint32), v_ref.view(np.uint32)), (
            f"call {call} ({rows}x{cols}): v differs from muon_update_units")
        if call > 0:
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
