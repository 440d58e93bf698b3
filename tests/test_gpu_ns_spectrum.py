"""Spectral validity of the GPU's Newton-Schulz output.

Many bf16 results lie within the relative Frobenius bound of the fp32
oracle; what every correct one shares is how the iteration acts on singular
values.  For u = U diag(sigma) V^T and sigma_hat = sigma / (||u||_F + eps),
the exact iteration gives U diag(p^5(sigma_hat)) V^T with
p(s) = a s + b s^3 + c s^5 (SS-HSDP section 3.1, example EG1: f1 applies
Newton-Schulz to the whole unit; coefficients and step count as configured).
So the GPU's v, expressed in the singular bases of its own u, must be
diagonal up to bf16 noise, its diagonal must follow p^5(sigma_hat_i) to
within 0.03, and every singular value of v must lie in the band
[0.68 - 0.02, max_i p^5(sigma_hat_i) + 0.02] (the quintic maps every
sigma_hat >= 0.006 into [0.6818, 1.1344]; these shapes stay above that).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import muon as OM  # noqa: E402

pytestmark = pytest.mark.gpu

SHAPES = [(64, 256, None), (256, 64, None), (128, 512, None), (384, 640, None), (640, 384, None)]


@pytest.fixture(scope="module")
def dev(hm):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def test_newton_schulz_acts_on_singular_values(hm, dev):
    from head_muon_mxfp8_gb300.session import MuonSession, muon_hparams
    cfg = workloads.scaled_muon("spectrum", SHAPES, so=4, sw=2, sg=2)
    g = workloads.gaussian(cfg.numel, 1e-3, 41)
    s = MuonSession.from_config(cfg, device=dev)
    s.load("g", g)
    s.load("m", np.zeros_like(g))
    s.load("w", np.zeros_like(g))
    h = cfg.muon
    hp = muon_hparams(h)
    s.run(hp, hm.HM_STAGE_F0 | hm.HM_STAGE_GATHER | hm.HM_STAGE_NS)
    torch.cuda.synchronize()
    assert hm.hm_device_error() == 0
    u_all = OM.bf16_bits_to_f32(s.fetch("u").numpy().view(np.uint16)).astype(np.float64)
    for i, un in enumerate(cfg.units):
        u = u_all[un.offset:un.offset + un.numel].reshape(un.rows, un.cols)
        v = s.unit_v(i).numpy().astype(np.float64).reshape(un.rows, un.cols)
        U, sig, Vt = np.linalg.svd(u, full_matrices=False)
        sh = sig / (np.linalg.norm(u) + hp.eps)
        want = OM.ns_polynomial(sh, hp.ns_steps, hp.ns_a, hp.ns_b, hp.ns_c)
        assert sh.min() >= 0.006, "shape chosen outside the band's premise"
        proj = U.T @ v @ Vt.T                          # v in u's singular bases
        diag = np.diag(proj)
        off = proj - np.diag(diag)
        assert np.max(np.abs(diag - want)) <= 0.03, f"unit {i} ({un.rows}x{un.cols})"
        assert np.linalg.norm(off) <= 0.03 * np.linalg.norm(diag), f"unit {i}: off-diagonal part"
        sv = np.linalg.svd(v, compute_uv=False)
        assert sv.min() >= 0.68 - 0.02 and sv.max() <= want.max() + 0.02, (
            f"unit {i}: singular values [{sv.min():.4f}, {sv.max():.4f}], p^5 max {want.max():.4f}")
    s.close()
