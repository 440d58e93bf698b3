"""Pins for oracle.muon (f0, f1, f2): library routines, closed forms and
identities, plus planted-mistake checks showing the closed-form pin catches
plausible errors in the iteration."""
import numpy as np
import pytest
import torch

from oracle import muon as M

NS = dict(steps=5, a=3.4445, b=-4.7750, c=2.0315, eps=1e-7)


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(1e-3),
        rng.standard_normal(100000).astype(np.float32) * np.float32(1e4),
    ])
    # exact ties: low 16 bits = 0x8000 with both parities of bit 16
    hi = rng.integers(0, 0x7F7F, 1000).astype(np.uint32)
    ties = ((hi << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.array([0.0, -0.0], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (M.bf16_rne_bits(x) == ref).all()
    back = M.bf16_bits_to_f32(ref)
    assert (back == torch.from_numpy(x).to(torch.bfloat16).float().numpy()).all()


def test_momentum_float32_ops_and_step1():
    rng = np.random.default_rng(1)
    m = rng.standard_normal(10000).astype(np.float32)
    g = rng.standard_normal(10000).astype(np.float32)
    m_new, u = M.momentum(m, g, 0.95)
    tm = torch.add(torch.mul(torch.from_numpy(m), torch.tensor(0.95, dtype=torch.float32)),
                   torch.from_numpy(g))
    assert (m_new == tm.numpy()).all()
    assert (u == M.bf16_rne_bits(m_new)).all()
    # step 1 (m0 = 0) and mu = 0: u = bf16(g), m = g
    m1, u1 = M.momentum(np.zeros_like(g), g, 0.95)
    assert (m1 == g).all() and (u1 == M.bf16_rne_bits(g)).all()
    m0, u0 = M.momentum(m, g, 0.0)
    assert (u0 == M.bf16_rne_bits(g)).all()
    # Nesterov: u = bf16(g + mu * m_new)
    mn, un = M.momentum(m, g, 0.95, nesterov=True)
    assert (un == M.bf16_rne_bits(g + np.float32(0.95) * mn)).all()


def _with_spectrum(r, c, sigma, seed):
    rng = np.random.default_rng(seed)
    k = min(r, c)
    U, _ = np.linalg.qr(rng.standard_normal((r, k)))
    Vt, _ = np.linalg.qr(rng.standard_normal((c, k)))
    return U, np.asarray(sigma, np.float64), Vt


def _closed_form(U, s, Vt, steps=5, a=3.4445, b=-4.7750, c=2.0315, eps=1e-7):
    sh = s / (np.sqrt(np.sum(s * s)) + eps)
    return U @ np.diag(M.ns_polynomial(sh, steps, a, b, c)) @ Vt.T


@pytest.mark.parametrize("r,c", [(64, 256), (256, 64), (48, 80), (96, 96), (8, 16)])
def test_newton_schulz_closed_form(r, c):
    k = min(r, c)
    sigma = np.geomspace(3.0, 0.03, k)
    U, s, Vt = _with_spectrum(r, c, sigma, seed=r * 1000 + c)
    x = U @ np.diag(s) @ Vt.T
    got = M.newton_schulz(x, dtype=np.float64, **NS)
    ref = _closed_form(U, s, Vt)
    assert np.linalg.norm(got - ref) <= 1e-10 * np.linalg.norm(ref)
    got32 = M.newton_schulz(x.astype(np.float32), dtype=np.float32, **NS)
    assert np.linalg.norm(got32 - ref) <= 1e-4 * np.linalg.norm(ref)


def test_newton_schulz_scale_invariance_and_zero():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((32, 64))
    ns0 = dict(NS, eps=0.0)   # eps breaks exact scale invariance; take it out
    a = M.newton_schulz(x, dtype=np.float64, **ns0)
    b = M.newton_schulz(x * 1e3, dtype=np.float64, **ns0)
    assert np.allclose(a, b, rtol=1e-9, atol=1e-11)
    z = M.newton_schulz(np.zeros((16, 32)), dtype=np.float64, **NS)
    assert (z == 0).all()


def test_newton_schulz_band_on_gaussian_units():
    for (r, c, seed) in [(64, 256, 0), (128, 512, 1), (256, 128, 2)]:
        x = np.random.default_rng(seed).standard_normal((r, c)) * 1e-3
        sig_in = np.linalg.svd(x, compute_uv=False)
        sh = sig_in / (np.sqrt(np.sum(sig_in ** 2)) + 1e-7)
        p = M.ns_polynomial(sh, 5, 3.4445, -4.7750, 2.0315)
        out = np.linalg.svd(M.newton_schulz(x, dtype=np.float64, **NS), compute_uv=False)
        assert out.min() >= 0.68 - 0.02 and out.max() <= p.max() + 0.02
        # in exact arithmetic the iteration maps each singular value through p^5
        assert np.allclose(np.sort(out), np.sort(p), atol=1e-9)


def test_distance_to_polar_factor_on_tiny_matrices():
    for seed in range(4):
        x = np.random.default_rng(seed).standard_normal((8, 16))
        U, s, Vt = np.linalg.svd(x, full_matrices=False)
        polar = U @ Vt
        got = M.newton_schulz(x, dtype=np.float64, **NS)
        sh = s / (np.sqrt(np.sum(s * s)) + 1e-7)
        bound = np.max(np.abs(M.ns_polynomial(sh, 5, 3.4445, -4.7750, 2.0315) - 1))
        assert np.linalg.norm(got - polar, 2) <= bound + 1e-9
        assert bound < 0.33


def _ns_spectral(x, steps, a, b, c, eps):
    """Newton-Schulz normalised by the spectral norm instead of the Frobenius norm."""
    x = x / (np.linalg.norm(x, 2) + eps)
    for _ in range(steps):
        A = x @ x.T
        x = a * x + (b * A + c * (A @ A)) @ x
    return x


def _mutants():
    def no_transpose_back(u, steps, a, b, c, eps, dtype):
        x = (np.asarray(u, np.float64) / (np.linalg.norm(u) + eps)).astype(dtype)
        x = x.T if x.shape[0] > x.shape[1] else x
        for _ in range(steps):
            A = x @ x.T
            B = b * A + c * (A @ A)
            x = a * x + B @ x
        return x

    def spectral_norm_scaling(u, steps, a, b, c, eps, dtype):
        return _ns_spectral(np.asarray(u, np.float64), steps, a, b, c, eps)

    def wrong_sign_b(u, steps, a, b, c, eps, dtype):
        return M.newton_schulz(u, steps, a, -b, c, eps, dtype)

    def uses_a_for_b(u, steps, a, b, c, eps, dtype):
        x = (np.asarray(u, np.float64) / (np.linalg.norm(u) + eps)).astype(dtype)
        t = x.shape[0] > x.shape[1]
        x = x.T if t else x
        for _ in range(steps):
            A = x @ x.T
            x = a * x + A @ x
        return x.T if t else x

    def one_step_short(u, steps, a, b, c, eps, dtype):
        return M.newton_schulz(u, steps - 1, a, b, c, eps, dtype)

    return [no_transpose_back, spectral_norm_scaling, wrong_sign_b, uses_a_for_b, one_step_short]


@pytest.mark.parametrize("mutant", _mutants())
def test_closed_form_catches_planted_mistakes(mutant):
    r, c = 48, 80
    sigma = np.geomspace(3.0, 0.03, min(r, c))
    U, s, Vt = _with_spectrum(r, c, sigma, seed=7)
    ref = _closed_form(U, s, Vt)
    caught = False
    for (rr, cc, UU, VV) in [(r, c, U, Vt), (c, r, Vt, U)]:
        x = UU @ np.diag(s) @ VV.T
        try:
            got = mutant(x, 5, 3.4445, -4.7750, 2.0315, 1e-7, np.float64)
        except ValueError:
            caught = True
            continue
        want = _closed_form(UU, s, VV)
        if got.shape != want.shape or np.linalg.norm(got - want) > 1e-6 * np.linalg.norm(want):
            caught = True
    assert caught


def test_f2_identities_and_alpha():
    rng = np.random.default_rng(9)
    w = rng.standard_normal(1000).astype(np.float32)
    v = rng.standard_normal(1000).astype(np.float32)
    assert (M.main_weight_update(w, v, 0.0, 1.0) == w).all()
    got = M.main_weight_update(w, v, 0.02, 1.0)
    assert (got == (w - np.float32(0.02) * v)).all()
    gw = M.main_weight_update(w, v, 0.02, 1.0, wd=0.1)
    assert (gw == (w * np.float32(1 - 0.002)) - np.float32(0.02) * v).all()
    assert M.alpha(0, 4096, 14336) == 1.0
    assert M.alpha(1, 14336, 4096) == pytest.approx(np.sqrt(14336 / 4096))
    assert M.alpha(1, 4096, 14336) == 1.0
    assert M.alpha(2, 128, 5120) == pytest.approx(0.2 * np.sqrt(5120))
