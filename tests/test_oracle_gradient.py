"""Pins for oracle.gradient: Philox known answers, stochastic-rounding
identities, FP32 reduction against float64, unbiasedness of the SR mode."""
import os

import numpy as np

from oracle import gradient as G
from oracle import muon as M

KAT = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answers():
    n = 0
    for line in open(KAT):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(x, 16) for x in line.split()]
        out = G.philox4x32_10(*[np.uint64(x) for x in v[:6]])
        assert [int(o) for o in out] == v[6:]
        n += 1
    assert n == 3


def test_sr_identities_and_exact_mean():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200) * 10.0 ** rng.integers(-6, 6, 200)).astype(np.float32)
    exact = M.bf16_bits_to_f32(M.bf16_rne_bits(x))                    # bf16-representable values
    for rb in (0, 1, 0x7FFF, 0xFFFF):
        assert (M.bf16_bits_to_f32(G.bf16_sr_bits(exact, np.full(200, rb))) == exact).all()
    all_bits = np.arange(65536, dtype=np.uint32)
    for xi in x[:40]:
        r = M.bf16_bits_to_f32(G.bf16_sr_bits(np.full(65536, xi, np.float32), all_bits)).astype(np.float64)
        lo, hi = np.min(r), np.max(r)
        assert set(np.unique(r)) <= {lo, hi} and lo <= xi <= hi
        assert r.mean() == float(xi)                                   # E[SR(x)] = x, exactly
    assert (G.bf16_sr_bits(np.float32([1.0 + 2 ** -9]), np.array([0])) == 0x3F80).all()    # truncates
    assert (G.bf16_sr_bits(np.float32([1.0 + 2 ** -9]), np.array([0xFFFF])) == 0x3F81).all()  # rounds up


def test_fp32_mode_matches_float64_sum():
    rng = np.random.default_rng(1)
    parts = (rng.standard_normal((8, 4096)) * 1e-3).astype(np.float32)
    got = G.reduce_scatter(parts, 4, "fp32").astype(np.float64)
    want = parts.astype(np.float64).sum(axis=0)
    assert np.allclose(got, want, rtol=1e-6, atol=1e-9)
    bf = G.reduce_scatter(parts, 4, "bf16").astype(np.float64)
    # two node partials, each rounded to bf16 (half an ulp: at most 2^-8 relative)
    nodes = np.abs(parts.astype(np.float64).reshape(2, 4, -1).sum(axis=1))
    assert (np.abs(bf - want) <= 2.0 ** -8 * nodes.sum(axis=0) + 1e-9).all()


def test_sr_mode_is_unbiased_over_seeds():
    rng = np.random.default_rng(2)
    parts = (rng.standard_normal((4, 2048)) * 1e-3).astype(np.float32)
    exact = G.reduce_scatter(parts, 2, "fp32").astype(np.float64)
    runs = np.stack([G.reduce_scatter(parts, 2, "bf16_sr", seed=s, offset=7) for s in range(64)]).astype(np.float64)
    err_mean = np.abs(runs.mean(axis=0) - exact)
    err_one = np.abs(runs[0] - exact)
    assert err_mean.mean() < 0.25 * err_one.mean()                    # averaging 64 draws shrinks the error
    nearest = G.reduce_scatter(parts, 2, "bf16").astype(np.float64)
    assert np.abs(runs.mean(axis=0) - exact).mean() < np.abs(nearest - exact).mean()
    # the same seed and counter replay the same draw
    assert (G.reduce_scatter(parts, 2, "bf16_sr", seed=5, offset=7) ==
            G.reduce_scatter(parts, 2, "bf16_sr", seed=5, offset=7)).all()
