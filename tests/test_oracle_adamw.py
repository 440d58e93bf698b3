"""Pins for oracle.adamw: the step-1 closed form and torch.optim.AdamW (an
independent library implementation) run in float64 on the CPU."""
import numpy as np
import torch

from oracle import adamw as A

HP = dict(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)


def test_step1_closed_form():
    rng = np.random.default_rng(0)
    w0 = rng.standard_normal(10000) * 0.02
    g = rng.standard_normal(10000) * 1e-3
    w1, m1, v1 = A.adamw_step(w0, g, np.zeros_like(w0), np.zeros_like(w0), HP["lr"], HP["beta1"],
                              HP["beta2"], HP["eps"], HP["wd"], 1)
    want = w0 * (1 - HP["lr"] * HP["wd"]) - HP["lr"] * g / (np.abs(g) + HP["eps"])
    assert np.allclose(w1, want, rtol=1e-12, atol=1e-18)
    assert np.allclose(m1, 0.1 * g, rtol=1e-15) and np.allclose(v1, 0.05 * g * g, rtol=1e-15)


def test_matches_torch_adamw_over_steps():
    rng = np.random.default_rng(1)
    n = 5000
    w = rng.standard_normal(n) * 0.02
    p = torch.nn.Parameter(torch.from_numpy(w.copy()))
    opt = torch.optim.AdamW([p], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["wd"], foreach=False)
    m = np.zeros(n)
    v = np.zeros(n)
    for t in range(1, 5):
        g = rng.standard_normal(n) * 1e-3
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        w, m, v = A.adamw_step(w, g, m, v, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["wd"], t)
        st = opt.state[p]
        assert np.allclose(p.detach().numpy(), w, rtol=1e-13, atol=1e-17)
        assert np.allclose(st["exp_avg"].numpy(), m, rtol=1e-13, atol=1e-20)
        assert np.allclose(st["exp_avg_sq"].numpy(), v, rtol=1e-13, atol=1e-24)
