"""Parity at the full workload sizes, in the launch configuration the
benchmark times (one muon_update_units call over the whole tensor list):
sampled units through Newton-Schulz, sampled elements through f0 and f2,
sampled MXFP8 blocks, canaries and the device error word.  The oracle sees
the exact device inputs (copied back)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import adamw as OA  # noqa: E402
from oracle import muon as OM  # noqa: E402
from oracle import mxfp8 as OX  # noqa: E402

from muon_parity import NS_TOL  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(hm):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _sample_units(cfg, s, hm, rng):
    """A head (or smallest) unit, the last unit of its shape class (with more
    units than SMs, one that runs in the last round, split over a CTA pair),
    a straddling unit and a largest unit."""
    sizes = [u.numel for u in cfg.units]
    small = int(np.argmin(sizes))
    big = int(np.argmax(sizes))
    cls = lambda u: (min(u.rows, u.cols), max(u.rows, u.cols))  # noqa: E731
    last_small = max(i for i, u in enumerate(cfg.units) if cls(u) == cls(cfg.units[small]))
    strad = [i for i in range(len(cfg.units)) if not hm.muon_plan_unit(s.plan, i)["local"]]
    pick = {small, last_small, big}
    if strad:
        pick.add(int(rng.choice(strad)))
    return sorted(pick)


@pytest.mark.parametrize("name,variant", [("lm_layer", "plain"), ("moe_layer", "plain"), ("video_dit", "plain"),
                                          ("moe_layer", "nesterov_decay")])
def test_fullsize_update_sampled(hm, dev, name, variant):
    """The benchmark's stage set (HM_STAGE_STEP: f0 inside the Newton-Schulz
    input pass, f2 and G in the last product's epilogue, neither u nor v
    stored) against the same update through v (HM_STAGE_ALL_FUSED) on a
    second session: m, w, q, s equal bit for bit over the whole tensor list;
    the second session's u and v then carry the f0, Newton-Schulz and f2
    checks.  nesterov_decay: Nesterov momentum, decoupled weight decay and
    the shape-dependent step scale sqrt(max(1, rows / cols)) at full size."""
    import dataclasses
    from head_muon_mxfp8_gb300.session import MuonSession, muon_hparams
    cfg = workloads.get(name)
    if variant == "nesterov_decay":
        cfg.muon = dataclasses.replace(cfg.muon, nesterov=True, weight_decay=0.1, alpha_mode=1,
                                       lr=float(np.float32(0.02)))
    rng = np.random.default_rng(7)
    s = MuonSession.from_config(cfg, device=dev)
    s_v = MuonSession.from_config(cfg, device=dev)
    data = workloads.generate_device(cfg, dev, seed=3)
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    m0 = torch.empty(cfg.numel, dtype=torch.float32, device=dev).normal_(0.0, 1e-3, generator=gen)
    for x in (s, s_v):
        x.load("w", data["w"])
        x.load("g", data["g"])
        x.load("m", m0)
    # the samples the oracle will need, taken before the update
    idx = torch.from_numpy(np.sort(rng.choice(cfg.numel, 1 << 20, replace=False))).to(dev)
    w0_s, g_s, m0_s = data["w"][idx].cpu().numpy(), data["g"][idx].cpu().numpy(), m0[idx].cpu().numpy()
    units = _sample_units(cfg, s, hm, rng)
    w0_units = {i: data["w"][cfg.units[i].offset:cfg.units[i].offset + cfg.units[i].numel].cpu().numpy()
                for i in units}
    del data, m0
    s.run(muon_hparams(cfg.muon), hm.HM_STAGE_STEP)
    s_v.run(muon_hparams(cfg.muon), hm.HM_STAGE_ALL_FUSED)
    torch.cuda.synchronize()
    assert hm.hm_device_error() == 0
    for f in ("m", "w", "q", "s"):
        a, b = getattr(s, f), getattr(s_v, f)
        if a.dtype == torch.float32:  # bit patterns: the guard words between segments are NaNs
            a, b = a.view(torch.int32), b.view(torch.int32)
        assert torch.equal(a, b), f"{f}: HM_STAGE_STEP differs from the pass through v"
    u_v = s_v.fetch("u")
    for i, un in enumerate(cfg.units):
        if not hm.muon_plan_unit(s.plan, i)["local"]:
            sl = slice(un.offset, un.offset + un.numel)
            assert torch.equal(s_v.staging(i)[0].cpu(), u_v[sl])
    del u_v
    # f0 on sampled elements (bit-exact)
    m_ref, u_ref = OM.momentum(m0_s, g_s, cfg.muon.momentum, cfg.muon.nesterov)
    m_all = s.fetch("m")
    u_all = s_v.fetch("u")
    assert np.array_equal(m_all[idx.cpu()].numpy().view(np.uint32), m_ref.view(np.uint32))
    assert np.array_equal(u_all[idx.cpu()].numpy().view(np.uint16), u_ref)
    # Newton-Schulz and f2 on whole sampled units
    h = cfg.muon
    for i in units:
        un = cfg.units[i]
        u_bits = u_all[un.offset:un.offset + un.numel].numpy().view(np.uint16)
        ref = OM.newton_schulz(OM.bf16_bits_to_f32(u_bits).reshape(un.rows, un.cols), h.ns_steps, h.ns_a, h.ns_b,
                               h.ns_c, h.eps)
        v = s_v.unit_v(i).numpy()
        err = np.linalg.norm(v.astype(np.float64) - ref.ravel()) / np.linalg.norm(ref)
        assert err <= NS_TOL, f"unit {i} {un.rows}x{un.cols}: {err:.3e}"
        w1 = s.fetch_range("w", un.offset, un.offset + un.numel).numpy()
        want = OM.main_weight_update(w0_units[i], v, h.lr, OM.alpha(h.alpha_mode, un.rows, un.cols), h.weight_decay)
        assert np.array_equal(w1.view(np.uint32), want.view(np.uint32))
    del m_all, u_all
    assert all(s_v.canary_intact().values())
    s_v.close()
    # MXFP8 on sampled blocks (bit-exact on the device's updated w)
    w_all = s.fetch("w").numpy()
    q_all = s.fetch("q").numpy()
    s_all = s.fetch("s").numpy()
    blocks = rng.choice(cfg.numel // 32, 8192, replace=False)
    for b in blocks[:8192]:
        codes, sc = OX.quantize_block(w_all[32 * b:32 * b + 32])
        assert np.array_equal(q_all[32 * b:32 * b + 32], codes) and s_all[b] == sc
    assert all(s.canary_intact().values())
    s.close()


def test_fullsize_adamw_and_requant_sampled(hm, dev):
    from head_muon_mxfp8_gb300.session import adamw_hparams
    cfg = workloads.flat_adamw()
    n = cfg.numel
    gen = torch.Generator(device=dev)
    gen.manual_seed(9)
    w = torch.empty(n, device=dev).normal_(0, cfg.w_std, generator=gen)
    g = torch.empty(n, device=dev).normal_(0, cfg.g_std, generator=gen).to(torch.bfloat16)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    rng = np.random.default_rng(1)
    idx = torch.from_numpy(np.sort(rng.choice(n, 1 << 20, replace=False))).to(dev)
    w0 = w[idx].cpu().numpy().astype(np.float64)
    g_s = g[idx].float().cpu().numpy().astype(np.float64)
    h = cfg.adamw
    hm.adamw_update_flat(w.data_ptr(), g.data_ptr(), hm.HM_BF16, m.data_ptr(), v.data_ptr(), n, adamw_hparams(h, 1))
    q = torch.empty(n, dtype=torch.uint8, device=dev)
    sc = torch.empty(n // 32, dtype=torch.uint8, device=dev)
    hm.mxfp8_requant_packed(w.data_ptr(), q.data_ptr(), sc.data_ptr(), [(0, 0, 0, 16384, 4096)])
    torch.cuda.synchronize()
    f = lambda x: float(np.float32(x))  # noqa: E731
    lr, b1, b2, eps, wd = f(h.lr), f(h.beta1), f(h.beta2), f(h.eps), f(h.weight_decay)
    w64, m64, v64 = OA.adamw_step(w0, g_s, 0 * w0, 0 * w0, lr, b1, b2, eps, wd, 1)
    gw = w[idx].cpu().numpy()
    sm = np.abs((1 - b1) * g_s)
    sw = np.abs(w0 * (1 - lr * wd)) + lr / (1 - b1) * sm / (np.sqrt(v64 / (1 - b2)) + eps)
    assert (np.abs(gw - w64) <= 1e-6 * sw).all()
    assert (np.abs(m[idx].cpu().numpy() - m64) <= 1e-6 * sm).all()
    wn = w.cpu().numpy()
    qn, sn = q.cpu().numpy(), sc.cpu().numpy()
    for b in rng.choice(n // 32, 8192, replace=False):
        codes, s1 = OX.quantize_block(wn[32 * b:32 * b + 32])
        assert np.array_equal(qn[32 * b:32 * b + 32], codes) and sn[b] == s1
