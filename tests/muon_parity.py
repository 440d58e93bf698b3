"""Parity helpers shared by the GPU tests: run the update phase through the
C ABI and compare every stage's output with the oracle."""
from __future__ import annotations

import numpy as np

from oracle import muon as OM
from oracle import mxfp8 as OX
from oracle import views as OV

NS_TOL = 2e-2   # relative Frobenius error of bf16 Newton-Schulz vs the fp32 oracle


def unit_tuples(cfg):
    return [(u.offset, u.rows, u.cols) for u in cfg.units]


def check_f0(m_prev, g, m_gpu, u_gpu, mu, nesterov=False):
    m_ref, u_ref = OM.momentum(m_prev, g, mu, nesterov)
    assert np.array_equal(m_gpu.view(np.uint32), m_ref.view(np.uint32)), "f0: momentum not bit-exact"
    assert np.array_equal(u_gpu, u_ref), "f0: u not bit-exact"


def check_staging(session, cfg, u_bits_logical):
    """u staging of every straddling unit equals the gathered fragments."""
    e = OV.z1_edges(cfg.numel, cfg.so, cfg.edge_shift)
    bases, _ = OV.segment_layout(e, cfg.so, cfg.sw)
    root = OV.to_segments(u_bits_logical, e, cfg.so, cfg.sw)
    n = 0
    for i, (o, r, c) in enumerate(unit_tuples(cfg)):
        fr = OV.fragments(o, o + r * c, e, cfg.so, cfg.sw, bases)
        if len(fr) == 1:
            continue
        us, _ = session.staging(i)
        got = us.cpu().numpy().view(np.uint16)
        assert np.array_equal(got, OV.gather(root, fr, r * c)), f"gather mismatch in unit {i}"
        n += 1
    return n


def check_ns(cfg, u_bits, v_gpu, hp, units=None, tol=NS_TOL):
    """Per unit relative Frobenius error of v against the fp32 oracle."""
    u32 = OM.bf16_bits_to_f32(u_bits)
    worst = 0.0
    for i in (range(len(cfg.units)) if units is None else units):
        un = cfg.units[i]
        sl = slice(un.offset, un.offset + un.numel)
        ref = OM.newton_schulz(u32[sl].reshape(un.rows, un.cols), hp.ns_steps, hp.ns_a, hp.ns_b, hp.ns_c, hp.eps)
        nrm = np.linalg.norm(ref)
        err = np.linalg.norm(v_gpu[sl].astype(np.float64) - ref.ravel()) / nrm if nrm > 0 else np.abs(v_gpu[sl]).max()
        assert err <= tol, f"Newton-Schulz unit {i} ({un.rows}x{un.cols}): rel err {err:.3e}"
        worst = max(worst, err)
    return worst


def check_f2(cfg, w_prev, v_gpu, w_gpu, hp):
    for un in cfg.units:
        sl = slice(un.offset, un.offset + un.numel)
        want = OM.main_weight_update(w_prev[sl], v_gpu[sl], hp.lr, OM.alpha(hp.alpha_mode, un.rows, un.cols),
                                     hp.weight_decay)
        assert np.array_equal(w_gpu[sl].view(np.uint32), want.view(np.uint32)), "f2 not bit-exact"


def check_requant(cfg, w_gpu, q_gpu, s_gpu):
    q_ref, s_ref = OX.requant_list(w_gpu, cfg.mx_tensors)
    assert np.array_equal(q_gpu, q_ref), "MXFP8 codes not bit-exact"
    assert np.array_equal(s_gpu, s_ref), "MXFP8 scales not bit-exact"
