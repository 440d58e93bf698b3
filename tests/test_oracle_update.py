"""Pins for oracle.update: the composed update phase reduces to its parts in
the cases the method fixes (lr = 0, mu = 0 at step 1, one unit per matrix)."""
import dataclasses

import numpy as np

import workloads
from oracle import muon as M
from oracle import mxfp8 as MX
from oracle import update as U


def _tiny():
    cfg = workloads.tiny()
    data = workloads.generate(cfg)
    units = [(u.offset, u.rows, u.cols) for u in cfg.units]
    return cfg, data, units


def test_lr_zero_leaves_w_and_requantizes_it():
    cfg, data, units = _tiny()
    hp = dataclasses.replace(cfg.muon, lr=0.0)
    out = U.muon_update(data["w"], np.zeros_like(data["w"]), data["g"], units, cfg.mx_tensors, hp)
    assert (out["w"] == data["w"]).all()
    q, s = MX.requant_list(data["w"], cfg.mx_tensors)
    assert (out["q"] == q).all() and (out["s"] == s).all()


def test_step1_u_is_bf16_of_g_and_v_is_ns_of_u():
    cfg, data, units = _tiny()
    out = U.muon_update(data["w"], np.zeros_like(data["w"]), data["g"], units, cfg.mx_tensors, cfg.muon)
    assert (out["u"] == M.bf16_rne_bits(data["g"])).all()
    assert (out["m"] == data["g"]).all()
    u = M.bf16_bits_to_f32(out["u"])
    off, r, c = units[5]
    v5 = M.newton_schulz(u[off:off + r * c].reshape(r, c), 5, 3.4445, -4.7750, 2.0315, 1e-7)
    assert (out["v"][off:off + r * c] == v5.ravel()).all()
    # the update moves w by lr * v exactly as f2 says
    want = M.main_weight_update(data["w"][off:off + r * c], v5.ravel(), 0.02, 1.0)
    assert (out["w"][off:off + r * c] == want).all()
    # NS output of every unit sits in the quintic's band
    for (off, r, c) in units:
        sv = np.linalg.svd(out["v"][off:off + r * c].reshape(r, c).astype(np.float64), compute_uv=False)
        assert sv.min() > 0.66 and sv.max() < 1.25
