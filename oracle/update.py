"""The composed update phase on logical (unsharded) arrays (oracle).

Follows "SS-HSDP" section 3.4 ("Update", Figure 4 right): f0 on every
fragment, f1 Newton-Schulz on every complete unit, f2 on every fragment, then
G (MXFP8) over the updated main weight.  Sharding does not change the
arithmetic: f0, f2 and G are elementwise or blockwise inside 32-aligned
fragments, and f1 sees each complete unit, so the logical result is the
definition that the sharded, emulated-rank GPU path must reproduce.

Units are (flat offset, rows, cols) triples; MX tensors are (flat offset,
rows, K) triples.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence, Tuple

import numpy as np

from . import adamw as _adamw
from . import muon as _muon
from . import mxfp8 as _mx


def muon_directions(u_f32: np.ndarray, units: Sequence[Tuple[int, int, int]], steps, a, b, c,
                    eps, dtype=np.float32, only: Optional[Sequence[int]] = None) -> Dict[int, np.ndarray]:
    """f1 for the chosen units (all by default): unit index -> v (rows x cols)."""
    out = {}
    for i in (range(len(units)) if only is None else only):
        off, r, cc = units[i]
        out[i] = _muon.newton_schulz(u_f32[off:off + r * cc].reshape(r, cc), steps, a, b, c,
                                     eps, dtype=dtype)
    return out


def apply_f2(w: np.ndarray, v_flat: np.ndarray, units, lr, alpha_mode, wd) -> np.ndarray:
    """f2 on every unit, given the flat direction field v."""
    w_new = np.array(w, dtype=np.float32, copy=True)
    for off, r, cc in units:
        sl = slice(off, off + r * cc)
        w_new[sl] = _muon.main_weight_update(w[sl], v_flat[sl], lr, _muon.alpha(alpha_mode, r, cc), wd)
    return w_new


def muon_update(w, m, g, units, mx_tensors, hp) -> Dict[str, np.ndarray]:
    """One Muon update phase: returns m, u (bf16 bits), v, w, q, s."""
    m_new, u_bits = _muon.momentum(m, g, hp.momentum, hp.nesterov)
    u = _muon.bf16_bits_to_f32(u_bits)
    dirs = muon_directions(u, units, hp.ns_steps, hp.ns_a, hp.ns_b, hp.ns_c, hp.eps)
    v = np.zeros_like(np.asarray(w, dtype=np.float32))
    for i, (off, r, cc) in enumerate(units):
        v[off:off + r * cc] = dirs[i].ravel()
    w_new = apply_f2(w, v, units, hp.lr, hp.alpha_mode, hp.weight_decay)
    q, s = _mx.requant_list(w_new, mx_tensors)
    return {"m": m_new, "u": u_bits, "v": v, "w": w_new, "q": q, "s": s}


def adamw_update(w, g_bf16_bits, m, v, hp, step, mx_tensors=None):
    """One AdamW update (float64 arithmetic) and, optionally, G on the
    float32-rounded result."""
    g = _muon.bf16_bits_to_f32(g_bf16_bits)
    w64, m64, v64 = _adamw.adamw_step(w, g, m, v, hp.lr, hp.beta1, hp.beta2, hp.eps,
                                      hp.weight_decay, step)
    out = {"w": w64, "m": m64, "v": v64}
    if mx_tensors is not None:
        out["q"], out["s"] = _mx.requant_list(w64.astype(np.float32), mx_tensors)
    return out
