"""Elementwise AdamW update (oracle), float64.

"SS-HSDP" section 5.2 (Table 3 discussion) updates the parameters that Muon
does not handle with AdamW and section 2.1 writes the update as
(w_main, m) <- F(w_main, g, m); the paper prints no AdamW formula.  Reading
(design note R11): PyTorch's documented AdamW with decoupled weight decay,
bias correction and step counter t (t = 1 on the first update):
    w <- w (1 - lr wd)
    m <- b1 m + (1 - b1) g
    v <- b2 v + (1 - b2) g^2
    m_hat = m / (1 - b1^t);  v_hat = v / (1 - b2^t)
    w <- w - lr m_hat / (sqrt(v_hat) + eps)
computed here in float64 from the float32 state and the bf16 gradient
(up-converted exactly).

Pins (tests/test_oracle_adamw.py): the step-1 closed form
w1 = w0 (1 - lr wd) - lr g / (|g| + eps) (m0 = v0 = 0), and agreement with
torch.optim.AdamW run in float64 on the CPU over several steps.
"""
from __future__ import annotations

import numpy as np


def adamw_step(w, g, m, v, lr, beta1, beta2, eps, wd, step):
    w = np.asarray(w, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    w = w * (1.0 - lr * wd)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** step)
    v_hat = v / (1.0 - beta2 ** step)
    w = w - lr * m_hat / (np.sqrt(v_hat) + eps)
    return w, m, v
