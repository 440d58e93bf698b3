"""Muon update of one update parameter (oracle): F = [f0, f1, f2].

Follows "SS-HSDP" section 3.1 example EG1 and Figure 4 (per-head Muon):
  f0 updates the momentum m from the main gradient g and writes a BF16
     intermediate u ("Local momentum g, m -> u (BF16)");
  f1 applies Newton-Schulz to the complete unit u and writes an FP32 update
     direction v to separate scratch;
  f2 updates the main weight using v ("Local main-weight update").
The paper cites Muon as its reference [17] and prints no formula; the
readings used here (design notes R8-R10) are:
  f0: m <- mu*m + g in float32 (multiply, then add, each rounded);
      u = bf16_RNE(m)   (Nesterov variant: u = bf16_RNE(g + mu*m_new));
  f1: X0 = u / (||u||_F + eps), transposed when rows > cols so that X X^T is
      the smaller Gram matrix; then `steps` times
          A = X X^T;  B = b A + c A A;  X = a X + B X
      with (a, b, c) = (3.4445, -4.7750, 2.0315); v = X (transposed back);
  f2: w <- w * (1 - lr*wd) (only when wd != 0), then w <- w - (lr*alpha) v,
      in float32 with the scalars rounded to float32 first.

Pins (tests/test_oracle_muon.py): bf16 rounding against PyTorch's bfloat16
cast; Newton-Schulz against its closed form U diag(p^k(sigma)) V^T on
matrices built with a chosen spectrum (both orientations); the output
spectrum band; distance to the SVD polar factor U V^T on tiny matrices;
step-1 identities (u = bf16(g), lr = 0 leaves w unchanged).
"""
from __future__ import annotations

import math

import numpy as np


def bf16_rne_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    bits = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    return ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def momentum(m: np.ndarray, g: np.ndarray, mu: float, nesterov: bool = False):
    """f0.  Returns (m_new float32, u as bf16 bit patterns)."""
    m = np.asarray(m, dtype=np.float32)
    g = np.asarray(g, dtype=np.float32)
    mu32 = np.float32(mu)
    m_new = (mu32 * m) + g
    src = (g + mu32 * m_new) if nesterov else m_new
    return m_new.astype(np.float32), bf16_rne_bits(src)


def newton_schulz(u: np.ndarray, steps: int, a: float, b: float, c: float,
                  eps: float, dtype=np.float32) -> np.ndarray:
    """f1 on one complete unit (rows x cols).  dtype sets the arithmetic of
    the iteration (float32 for parity, float64 for the closed-form pin)."""
    u64 = np.asarray(u, dtype=np.float64)
    s = math.sqrt(float(np.sum(u64 * u64)))
    x = (u64 / (s + eps)).astype(dtype)
    transposed = x.shape[0] > x.shape[1]
    if transposed:
        x = np.ascontiguousarray(x.T)
    a, b, c = dtype(a), dtype(b), dtype(c)
    for _ in range(steps):
        A = x @ x.T
        B = b * A + c * (A @ A)
        x = a * x + B @ x
    if transposed:
        x = np.ascontiguousarray(x.T)
    return x


def ns_polynomial(sigma: np.ndarray, steps: int, a: float, b: float, c: float) -> np.ndarray:
    """p^steps(sigma) for p(s) = a s + b s^3 + c s^5 (the action of the
    iteration on each singular value; used by the closed-form pin)."""
    s = np.asarray(sigma, dtype=np.float64)
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def alpha(mode: int, rows: int, cols: int) -> float:
    if mode == 0:
        return 1.0
    if mode == 1:
        return math.sqrt(max(1.0, rows / cols))
    if mode == 2:
        return 0.2 * math.sqrt(max(rows, cols))
    raise ValueError("alpha mode")


def main_weight_update(w: np.ndarray, v: np.ndarray, lr: float, alpha_: float,
                       wd: float = 0.0) -> np.ndarray:
    """f2 in float32."""
    w = np.asarray(w, dtype=np.float32)
    if wd != 0.0:
        w = w * np.float32(1.0 - lr * wd)
    step = np.float32(lr * alpha_)
    return (w - step * np.asarray(v, dtype=np.float32)).astype(np.float32)
