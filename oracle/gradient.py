"""Update-side gradient path (oracle): the outer reduce-scatter that turns
per-rank gradient contributions into the ZeRO-1 main-gradient shards, with
the paper's partial-precision modes.

Follows "SS-HSDP" section 3.4 (Update: Tg maps the accumulated gradients to
the update representation and the outer reduce-scatter produces the ZeRO-1
main-gradient shards), section 4.3 (ZeroSM reduce-scatter: intra-node
exchange and FP32 reduce, inter-node exchange, final FP32 reduce accumulating
into the persistent gradient; node-local partials may be stored in BF16 with
stochastic rounding, E[SR(s)] = s) and Table 4 (SR needs a seed / counter
state that is restored on the same logical rank).

Readings (design notes): ranks are grouped in nodes of L consecutive
contributions; node sum s_k = fp32 sum over its L contributions in order;
mode FP32 keeps s_k, BF16 rounds it to bf16 (RNE), BF16SR rounds it
stochastically; the total is the fp32 sum of the node partials in node order;
accumulate adds it to the existing gradient (fp32).  Stochastic rounding of
an fp32 value to bf16 adds 16 random bits to the low half of its bit pattern
and truncates (round up with probability equal to the discarded fraction).
The random bits of element i and node k are 16-bit field (i mod 8) of the
128-bit output of Philox4x32-10 (Salmon et al., SC'11) with counter
(i div 8 mod 2^32, i div 8 div 2^32, k, offset) and key (seed mod 2^32,
seed div 2^32); field f is bits 16 (f mod 2) .. +15 of word f div 2.

Pins (tests/test_oracle_gradient.py): Philox known-answer vectors
(tests/golden/philox4x32_10_kat.txt); SR leaves bf16-representable values
unchanged, rounds to a neighbour otherwise, and averaged over all 65536
random-bit values equals its input exactly; FP32 mode against a float64 sum;
SR mode unbiased over seeds.
"""
from __future__ import annotations

import numpy as np

from .muon import bf16_bits_to_f32, bf16_rne_bits

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32 with 10 rounds; uint64 arrays holding 32-bit
    values in, a tuple of four uint64 arrays of 32-bit words out."""
    c = [np.asarray(x, dtype=np.uint64) & np.uint64(MASK) for x in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, dtype=np.uint64) & np.uint64(MASK)
    k1 = np.asarray(k1, dtype=np.uint64) & np.uint64(MASK)
    for r in range(10):
        if r:
            k0 = (k0 + np.uint64(W0)) & np.uint64(MASK)
            k1 = (k1 + np.uint64(W1)) & np.uint64(MASK)
        p0 = c[0] * np.uint64(M0)
        p1 = c[2] * np.uint64(M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(MASK)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(MASK)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return tuple(c)


def sr_bits(index, node, seed, offset):
    """16 random bits for element `index` of node `node`: field index mod 8 of
    the 128-bit Philox4x32-10 output for counter (index div 8 mod 2^32,
    index div 8 div 2^32, node, offset) and key (seed mod 2^32, seed div 2^32);
    field f is bits 16 (f mod 2) .. 16 (f mod 2) + 15 of word f div 2."""
    index = np.asarray(index, dtype=np.uint64)
    blk = index >> np.uint64(3)
    out = philox4x32_10(blk & np.uint64(MASK), blk >> np.uint64(32), np.full_like(index, node),
                        np.full_like(index, offset & MASK), seed & MASK, (seed >> 32) & MASK)
    f = index & np.uint64(7)
    word = np.choose((f >> np.uint64(1)).astype(np.int64), out)
    return ((word >> ((f & np.uint64(1)) * np.uint64(16))) & np.uint64(0xFFFF)).astype(np.uint32)


def bf16_sr_bits(x: np.ndarray, rbits: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns by stochastic rounding (finite inputs)."""
    bits = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((bits + (np.asarray(rbits, dtype=np.uint64) & np.uint64(0xFFFF))) >> np.uint64(16)).astype(np.uint16)


def reduce_scatter(parts: np.ndarray, ranks_per_node: int, mode: str, seed: int = 0, offset: int = 0):
    """parts [P][n] float32 -> total [n] float32 (logical order)."""
    parts = np.asarray(parts, dtype=np.float32)
    P, n = parts.shape
    if P % ranks_per_node:
        raise ValueError("ranks must fill whole nodes")
    total = np.zeros(n, dtype=np.float32)
    idx = np.arange(n, dtype=np.uint64)
    for k in range(P // ranks_per_node):
        s = np.zeros(n, dtype=np.float32)
        for l in range(ranks_per_node):
            s = (s + parts[k * ranks_per_node + l]).astype(np.float32)
        if mode == "bf16":
            s = bf16_bits_to_f32(bf16_rne_bits(s))
        elif mode == "bf16_sr":
            s = bf16_bits_to_f32(bf16_sr_bits(s, sr_bits(idx, k, seed, offset)))
        elif mode != "fp32":
            raise ValueError("mode")
        total = (total + s).astype(np.float32)
    return total
