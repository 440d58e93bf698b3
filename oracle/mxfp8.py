"""G: MXFP8 quantization of the main weight (oracle).

Follows "SS-HSDP" section 3.1 example EG1 and Figure 4 (G produces FP8 w and
UE8M0 scales s in a K-major layout) and the OCP Microscaling (MX) format that
the paper cites as [28]: a block of 32 elements shares one power-of-two scale
stored as an unsigned 8-bit exponent (E8M0, bias 127); every element is an
FP8 E4M3 number (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
infinities; S.1111.111 is NaN; largest finite value 448 = 1.75 * 2^8).

Readings (design notes R1-R4): blocks are 1 x 32 along K (the contiguous
dimension of a [rows][K] runtime weight); scale exponent
e = clamp(floor(log2 amax) - 8, -127, 127) with 8 = the E4M3 emax, amax = 0
giving e = -127; elements y = x * 2^-e are rounded to the nearest finite
E4M3 value, ties to the even code, magnitudes above 448 saturating to 448;
the sign is copied from x; scales are stored [rows][K/32].

Method: the element code is found by exhaustive search over the 127 finite
non-negative E4M3 values, with exact float64 arithmetic (y is a float32
times a power of two, exact in float64).

Pins (tests/test_oracle_mxfp8.py): every finite code round-trips; every
midpoint between neighbouring codes goes to the even code and one float32 ulp
either side goes to the nearer code; saturation above 448; agreement with
PyTorch's float8_e4m3fn cast on all in-range inputs (an independent library
routine); scale exponent at powers of two, just below them, at zero and at
the clamps.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8
SCALE_BIAS = 127
BLOCK = 32


def e4m3_decode(code: int) -> float:
    """Value of an 8-bit E4M3 code from the format definition (NaN for
    S.1111.111)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# values of the 127 finite non-negative codes 0x00..0x7E (float64, exact)
E4M3_TABLE = np.array([e4m3_decode(c) for c in range(0x7F)], dtype=np.float64)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code to each y (float64, exact); ties to the even
    code; |y| above the largest finite value saturates to it; sign copied."""
    y = np.asarray(y, dtype=np.float64).ravel()
    out = np.empty(y.shape, dtype=np.uint8)
    # saturation: every magnitude above the largest finite value maps to it
    # (clamping first also keeps the distances below exact in float64)
    mag = np.minimum(np.abs(y), E4M3_MAX)
    sign = np.signbit(y)
    step = 1 << 14
    for lo in range(0, y.size, step):
        a = mag[lo:lo + step]
        dist = np.abs(a[:, None] - E4M3_TABLE[None, :])
        best = dist.min(axis=1, keepdims=True)
        cand = dist == best
        # among equally near codes take the even one; else the only one
        even = cand & ((np.arange(0x7F) & 1) == 0)[None, :]
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        out[lo:lo + step] = pick.astype(np.uint8)
    out[sign] |= 0x80
    return out


def floor_log2(a: float) -> int:
    """floor(log2 a) for a > 0, exact (frexp returns a = f * 2^k, f in [0.5,1))."""
    _, k = np.frexp(np.float64(a))
    return int(k) - 1


def scale_exponent(amax: float) -> int:
    if amax == 0.0:
        return -127
    return int(min(127, max(-127, floor_log2(amax) - E4M3_EMAX)))


def quantize_block(x: np.ndarray):
    """One 32-element block of float32 -> (32 E4M3 codes, UE8M0 scale code)."""
    x = np.asarray(x, dtype=np.float32)
    amax = float(np.max(np.abs(x.astype(np.float64))))
    e = scale_exponent(amax)
    y = x.astype(np.float64) * np.ldexp(1.0, -e)
    return e4m3_encode(y), np.uint8(e + SCALE_BIAS)


def quantize_tensor(w: np.ndarray):
    """[rows][K] float32 -> (codes [rows][K] uint8, scales [rows][K/32] uint8),
    1 x 32 blocks along K (vectorised over blocks, same steps as
    quantize_block)."""
    w = np.asarray(w, dtype=np.float32)
    rows, k = w.shape
    if k % BLOCK:
        raise ValueError("K must be a multiple of 32")
    blocks = w.reshape(rows, k // BLOCK, BLOCK).astype(np.float64)
    amax = np.abs(blocks).max(axis=2)
    e = np.full(amax.shape, -127, dtype=np.int64)
    nz = amax > 0
    _, kexp = np.frexp(amax[nz])
    e[nz] = np.clip(kexp.astype(np.int64) - 1 - E4M3_EMAX, -127, 127)
    y = blocks * np.ldexp(1.0, -e)[:, :, None]
    codes = e4m3_encode(y).reshape(rows, k)
    return codes, (e + SCALE_BIAS).astype(np.uint8)


def requant_list(w_flat: np.ndarray, tensors):
    """G over a flat tensor list: tensors = [(flat offset, rows, K)].  Returns
    flat codes (same element offsets as w) and flat scales (offset / 32)."""
    w_flat = np.asarray(w_flat, dtype=np.float32)
    q = np.zeros(w_flat.size, dtype=np.uint8)
    s = np.zeros(w_flat.size // BLOCK, dtype=np.uint8)
    for off, rows, k in tensors:
        codes, sc = quantize_tensor(w_flat[off:off + rows * k].reshape(rows, k))
        q[off:off + rows * k] = codes.ravel()
        s[off // BLOCK:(off + rows * k) // BLOCK] = sc.ravel()
    return q, s


def dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Flat codes and scales -> float64 values (used by invariants in tests)."""
    vals = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    scale = np.ldexp(1.0, s.astype(np.int64) - SCALE_BIAS)
    return vals[q] * np.repeat(scale, BLOCK)


# ---------------------------------------------------------------------------
# 32 x 32 blocks (section 3.1 EG1: "32 x 32 block quantization in a k-major
# layout") and the kernel-facing scale layout of Tw.
# ---------------------------------------------------------------------------
def quantize_tensor_32x32(w: np.ndarray):
    """[rows][K] float32 -> (codes [rows][K], scales [rows/32][K/32]); one
    UE8M0 scale per 32 x 32 block, same exponent rule and element rounding as
    the 1 x 32 case, the block amax taken over all 1024 elements."""
    w = np.asarray(w, dtype=np.float32)
    rows, k = w.shape
    if rows % BLOCK or k % BLOCK:
        raise ValueError("rows and K must be multiples of 32")
    blocks = w.reshape(rows // BLOCK, BLOCK, k // BLOCK, BLOCK).astype(np.float64)
    amax = np.abs(blocks).max(axis=(1, 3))
    e = np.full(amax.shape, -127, dtype=np.int64)
    nz = amax > 0
    _, kexp = np.frexp(amax[nz])
    e[nz] = np.clip(kexp.astype(np.int64) - 1 - E4M3_EMAX, -127, 127)
    y = blocks * np.ldexp(1.0, -e)[:, None, :, None]
    codes = e4m3_encode(y).reshape(rows, k)
    return codes, (e + SCALE_BIAS).astype(np.uint8)


def scale_tile_128x4(sf: np.ndarray) -> np.ndarray:
    """Row-wise scale matrix sf [rows][kb] (kb = K/32 scales per row) ->
    the 128 x 4 tiled layout that block-scaled tensor-core GEMMs read
    (cuBLAS documentation, "1D block scaling factors layout"): rows and kb are
    padded with zeros to multiples of 128 and 4; tile (i, j) of 128 rows x 4
    scale columns occupies 512 bytes at (i * ceil(kb/4) + j) * 512, and inside
    a tile, row r and column c sit at (r % 32) * 16 + (r // 32) * 4 + c."""
    sf = np.asarray(sf, dtype=np.uint8)
    rows, kb = sf.shape
    rt, ct = -(-rows // 128), -(-kb // 4)
    out = np.zeros(rt * ct * 512, dtype=np.uint8)
    for r in range(rows):
        for c in range(kb):
            tile = (r // 128) * ct + c // 4
            rr, cc = r % 128, c % 4
            out[tile * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc] = sf[r, c]
    return out


def expand_block_rows(sf32: np.ndarray, block_rows: int = BLOCK) -> np.ndarray:
    """Scales of 32 x 32 blocks [rows/32][kb] -> one row per weight row
    [rows][kb] (each block's scale repeated over its 32 rows)."""
    return np.repeat(np.asarray(sf32, dtype=np.uint8), block_rows, axis=0)
