"""Tw's 128 x 4 tiled scale layout, read by a consumer that does not share
this repository's reading of it.

SS-HSDP section 3.1 (example EG1): after G, Tw relays the UE8M0 scales out
into the layout the MXFP8 GEMM kernels need; section 4.1 batches that step.
The layout (`mxfp8_scale_relayout`, and `scale_tile_128x4` in the oracle) is
taken from cuBLAS's public description of its block-scaling factors.  The
bit-exact GPU-vs-oracle test of the relayout cannot catch a misreading that
both sides share, so here cuBLAS itself -- its block-scaled MXFP8 GEMM, reached
through torch._scaled_mm -- consumes the codes and tiled scales and its product
is compared with the float64 product of the operands the oracle dequantizes
from the same codes and K-major scales.  A wrong tile order or lane
interleave would multiply blocks by other blocks' powers of two; the operands
give every block its own power of two, so such a mistake is far outside the
tolerance (and two such mistakes are planted below, on the CPU, to show it).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import mxfp8 as OX  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(hm):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _rup(x, k):
    return -(-x // k) * k


def _operand(rng, rows, k, block_rows):
    """Gaussian values times one power of two (2^-6 .. 2^6) per MX block."""
    x = rng.standard_normal((rows, k)) * 0.02
    e = rng.integers(-6, 7, size=(-(-rows // block_rows), k // 32))
    e = np.repeat(np.repeat(e, block_rows, axis=0)[:rows], 32, axis=1)
    return (x * np.ldexp(1.0, e)).astype(np.float32)


def _quantize(hm, dev, x, block_rows):
    """GPU G (1 x 32 or 32 x 32 blocks) -> codes [rows][K] and K-major scales
    [rows / block_rows][K / 32], checked bit-exactly against the oracle."""
    rows, k = x.shape
    xd = torch.from_numpy(x).to(dev)
    q = torch.empty(rows * k, dtype=torch.uint8, device=dev)
    s = torch.empty((rows // block_rows) * (k // 32), dtype=torch.uint8, device=dev)
    if block_rows == 1:
        hm.mxfp8_requant_packed(xd.data_ptr(), q.data_ptr(), s.data_ptr(), [(0, 0, 0, rows, k)])
        codes, sf = OX.quantize_tensor(x)
    else:
        hm.mxfp8_requant_32x32(0, xd.data_ptr(), q.data_ptr(), s.data_ptr(), [(0, 0, 0, rows, k)])
        codes, sf = OX.quantize_tensor_32x32(x)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), codes.ravel())
    assert np.array_equal(s.cpu().numpy(), sf.ravel())
    return q, s, codes, sf


def _relayout(hm, dev, s, rows, kb, block_rows):
    out = torch.full((_rup(rows, 128) * _rup(kb, 4),), 0xEE, dtype=torch.uint8, device=dev)
    hm.mxfp8_scale_relayout(s.data_ptr(), out.data_ptr(), [(0, 0, rows, kb, block_rows)])
    torch.cuda.synchronize()
    return out


def _row_scales(sf, block_rows):
    return OX.expand_block_rows(sf, block_rows) if block_rows > 1 else sf


def _dequant(codes, sf, block_rows):
    """Oracle dequantization of [rows][K] codes with their K-major scales."""
    rows, k = codes.shape
    return OX.dequantize(codes.ravel(), _row_scales(sf, block_rows).ravel()).reshape(rows, k)


def _mx_gemm(qa, ta, qb, tb, m, n, k):
    """cuBLAS block-scaled MXFP8 GEMM: A [m][k] row-major, B [n][k] row-major
    (passed as the column-major k x n operand), scales in the tiled layout."""
    a = qa.view(torch.float8_e4m3fn).view(m, k)
    b = qb.view(torch.float8_e4m3fn).view(n, k).t()
    sa = ta.view(torch.float8_e8m0fnu).view(_rup(m, 128), _rup(k // 32, 4))
    sb = tb.view(torch.float8_e8m0fnu).view(_rup(n, 128), _rup(k // 32, 4))
    out = torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def _excess(out, ref, bound):
    """Largest |out - ref| measured in units of its allowance: bf16 rounding of
    the output (2^-8 relative, twice the half-ulp) plus the fp32 accumulation
    over K (1e-4 of the sum of |products|, about 40x K * 2^-24 at K = 640)."""
    tol = 2.0 ** -8 * np.abs(ref) + 1e-4 * bound
    return float(np.max(np.abs(out - ref) / tol))


# planted misreadings of the layout (CPU): each must be rejected by the consumer
def _tiles_column_major(sf):
    rows, kb = sf.shape
    rt, ct = -(-rows // 128), -(-kb // 4)
    good = OX.scale_tile_128x4(sf).reshape(rt, ct, 512)
    return np.ascontiguousarray(good.transpose(1, 0, 2)).ravel()


def _no_lane_interleave(sf):
    rows, kb = sf.shape
    rt, ct = -(-rows // 128), -(-kb // 4)
    pad = np.zeros((rt * 128, ct * 4), dtype=np.uint8)
    pad[:rows, :kb] = sf
    return np.ascontiguousarray(pad.reshape(rt, 128, ct, 4).transpose(0, 2, 1, 3)).ravel()


@pytest.mark.parametrize("m,n,k,block_rows", [
    (256, 256, 512, 1),     # 2 x 4 tiles per operand
    (384, 128, 640, 1),     # 3 x 5 and 1 x 5 tiles
    (208, 144, 352, 1),     # rows and K/32 = 11 not multiples of 128 and 4: zero padding read
    (256, 256, 512, 32),    # 32 x 32 blocks, scales repeated over their 32 rows
    (224, 160, 352, 32),
])
def test_tiled_scales_feed_cublas_block_scaled_gemm(hm, dev, m, n, k, block_rows):
    rng = np.random.default_rng(1000 + m + n + k + block_rows)
    xa = _operand(rng, m, k, block_rows)
    xb = _operand(rng, n, k, block_rows)
    qa, sa, ca, sfa = _quantize(hm, dev, xa, block_rows)
    qb, sb, cb, sfb = _quantize(hm, dev, xb, block_rows)
    kb = k // 32
    ta = _relayout(hm, dev, sa, m, kb, block_rows)
    tb = _relayout(hm, dev, sb, n, kb, block_rows)
    # the relayout equals the oracle's layout (bit-exact) ...
    la = OX.scale_tile_128x4(_row_scales(sfa, block_rows))
    lb = OX.scale_tile_128x4(_row_scales(sfb, block_rows))
    assert np.array_equal(ta.cpu().numpy(), la) and np.array_equal(tb.cpu().numpy(), lb)

    da, db = _dequant(ca, sfa, block_rows), _dequant(cb, sfb, block_rows)
    ref = da @ db.T
    bound = np.abs(da) @ np.abs(db).T
    # ... and cuBLAS, reading it, multiplies every block by its own scale
    out = _mx_gemm(qa, ta, qb, tb, m, n, k)
    assert _excess(out, ref, bound) <= 1.0

    # the oracle's layout, handed to cuBLAS from the CPU, pins the oracle itself
    out_oracle = _mx_gemm(qa, torch.from_numpy(la).to(dev), qb, torch.from_numpy(lb).to(dev), m, n, k)
    assert _excess(out_oracle, ref, bound) <= 1.0

    # planted misreadings of the layout are rejected by the same comparison
    for wrong in (_tiles_column_major, _no_lane_interleave):
        wa = torch.from_numpy(wrong(_row_scales(sfa, block_rows))).to(dev)
        wb = torch.from_numpy(wrong(_row_scales(sfb, block_rows))).to(dev)
        if torch.equal(wa, ta) and torch.equal(wb, tb):
            continue    # one tile column: the column-major order is the same layout
        assert _excess(_mx_gemm(qa, wa, qb, wb, m, n, k), ref, bound) > 100.0, wrong.__name__
