"""Pins for oracle.mxfp8 against the E4M3 / E8M0 format definitions and an
independent library routine (PyTorch's float8_e4m3fn cast)."""
import numpy as np
import pytest
import torch

from oracle import mxfp8 as MX


def test_table_shape():
    t = MX.E4M3_TABLE
    assert t.size == 127 and t[0] == 0.0 and t[0x7E] == 448.0
    assert t[1] == 2.0 ** -9              # smallest subnormal
    assert t[8] == 2.0 ** -6              # smallest normal
    assert (np.diff(t) > 0).all()
    assert np.isnan(MX.e4m3_decode(0x7F)) and np.isnan(MX.e4m3_decode(0xFF))


def test_every_code_roundtrips():
    codes = np.arange(0x7F)
    assert (MX.e4m3_encode(MX.E4M3_TABLE) == codes).all()
    assert (MX.e4m3_encode(-MX.E4M3_TABLE[1:]) == codes[1:] | 0x80).all()
    assert MX.e4m3_encode(np.array([-0.0]))[0] == 0x80


def test_midpoints_go_to_even_and_neighbours_to_nearer():
    t = MX.E4M3_TABLE
    for k in range(0x7E):
        mid = (t[k] + t[k + 1]) / 2
        even = k if k % 2 == 0 else k + 1
        assert MX.e4m3_encode(np.array([mid]))[0] == even
        m32 = np.float32(mid)
        assert float(m32) == mid          # midpoints are exact in float32
        below = float(np.nextafter(m32, np.float32(0)))
        above = float(np.nextafter(m32, np.float32(np.inf)))
        assert MX.e4m3_encode(np.array([below]))[0] == k
        assert MX.e4m3_encode(np.array([above]))[0] == k + 1


def test_saturation():
    y = np.array([448.0, 448.0001, 464.0, 470.0, 511.9, 1e30, -1e30, -500.0])
    assert list(MX.e4m3_encode(y)) == [0x7E] * 6 + [0xFE, 0xFE]


def test_matches_torch_float8_cast_in_range():
    rng = np.random.default_rng(0)
    y = np.concatenate([
        rng.uniform(-448, 448, 200000),
        rng.standard_normal(100000) * 2.0 ** rng.integers(-14, 8, 100000),
        (MX.E4M3_TABLE[:-1] + MX.E4M3_TABLE[1:]) / 2,
        -(MX.E4M3_TABLE[:-1] + MX.E4M3_TABLE[1:]) / 2,
        [0.0, -0.0, 2.0 ** -10, -2.0 ** -10, 2.0 ** -11, 1e-30, -1e-30],
    ]).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (MX.e4m3_encode(y.astype(np.float64)) == ref).all()


def test_scale_exponent():
    for k in range(-126, 128):
        assert MX.scale_exponent(2.0 ** k) == max(-127, k - 8)
        assert MX.scale_exponent(float(np.float32(2.0 ** k * (2 - 2.0 ** -23)))) == max(-127, k - 8)
    assert MX.scale_exponent(0.0) == -127
    assert MX.scale_exponent(float(np.float32(2.0 ** -140))) == -127   # fp32 subnormal
    assert MX.scale_exponent(2.0 ** -118) == -126
    assert MX.scale_exponent(2.0 ** -119) == -127


def test_block_invariants_and_vectorised_form():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    w[3, :32] = 0.0                                  # an all-zero block
    w[5, 32:64] *= np.float32(1e-30)                 # a block of tiny magnitude
    codes, sc = MX.quantize_tensor(w)
    for r in range(64):
        for b in range(8):
            c1, s1 = MX.quantize_block(w[r, 32 * b:32 * b + 32])
            assert (c1 == codes[r, 32 * b:32 * b + 32]).all() and s1 == sc[r, b]
    assert sc[3, 0] == 0 and (codes[3, :32] == 0).all()
    deq = MX.dequantize(codes.ravel(), sc.ravel()).reshape(64, 256)
    blocks = np.abs(w.astype(np.float64)).reshape(64, 8, 32)
    amax = blocks.max(axis=2)
    e = sc.astype(np.int64) - 127
    nz = amax > 0
    # the block maximum lands in [256, 448] * 2^e
    qmax = np.abs(deq).reshape(64, 8, 32).max(axis=2)
    assert (qmax[nz] >= 256 * np.ldexp(1.0, e[nz])).all()
    assert (qmax[nz] <= 448 * np.ldexp(1.0, e[nz])).all()
    # elements at or above the normal range keep 3 mantissa bits: rel. error <= 2^-4
    big = np.abs(w) >= np.repeat(np.ldexp(1.0, e - 6), 32, axis=1)
    unsat = np.abs(w) <= np.repeat(448 * np.ldexp(1.0, e), 32, axis=1)
    sel = big & unsat
    assert (np.abs(deq[sel] - w[sel]) <= 2.0 ** -4 * np.abs(w[sel])).all()


def test_requant_list_offsets():
    rng = np.random.default_rng(2)
    tensors = [(0, 4, 64), (256, 8, 32), (512, 2, 128)]
    w = rng.standard_normal(768).astype(np.float32)
    q, s = MX.requant_list(w, tensors)
    for off, rows, k in tensors:
        c, sc = MX.quantize_tensor(w[off:off + rows * k].reshape(rows, k))
        assert (q[off:off + rows * k] == c.ravel()).all()
        assert (s[off // 32:(off + rows * k) // 32] == sc.ravel()).all()


def test_power_of_two_multiples_of_codes_are_exact():
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 0x7F, size=(16, 64))
    codes[:, 0] = 0x7E                                    # force every block's amax
    codes[:, 32] = 0x7E                                   # to be 448 * 2^k
    sign = rng.integers(0, 2, size=codes.shape) * 0x80
    k = rng.integers(-20, 20, size=(16, 1))
    vals = MX.E4M3_TABLE[codes] * np.where(sign, -1.0, 1.0) * np.ldexp(1.0, k)
    q, s = MX.quantize_tensor(vals.astype(np.float32))
    expect = (codes | sign).astype(np.uint8)
    assert (q == expect).all()
    assert (s.astype(np.int64) - 127 == k).all()


def test_32x32_scale_is_the_max_of_its_row_block_scales():
    """floor(log2) and the clamp are monotone, so a 32 x 32 block's exponent is
    the largest of its 32 row-block (1 x 32) exponents; elements then use the
    same encoder with that exponent."""
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((96, 128)) * 0.02).astype(np.float32)
    w[:32, :32] *= np.float32(1e-6)                       # a block of tiny magnitude
    w[32:64, 64:96] = 0.0                                 # an all-zero block
    w[70, 100] = np.float32(3e4)                          # one outlier dominates its block
    c32, s32 = MX.quantize_tensor_32x32(w)
    c1, s1 = MX.quantize_tensor(w)
    assert (s32 == s1.reshape(3, 32, 4).max(axis=1)).all()
    e = s32.astype(np.int64) - 127
    for bi in range(3):
        for bj in range(4):
            blk = w[32 * bi:32 * bi + 32, 32 * bj:32 * bj + 32].astype(np.float64)
            want = MX.e4m3_encode(blk * np.ldexp(1.0, -e[bi, bj])).reshape(32, 32)
            assert (c32[32 * bi:32 * bi + 32, 32 * bj:32 * bj + 32] == want).all()
    assert s32[1, 2] == 0 and (c32[32:64, 64:96] == 0).all()


def test_scale_tile_128x4_structure():
    """The 128 x 4 tiled scale layout is a permutation of the padded scale
    matrix; each 512-byte tile holds exactly its 128 x 4 sub-block; inside a
    tile, the 16 bytes at 16 * l are rows l, l + 32, l + 64, l + 96 (4 scale
    columns each) - the 32-row interleave a 32-lane warp reads as one row per
    lane."""
    rng = np.random.default_rng(12)
    rows, kb = 256, 8
    sf = rng.integers(0, 255, size=(rows, kb)).astype(np.uint8)
    out = MX.scale_tile_128x4(sf)
    assert out.size == rows * kb and sorted(out.tolist()) == sorted(sf.ravel().tolist())
    ct = kb // 4
    for ti in range(rows // 128):
        for tj in range(ct):
            tile = out[(ti * ct + tj) * 512:(ti * ct + tj + 1) * 512]
            sub = sf[128 * ti:128 * ti + 128, 4 * tj:4 * tj + 4]
            assert sorted(tile.tolist()) == sorted(sub.ravel().tolist())
            for lane in range(32):
                grp = tile[16 * lane:16 * lane + 16].reshape(4, 4)
                assert (grp == sub[[lane, lane + 32, lane + 64, lane + 96], :]).all()
    # ragged sizes are zero-padded to whole tiles
    small = MX.scale_tile_128x4(np.full((5, 3), 7, np.uint8))
    assert small.size == 512 and int((small == 7).sum()) == 15
