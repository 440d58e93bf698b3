"""GPU parity of G with 32 x 32 MX blocks over ragged rank segments, and of
Tw's 128 x 4 scale relayout, against the oracle (bit-exact)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import mxfp8 as OX  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(hm):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _tensors(cfg):
    out, s_off = [], 0
    for m in cfg.members:
        out.append((m.offset, 0, s_off, m.rows, m.cols))
        s_off += (m.rows // 32) * (m.cols // 32)
    return out, s_off


@pytest.mark.parametrize("name", ["tiny_ragged", "mixed"])
def test_requant_32x32_over_ragged_segments(hm, dev, name):
    from head_muon_mxfp8_gb300.session import MuonSession
    cfg = workloads.get(name)
    w = workloads.generate(cfg, seed=23)["w"]
    w[:32 * cfg.members[0].cols] *= np.float32(1e-5)      # the first block row: tiny values
    s = MuonSession.from_config(cfg, device=dev)
    s.load("w", w)
    tensors, n_scales = _tensors(cfg)
    scales = torch.full((n_scales,), 0x5A, dtype=torch.uint8, device=dev)
    hm.mxfp8_requant_32x32(s.chain, s.w.data_ptr(), s.q.data_ptr(), scales.data_ptr(), tensors)
    torch.cuda.synchronize()
    q = s.fetch("q").numpy()
    sc = scales.cpu().numpy()
    for (off, _, s_off, rows, k) in tensors:
        codes, ref_s = OX.quantize_tensor_32x32(w[off:off + rows * k].reshape(rows, k))
        assert np.array_equal(q[off:off + rows * k], codes.ravel())
        assert np.array_equal(sc[s_off:s_off + ref_s.size], ref_s.ravel())
    ok = s.canary_intact()
    assert ok["q"] and ok["w"]
    assert hm.hm_device_error() == 0
    s.close()


def test_requant_32x32_flat(hm, dev):
    rng = np.random.default_rng(24)
    tensors = [(0, 0, 0, 64, 96), (64 * 96 + 512, 0, 6, 32, 32), (64 * 96 + 512 + 1024, 0, 7, 96, 64)]
    n = 64 * 96 + 512 + 1024 + 96 * 64
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    w[64 * 96:64 * 96 + 512] = 9.0
    wt = torch.from_numpy(w).to(dev)
    q = torch.full((n,), 0x5A, dtype=torch.uint8, device=dev)
    sc = torch.zeros(7 + 6, dtype=torch.uint8, device=dev)
    hm.mxfp8_requant_32x32(0, wt.data_ptr(), q.data_ptr(), sc.data_ptr(), tensors)
    torch.cuda.synchronize()
    qn, sn = q.cpu().numpy(), sc.cpu().numpy()
    for (off, _, s_off, rows, k) in tensors:
        codes, ref_s = OX.quantize_tensor_32x32(w[off:off + rows * k].reshape(rows, k))
        assert np.array_equal(qn[off:off + rows * k], codes.ravel())
        assert np.array_equal(sn[s_off:s_off + ref_s.size], ref_s.ravel())
    assert (qn[64 * 96:64 * 96 + 512] == 0x5A).all()           # the gap is untouched


def test_scale_relayout_128x4(hm, dev):
    """Aligned items take 4-byte source loads and 16-byte stores; the others
    (kb not a multiple of 4, a source or destination offset off alignment)
    take byte accesses: both must give the oracle's layout."""
    rng = np.random.default_rng(25)
    # rows, kb, block_rows, source pad before the item, destination gap after it
    mats = [(256, 8, 1, 0, 64), (200, 5, 1, 0, 67), (64, 6, 32, 0, 64), (1408, 64, 32, 0, 61),
            (128, 12, 1, 1, 64), (384, 16, 1, 3, 64),
            # wider than one 160-column work unit: exactly two, and two with a ragged second
            (256, 320, 1, 0, 64), (200, 200, 1, 0, 64), (96, 176, 32, 0, 64)]
    src_parts, items, refs = [], [], []
    s_off, d_off = 0, 0
    for rows, kb, br, s_pad, gap in mats:
        sf = rng.integers(0, 255, size=(rows // br, kb)).astype(np.uint8)
        src_parts.append(np.full(s_pad, 0x77, dtype=np.uint8))
        s_off += s_pad
        src_parts.append(sf.ravel())
        ref = OX.scale_tile_128x4(OX.expand_block_rows(sf, br) if br > 1 else sf)
        items.append((s_off, d_off, rows, kb, br))
        refs.append((d_off, ref))
        s_off += sf.size
        d_off += ref.size + gap                                 # a gap between outputs
    src = torch.from_numpy(np.concatenate(src_parts)).to(dev)
    dst = torch.full((d_off,), 0xEE, dtype=torch.uint8, device=dev)
    hm.mxfp8_scale_relayout(src.data_ptr(), dst.data_ptr(), items)
    torch.cuda.synchronize()
    out = dst.cpu().numpy()
    for (off, ref), m in zip(refs, mats):
        assert np.array_equal(out[off:off + ref.size], ref)
        assert (out[off + ref.size:off + ref.size + m[4]] == 0xEE).all()


def test_requant_32x32_fullsize_lm_sampled(hm, dev):
    """The LM layer (201 M elements, 8 ranks): every tensor requantised with
    32 x 32 blocks in one call; 2048 sampled blocks compared bit-exactly."""
    from head_muon_mxfp8_gb300.session import MuonSession
    cfg = workloads.get("lm_layer")
    s = MuonSession.from_config(cfg, device=dev)
    data = workloads.generate_device(cfg, dev, seed=29)
    s.load("w", data["w"])
    tensors, n_scales = _tensors(cfg)
    scales = torch.zeros(n_scales, dtype=torch.uint8, device=dev)
    hm.mxfp8_requant_32x32(s.chain, s.w.data_ptr(), s.q.data_ptr(), scales.data_ptr(), tensors)
    torch.cuda.synchronize()
    w = data["w"].cpu().numpy()
    q = s.fetch("q").numpy()
    sc = scales.cpu().numpy()
    rng = np.random.default_rng(3)
    for _ in range(2048):
        t = int(rng.integers(len(tensors)))
        off, _, s_off, rows, k = tensors[t]
        br, bc = int(rng.integers(rows // 32)), int(rng.integers(k // 32))
        blk = w[off:off + rows * k].reshape(rows, k)[32 * br:32 * br + 32, 32 * bc:32 * bc + 32]
        codes, ref_s = OX.quantize_tensor_32x32(blk)
        got = q[off:off + rows * k].reshape(rows, k)[32 * br:32 * br + 32, 32 * bc:32 * bc + 32]
        assert np.array_equal(got, codes) and sc[s_off + br * (k // 32) + bc] == ref_s[0, 0]
    s.close()
