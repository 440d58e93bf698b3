"""The benchmark's FLOP counts: the algorithmic count is the closed form
5 (4 m^2 n + 2 m^3) per unit; the executed count matches a brute-force walk
over the tiles each kernel computes (single-CTA 128-row tiles, or 256 x 256
CTA-pair tiles when the padded Gram size is a multiple of 256)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
import workloads  # noqa: E402


def _brute_executed(m, n, steps):
    mp, np_ = -(-m // 128) * 128, -(-n // 64) * 64
    tot = 0
    if mp % 256 == 0:
        t = mp // 256
        for tm in range(t):
            for tn in range(t):
                if tn >= tm:  # X X^T (K = np) and bA + cAA (K = mp) on the upper triangle
                    tot += 2 * 256 * 256 * np_ + 2 * 256 * 256 * mp
        for tm in range(t):
            for tn in range(-(-np_ // 256)):  # B X on the full grid, K = mp
                tot += 2 * 256 * 256 * mp
    else:
        bn = 256 if mp >= 256 else 128
        for tm in range(mp // 128):
            for tn in range(-(-mp // bn)):
                if tn * bn + bn - 1 >= tm * 128:
                    tot += 2 * 128 * bn * np_ + 2 * 128 * bn * mp
        bn3 = 256 if np_ >= 256 else 128
        for tm in range(mp // 128):
            for tn in range(-(-np_ // bn3)):
                tot += 2 * 128 * bn3 * mp
    return steps * tot


def test_algorithmic_flops_closed_form():
    cfg = workloads.get("video_dit")
    assert bench.ns_flops(cfg, 5) == 960 * 5 * (4 * 128**2 * 5120 + 2 * 128**3) + \
        16 * 5 * (4 * 5120**2 * 20480 + 2 * 5120**3)


def test_executed_flops_match_the_tile_walk():
    for shapes in ([(128, 5120)], [(1408, 2048)], [(5120, 20480)], [(96, 160)], [(384, 640)], [(4096, 14336)]):
        cfg = workloads.scaled_muon("f", [(r, c, None) for r, c in shapes], so=1, sw=1, sg=1)
        m, n = min(shapes[0]), max(shapes[0])
        assert bench.ns_executed_flops(cfg, 5) == _brute_executed(m, n, 5), shapes
