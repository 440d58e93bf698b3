"""Pins for oracle.views: data tree, shard chain, fragments, segment layout."""
import os

import numpy as np
import pytest

from oracle import views as V

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fig4_shard_chain.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def test_fig4_owners_and_groups():
    g = _golden()
    so, sw, sg = int(g["so"][0]), int(g["sw"][0]), int(g["sg"][0])
    assert [V.owner(c, so, sw) for c in range(so)] == [int(x) for x in g["owners"]]
    n = 1024
    e = V.z1_edges(n, so)
    # outer groups: ranks sharing one z3 chunk; their z1 chunks tile it contiguously
    for grp in g["outer_groups"]:
        ranks = [int(x) for x in grp.split(",")]
        z3 = {V.rank_level_chunk(r, so, sw, sw) for r in ranks}
        assert len(z3) == 1
        lo, hi = V.level_range(e, so, sw, z3.pop())
        chunks = sorted(V.chunk_of_rank(r, so, sw) for r in ranks)
        assert e[chunks[0]] == lo and e[chunks[-1] + 1] == hi
        assert chunks == list(range(chunks[0], chunks[-1] + 1))
    # runtime groups: their z3 chunks cover the whole buffer
    for grp in g["runtime_groups"]:
        ranks = [int(x) for x in grp.split(",")]
        ks = sorted(V.rank_level_chunk(r, so, sw, sw) for r in ranks)
        assert ks == list(range(sw))


def test_fig4_head0_spans_ranks_2_and_1():
    g = _golden()
    so, sw = int(g["so"][0]), int(g["sw"][0])
    # tensor list: Linear (448 elements) then Head0..Head2 (192 each); N = 1024
    n = 1024
    e = V.z1_edges(n, so)
    bases, _ = V.segment_layout(e, so, sw)
    fr = V.fragments(448, 640, e, so, sw, bases)
    assert [f.rank for f in fr] == [int(x) for x in g["head0_ranks"]]
    assert V.execution_rank(fr) == int(g["head0_exec"][0])
    assert len(V.fragments(832, 1024, e, so, sw, bases)) == 1  # Head2 is local


def test_edges_properties():
    for n in [0, 32, 96, 196608, 201326592, 1024 * 37]:
        for so in [1, 2, 4, 8, 16, 32]:
            e = V.z1_edges(n, so)
            assert e[0] == 0 and e[-1] == n
            assert all(x % 32 == 0 for x in e)
            d = np.diff(e)
            assert (d >= 0).all() and d.max() - d.min() <= 32
    with pytest.raises(ValueError):
        V.z1_edges(100, 4)


def _brute_rank_map(n, so, sw):
    e = V.z1_edges(n, so)
    rk = np.empty(n, dtype=np.int64)
    ck = np.empty(n, dtype=np.int64)
    for p in range(n):  # per element: which chunk holds p, who owns it
        c = max(i for i in range(so) if e[i] <= p < e[i + 1])
        ck[p] = c
        rk[p] = V.owner(c, so, sw)
    return rk, ck


@pytest.mark.parametrize("so,sw", [(1, 1), (2, 1), (4, 2), (8, 4), (8, 2), (16, 8)])
def test_fragments_match_brute_force(so, sw):
    rng = np.random.default_rng(so * 10 + sw)
    n = 32 * int(rng.integers(so, 40 * so))
    rk, ck = _brute_rank_map(n, so, sw)
    e = V.z1_edges(n, so)
    bases, total = V.segment_layout(e, so, sw)
    root = V.to_segments(np.arange(n, dtype=np.int64), e, so, sw, fill=-1)
    cuts = np.sort(rng.choice(np.arange(1, n // 32), size=min(6, n // 32 - 1), replace=False)) * 32
    bounds = [0] + list(cuts) + [n]
    for a, b in zip(bounds[:-1], bounds[1:]):
        fr = V.fragments(a, b, e, so, sw, bases)
        assert sum(f.length for f in fr) == b - a
        pos = a
        for f in fr:
            assert f.unit_offset == pos - a
            assert (rk[pos:pos + f.length] == f.rank).all()
            assert (ck[pos:pos + f.length] == f.chunk).all()
            pos += f.length
        # a new fragment starts exactly where the chunk changes
        starts = {f.unit_offset + a for f in fr}
        for p in range(a + 1, b):
            assert (ck[p] != ck[p - 1]) == (p in starts)
        assert (V.gather(root, fr, b - a) == np.arange(a, b)).all()


def test_segment_layout_alignment_and_canaries():
    for n, so, sw in [(196608, 4, 2), (4096 * 7, 8, 4), (32 * 3, 4, 2)]:
        e = V.z1_edges(n, so)
        bases, total = V.segment_layout(e, so, sw)
        prev_end = 0
        for r in range(so):
            c = V.chunk_of_rank(r, so, sw)
            assert bases[r] % V.ALIGN == 0
            assert bases[r] - prev_end >= V.GAP
            prev_end = bases[r] + e[c + 1] - e[c]
        assert total - prev_end >= V.GAP
        mask = V.canary_mask(e, so, sw)
        assert (~mask).sum() == n


def test_gather_scatter_inverse():
    rng = np.random.default_rng(3)
    n, so, sw = 32 * 500, 8, 4
    e = V.z1_edges(n, so)
    bases, total = V.segment_layout(e, so, sw)
    logical = rng.standard_normal(n).astype(np.float32)
    root = V.to_segments(logical, e, so, sw, fill=np.float32(7.0))
    assert (V.from_segments(root, e, so, sw) == logical).all()
    a, b = 32 * 37, 32 * 311
    fr = V.fragments(a, b, e, so, sw, bases)
    assert len(fr) > 1
    unit = V.gather(root, fr, b - a)
    root2 = np.full_like(root, 7.0)
    V.scatter(root2, fr, unit)
    # scatter(gather(x)) restores exactly the unit's elements and nothing else
    touched = np.zeros(total, dtype=bool)
    for f in fr:
        touched[f.root_offset:f.root_offset + f.length] = True
    assert (root2[touched] == root[touched]).all()
    assert (root2[~touched] == 7.0).all()
    # gather(scatter(y)) == y
    y = rng.standard_normal(b - a).astype(np.float32)
    V.scatter(root2, fr, y)
    assert (V.gather(root2, fr, b - a) == y).all()


def test_levels_nest():
    for so, sw, sg in [(4, 2, 2), (8, 2, 4), (16, 8, 8), (32, 16, 16), (8, 1, 8)]:
        V.check_degrees(so, sw, sg)
        e = V.z1_edges(32 * 1000, so)
        for r in range(so):
            c = V.chunk_of_rank(r, so, sw)
            z1 = (e[c], e[c + 1])
            z2 = V.level_range(e, so, sg, V.rank_level_chunk(r, so, sw, sg))
            z3 = V.level_range(e, so, sw, V.rank_level_chunk(r, so, sw, sw))
            assert z3[0] <= z2[0] <= z1[0] and z1[1] <= z2[1] <= z3[1]
        assert sorted(V.owner(c, so, sw) for c in range(so)) == list(range(so))
    with pytest.raises(ValueError):
        V.check_degrees(8, 3, 3)
    with pytest.raises(ValueError):
        V.check_degrees(8, 4, 2)


def test_data_tree_aliases_root():
    t = V.DataTree(4096)
    child = t.add_view(0, 256, np.float32, (16, 8))
    grand = t.add_view(child, 64, np.float32, (8,))
    assert t.resolve(grand) == 320
    t.view(grand)[:] = np.arange(8, dtype=np.float32)
    assert (t.storage[320:352].view(np.float32) == np.arange(8)).all()
    assert (t.view(child).ravel()[16:24] == np.arange(8)).all()
    with pytest.raises(ValueError):
        t.add_view(child, 512, np.float32, (8,))      # exceeds the 512-byte child
    with pytest.raises(ValueError):
        t.add_view(0, 2, np.float32, (4,))            # misaligned
