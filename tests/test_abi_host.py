"""Host-side checks of libhm that need no GPU: the library loads and exports
every function the header declares; the shard chain, segment layout,
fragments and Muon plan agree exactly with the oracle; invalid metadata is
rejected with the documented status before anything is launched."""
import ctypes as C

import numpy as np
import pytest

import workloads
from oracle import views as V


def test_exports_every_header_symbol(hm):
    names = hm.header_symbols()
    assert len(names) >= 20
    for name in names:
        assert hasattr(hm.lib(), name), name
    assert set(hm._SIGS) == set(names)


def test_status_strings(hm):
    assert hm.status_str(hm.HM_OK) == "HM_OK"
    assert hm.status_str(hm.HM_ERR_OVERLAP) == "HM_ERR_OVERLAP"


CHAIN_CASES = [(196608, 4, 2, 2), (1024, 4, 2, 2), (32 * 1001, 8, 4, 4), (32 * 517, 8, 2, 4),
               (32 * 4099, 16, 8, 8), (32 * 12345, 32, 16, 16), (64, 4, 2, 2), (0, 2, 1, 1), (32 * 77, 1, 1, 1)]


@pytest.mark.parametrize("n,so,sw,sg", CHAIN_CASES)
def test_chain_layout_matches_oracle(hm, n, so, sw, sg):
    ch = hm.shard_chain(n, so, sw, sg)
    total, bases, lens, chunks = hm.shard_chain_layout(ch, so)
    e = V.z1_edges(n, so)
    obases, ototal = V.segment_layout(e, so, sw)
    assert total == ototal and bases == obases
    assert chunks == [V.chunk_of_rank(r, so, sw) for r in range(so)]
    assert lens == [e[c + 1] - e[c] for c in chunks]
    rng = np.random.default_rng(n + so)
    for _ in range(20):
        a, b = sorted(32 * rng.integers(0, n // 32 + 1, 2)) if n else (0, 0)
        got = hm.shard_chain_fragments(ch, int(a), int(b), 1)
        want = V.fragments(int(a), int(b), e, so, sw, obases)
        assert [(f.chunk, f.rank, f.seg_offset, f.unit_offset, f.length, f.root_offset) for f in got] == \
               [(w.chunk, w.rank, w.seg_offset, w.unit_offset, w.length, w.root_offset) for w in want]
        for level, s in ((2, sg), (3, sw)):
            got = hm.shard_chain_fragments(ch, int(a), int(b), level)
            cov = sum(f.length for f in got)
            assert cov == b - a
            for f in got:
                lo, hi = V.level_range(e, so, s, f.chunk)
                assert lo <= a + f.unit_offset and a + f.unit_offset + f.length <= hi
                assert V.rank_level_chunk(f.rank, so, sw, s) == f.chunk
    hm.chain_destroy(ch)


def test_chain_jittered_edges(hm):
    n, so, sw = 32 * 1000, 8, 4
    e = V.z1_edges(n, so)
    rng = np.random.default_rng(5)
    j = [e[0]] + [x + 32 * int(rng.integers(-3, 4)) for x in e[1:-1]] + [e[-1]]
    ch = hm.shard_chain(n, so, sw, sw, j)
    total, bases, lens, chunks = hm.shard_chain_layout(ch, so)
    ob, ot = V.segment_layout(j, so, sw)
    assert bases == ob and total == ot
    hm.chain_destroy(ch)


def test_chain_edge_shift(hm):
    n, so, sw = 32 * 1000, 8, 4
    sh = workloads.ragged_shift(so, 5, seed=3)
    ch = hm.shard_chain(n, so, sw, sw, None, sh)
    total, bases, lens, chunks = hm.shard_chain_layout(ch, so)
    e = V.z1_edges(n, so, sh)
    assert lens == [e[c + 1] - e[c] for c in chunks]
    assert (bases, total) == V.segment_layout(e, so, sw)
    hm.chain_destroy(ch)
    with pytest.raises(hm.HmError) as err:
        hm.shard_chain(n, so, sw, sw, None, [0, 16] + [0] * (so - 1))
    assert err.value.status == hm.HM_ERR_ALIGN
    with pytest.raises(hm.HmError) as err:
        hm.shard_chain(n, so, sw, sw, None, [32] + [0] * so)
    assert err.value.status == hm.HM_ERR_GEOMETRY
    with pytest.raises(hm.HmError) as err:
        hm.shard_chain(n, so, sw, sw, None, [0, 32 * 5000] + [0] * (so - 1))
    assert err.value.status == hm.HM_ERR_GEOMETRY


def test_chain_rejections(hm):
    with pytest.raises(hm.HmError) as e:
        hm.shard_chain(100, 4, 2, 2)
    assert e.value.status == hm.HM_ERR_ALIGN
    with pytest.raises(hm.HmError) as e:
        hm.shard_chain(1024, 8, 3, 3)
    assert e.value.status == hm.HM_ERR_GEOMETRY
    with pytest.raises(hm.HmError) as e:
        hm.shard_chain(1024, 8, 4, 2)          # sw must divide sg
    assert e.value.status == hm.HM_ERR_GEOMETRY
    with pytest.raises(hm.HmError) as e:
        hm.shard_chain(1024, 2, 1, 1, [0, 48, 1024])
    assert e.value.status == hm.HM_ERR_ALIGN
    with pytest.raises(hm.HmError) as e:
        hm.shard_chain(1024, 2, 1, 1, [0, 640, 512])
    assert e.value.status == hm.HM_ERR_GEOMETRY
    with pytest.raises(hm.HmError) as e:
        hm.shard_chain(1024, 0, 1, 1)
    assert e.value.status == hm.HM_ERR_ARG


@pytest.mark.parametrize("name", ["tiny", "lm_layer", "moe_layer", "video_dit"])
def test_plan_matches_oracle(hm, name):
    cfg = workloads.get(name)
    ch = hm.shard_chain(cfg.numel, cfg.so, cfg.sw, cfg.sg, None, cfg.edge_shift)
    units = [(u.offset, u.rows, u.cols) for u in cfg.units]
    plan = hm.muon_plan(ch, units)
    info = hm.muon_plan_query(plan)
    e = V.z1_edges(cfg.numel, cfg.so, cfg.edge_shift)
    bases, _ = V.segment_layout(e, cfg.so, cfg.sw)
    n_strad = 0
    for i, (o, r, c) in enumerate(units):
        fr = V.fragments(o, o + r * c, e, cfg.so, cfg.sw, bases)
        pu = hm.muon_plan_unit(plan, i)
        assert pu["n_frags"] == len(fr)
        assert pu["exec_rank"] == V.execution_rank(fr)
        assert pu["local"] == (len(fr) == 1)
        n_strad += len(fr) > 1
    assert info.n_units == len(units) and info.n_straddling == n_strad
    shapes = {(min(r, c), max(r, c)) for (_, r, c) in units}
    assert info.n_classes == len(shapes)
    assert info.workspace_bytes > 0
    if name == "moe_layer":
        assert n_strad == 15            # every interior edge splits one expert matrix
    hm.muon_plan_destroy(plan)
    hm.chain_destroy(ch)


def test_plan_rejections(hm):
    ch = hm.shard_chain(1024, 4, 2, 2)
    with pytest.raises(hm.HmError) as e:
        hm.muon_plan(ch, [(0, 16, 32), (544, 15, 32)])      # gap between units
    assert e.value.status == hm.HM_ERR_UNITS
    with pytest.raises(hm.HmError) as e:
        hm.muon_plan(ch, [(0, 16, 32)])                     # does not reach the end
    assert e.value.status == hm.HM_ERR_UNITS
    with pytest.raises(hm.HmError) as e:
        hm.muon_plan(ch, [(0, 5, 7)] + [(35, 1, 989)])      # not 32-aligned
    assert e.value.status == hm.HM_ERR_ALIGN
    plan = hm.muon_plan(ch, [(0, 16, 32), (512, 16, 32)])
    bufs = hm.hm_muon_bufs(16, 16, 16, 16, 16, 16, 16)
    hp = hm.hm_muon_hparams(0.02, 0.95, 0.0, 1e-7, 3.4445, -4.775, 2.0315, 5, 0, 0)
    st = hm.lib().muon_update_units(C.c_void_p(plan), C.byref(bufs), C.byref(hp), C.c_void_p(1 << 20), 1 << 20,
                                    hm.HM_STAGE_ALL, None)
    assert st == hm.HM_ERR_STATE                            # workspace never uploaded
    hm.muon_plan_destroy(plan)
    hm.chain_destroy(ch)


def test_stage_sets_are_checked_before_any_device_work(hm):
    """Which stage sets muon_update_units accepts is decided on the host,
    before the workspace is looked at: rejected sets return HM_ERR_ARG,
    accepted ones get as far as the missing upload (HM_ERR_STATE)."""
    ch = hm.shard_chain(1024, 4, 2, 2)
    plan = hm.muon_plan(ch, [(0, 16, 32), (512, 16, 32)])
    bufs = hm.hm_muon_bufs(16, 16, 16, 16, 16, 16, 16)
    hp = hm.hm_muon_hparams(0.02, 0.95, 0.0, 1e-7, 3.4445, -4.775, 2.0315, 5, 0, 0)
    F0, GA, NS, F2, RQ = hm.HM_STAGE_F0, hm.HM_STAGE_GATHER, hm.HM_STAGE_NS, hm.HM_STAGE_F2, hm.HM_STAGE_REQUANT
    FU, SC = hm.HM_STAGE_FUSED, hm.HM_STAGE_SCRATCH
    accepted = [hm.HM_STAGE_ALL, hm.HM_STAGE_ALL_FUSED, hm.HM_STAGE_STEP, F0, NS, F2 | RQ, F0 | GA | FU,
                F2 | RQ | FU, NS | F2 | RQ | FU, F0 | GA | FU | SC, NS | F2 | RQ | FU | SC, F2 | RQ | FU | SC,
                NS | FU]
    rejected = [-1, hm.HM_STAGE_STEP + 1, 128, F0 | FU, GA | FU, F2 | FU, RQ | FU, F0 | GA | F2 | FU,
                hm.HM_STAGE_ALL | SC, F0 | GA | SC, NS | SC, NS | FU | SC, NS | F2 | FU | SC, NS | F2 | RQ | SC]
    for stages in accepted + rejected:
        st = hm.lib().muon_update_units(C.c_void_p(plan), C.byref(bufs), C.byref(hp), C.c_void_p(1 << 20), 1 << 20,
                                        stages, None)
        want = hm.HM_ERR_STATE if stages in accepted else hm.HM_ERR_ARG
        assert st == want, (stages, st)
    hm.muon_plan_destroy(plan)
    hm.chain_destroy(ch)


def test_data_tree_views_alias_the_root(hm):
    base = 0x10000000
    t = hm.create_data_tree(base, 1 << 20)
    qkv = hm.data_tree_add_view(t, 0, 4096, hm.HM_F32, [768, 256])
    head3 = hm.data_tree_add_view(t, qkv, 3 * 64 * 256 * 4, hm.HM_F32, [64, 256])
    ptr, off = hm.data_tree_resolve(t, head3)
    assert off == 4096 + 3 * 64 * 256 * 4 and ptr == base + off
    with pytest.raises(hm.HmError) as e:
        hm.data_tree_add_view(t, head3, 4, hm.HM_F32, [64, 256])   # past the head's end
    assert e.value.status == hm.HM_ERR_GEOMETRY
    with pytest.raises(hm.HmError) as e:
        hm.data_tree_add_view(t, qkv, 2, hm.HM_F32, [4])
    assert e.value.status == hm.HM_ERR_ALIGN
    h4 = hm.data_tree_add_view(t, qkv, 4 * 64 * 256 * 4, hm.HM_F32, [64, 256])
    assert hm.data_tree_check_disjoint(t, [head3, h4]) == hm.HM_OK
    assert hm.data_tree_check_disjoint(t, [head3, qkv]) == hm.HM_ERR_OVERLAP
    hm.tree_destroy(t)


def test_segment_views(hm):
    n, so, sw = 196608, 4, 2
    ch = hm.shard_chain(n, so, sw, sw)
    total, bases, lens, _ = hm.shard_chain_layout(ch, so)
    t = hm.create_data_tree(0x40000000, total * 4)
    nodes = hm.shard_chain_segment_views(ch, t, hm.HM_F32, so)
    for r, nd in enumerate(nodes):
        assert hm.data_tree_resolve(t, nd)[1] == bases[r] * 4
    assert hm.data_tree_check_disjoint(t, nodes) == hm.HM_OK
    small = hm.create_data_tree(0x40000000, total * 2)
    with pytest.raises(hm.HmError) as e:
        hm.shard_chain_segment_views(ch, small, hm.HM_F32, so)
    assert e.value.status == hm.HM_ERR_GEOMETRY
    hm.tree_destroy(t)
    hm.tree_destroy(small)
    hm.chain_destroy(ch)


def test_checks_that_precede_any_launch(hm):
    L = hm.lib()
    hp = hm.hm_adamw_hparams(1e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    assert L.adamw_update_flat(None, None, hm.HM_BF16, None, None, 0, C.byref(hp), None) == hm.HM_OK
    assert L.adamw_update_flat(None, None, 7, None, None, 16, C.byref(hp), None) == hm.HM_ERR_DTYPE
    assert L.adamw_update_flat(C.c_void_p(16), C.c_void_p(18), hm.HM_BF16, C.c_void_p(16), C.c_void_p(16), 16,
                               C.byref(hp), None) == hm.HM_ERR_ALIGN
    bad = hm.hm_adamw_hparams(1e-4, 0.9, 0.95, 1e-8, 0.1, 0)
    assert L.adamw_update_flat(None, None, hm.HM_BF16, None, None, 16, C.byref(bad), None) == hm.HM_ERR_ARG
    arr = (hm.hm_mx_tensor * 1)(hm.hm_mx_tensor(0, 0, 0, 4, 48))
    assert L.mxfp8_requant_packed(C.c_void_p(256), C.c_void_p(256), C.c_void_p(256), arr, 1, None) == \
        hm.HM_ERR_ALIGN
    assert L.mxfp8_requant_packed(None, None, None, None, 0, None) == hm.HM_OK


def test_kernel_launch_counter_is_host_only(hm):
    """The launch counter reads without a device, and a call rejected by its
    host-side checks launches nothing."""
    n0 = hm.hm_kernel_launches()
    assert n0 >= 0
    assert hm.lib().adamw_update_flat(None, None, hm.HM_BF16, None, None, 16, None, None) == hm.HM_ERR_ARG
    assert hm.hm_kernel_launches() == n0
