"""Failure detection on the GPU without a fault: a Newton-Schulz GEMM whose
accumulator is never marked ready (test hook HM_INJECT_NS_WAIT_TIMEOUT) must
give up on its bounded waits, record HM_ERR_TIMEOUT in the device error
word, free its resources and return; the context stays usable and the next
update is correct."""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402

from muon_parity import check_f0, check_ns  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(hm):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.mark.parametrize("name", ["tiny", "heads1", "single", "pair", "paced"])
def test_injected_wait_timeout_is_reported_and_recovered(hm, dev, name):
    """tiny: 12 units of Gram size 128 on the one-launch kernel, each unit
    split over a CTA pair (the Gram pass never marks A ready, the peer waits
    on cluster barriers); heads1: 100 such units, one CTA each; single: a
    384 x 640 class on the single-CTA GEMM (Gram size not a multiple of 256);
    pair: a 512 x 768 class, whose GEMMs run on CTA pairs (cta_group::2);
    paced: two 256 x 139264 units, whose X (71 MB each) is more than half the
    L2, so the pairs also wait on each other's progress (bounded) while the
    injected wait runs out."""
    from head_muon_mxfp8_gb300.session import MuonSession, muon_hparams
    if name == "heads1":
        cfg = workloads.scaled_muon("heads1", [(64, 128, None)] * 100, so=4, sw=2, sg=2)
    elif name == "single":
        cfg = workloads.scaled_muon("single", [(384, 640, None), (640, 384, None)], so=4, sw=2, sg=2)
    elif name == "pair":
        cfg = workloads.scaled_muon("pair", [(512, 768, None), (768, 512, None)], so=4, sw=2, sg=2)
    elif name == "paced":
        cfg = workloads.scaled_muon("paced", [(256, 139264, None), (139264, 256, None)], so=4, sw=2, sg=2)
    else:
        cfg = workloads.get("tiny")
    data = workloads.generate(cfg, seed=41)
    s = MuonSession.from_config(cfg, device=dev)
    s.load("w", data["w"])
    s.load("g", data["g"])
    s.load("m", np.zeros_like(data["w"]))
    hp = muon_hparams(cfg.muon)
    assert hm.hm_device_error() == 0
    os.environ["HM_INJECT_NS_WAIT_TIMEOUT"] = "1"
    try:
        s.run(hp, hm.HM_STAGE_F0 | hm.HM_STAGE_GATHER | hm.HM_STAGE_NS)
        torch.cuda.synchronize()                  # returns: the waits are bounded
    finally:
        del os.environ["HM_INJECT_NS_WAIT_TIMEOUT"]
    assert hm.hm_device_error() == hm.HM_ERR_TIMEOUT
    assert hm.hm_device_error() == 0              # read-and-clear
    # the context is intact: a clean update gives the right answer
    s.load("m", np.zeros_like(data["w"]))
    s.run(hp, hm.HM_STAGE_F0 | hm.HM_STAGE_GATHER | hm.HM_STAGE_NS)
    torch.cuda.synchronize()
    assert hm.hm_device_error() == 0
    m = s.fetch("m").numpy()
    u = s.fetch("u").numpy().view(np.uint16)
    check_f0(np.zeros_like(data["w"]), data["g"], m, u, cfg.muon.momentum)
    v = s.fetch("v").numpy()
    for i, un in enumerate(cfg.units):            # straddling units keep v in the staging
        v[un.offset:un.offset + un.numel] = s.unit_v(i).numpy()
    check_ns(cfg, u, v, cfg.muon)
    s.close()
