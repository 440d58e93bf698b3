"""Seeded synthetic workloads for the update phase of runtime/update-decoupled
sharded data parallelism (SS-HSDP).

This module is shared by the CUDA path's tests/bench and by the CPU oracle.
It holds input *structure* and seeded random draws only: tensor-list members
with their shapes, the update units carved out of them, the hyperparameters
handed to the optimizer, and seeded Gaussian inputs.  It contains none of the
method's arithmetic: no shard edges, no owner map, no segment layout, no
momentum, Newton-Schulz, AdamW or MXFP8 step.  Those live separately in the
oracle (CPU) and in the C-ABI library (GPU).

Layout conventions (SS-HSDP paper, section 3.1 example EG1 and Appendix A):
  * a weight matrix is stored row-major as [out][in]; the packed QKV
    projection is [3*H*dh][d] with all Q heads, then K heads, then V heads;
    each head is a contiguous dh x d block, i.e. "consecutive views";
  * one tensor list per config: members are concatenated in the order listed
    (per layer: QKV, then the MLP / expert matrices);
  * an update unit is a contiguous r x c row-major block of the flat list
    (one head, one whole matrix or one expert matrix).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np


@dataclass(frozen=True)
class Member:
    """One tensor of the flat tensor list: rows x cols, row-major."""
    name: str
    rows: int
    cols: int
    offset: int  # element offset in the flat list

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass(frozen=True)
class Unit:
    """One update unit: a contiguous rows x cols row-major block."""
    offset: int
    rows: int
    cols: int
    member: int  # index of the member it belongs to

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass
class MuonHparams:
    lr: float = 0.02
    momentum: float = 0.95
    nesterov: bool = False
    ns_steps: int = 5
    ns_a: float = 3.4445
    ns_b: float = -4.7750
    ns_c: float = 2.0315
    eps: float = 1e-7
    alpha_mode: int = 0   # 0: alpha = 1
    weight_decay: float = 0.0


@dataclass
class AdamWHparams:
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1


@dataclass
class Config:
    name: str
    description: str
    optimizer: str               # "muon" or "adamw"
    members: List[Member]
    units: List[Unit]
    so: int                      # ZeRO-1 sharding degree (emulated ranks)
    sw: int                      # ZeRO-3 degree
    sg: int                      # ZeRO-2 degree
    edge_shift: Optional[List[int]] = None   # ragged ZeRO-1 edges: per-edge 32-aligned shift
    w_std: float = 0.02
    g_std: float = 1e-3
    seed: int = 0
    muon: MuonHparams = field(default_factory=MuonHparams)
    adamw: AdamWHparams = field(default_factory=AdamWHparams)

    @property
    def numel(self) -> int:
        return sum(m.numel for m in self.members)

    @property
    def mx_tensors(self) -> List[Tuple[int, int, int]]:
        """(flat offset, rows, K) of every runtime weight; K is the contiguous
        (reduction) dimension, so a 1x32 block runs along K."""
        return [(m.offset, m.rows, m.cols) for m in self.members]


class _ListBuilder:
    def __init__(self) -> None:
        self.members: List[Member] = []
        self.units: List[Unit] = []
        self.off = 0

    def add(self, name: str, rows: int, cols: int, unit_rows: Optional[int] = None) -> None:
        """Append a [rows][cols] member.  unit_rows=None: the whole matrix is one
        unit; otherwise it is cut into consecutive unit_rows x cols blocks."""
        idx = len(self.members)
        self.members.append(Member(name, rows, cols, self.off))
        if unit_rows is None:
            self.units.append(Unit(self.off, rows, cols, idx))
        else:
            assert rows % unit_rows == 0
            for h in range(rows // unit_rows):
                self.units.append(Unit(self.off + h * unit_rows * cols, unit_rows, cols, idx))
        self.off += rows * cols


def _qkv(b: _ListBuilder, prefix: str, d: int, hq: int, hkv: int, dh: int) -> None:
    b.add(prefix + "qkv", (hq + 2 * hkv) * dh, d, unit_rows=dh)


def tiny() -> Config:
    b = _ListBuilder()
    _qkv(b, "", d=256, hq=4, hkv=4, dh=64)
    return Config("tiny", "1 layer, hidden 256, 4 heads x 64; packed QKV [768][256]; "
                  "12 per-head 64x256 Muon units; 4 emulated ranks",
                  "muon", b.members, b.units, so=4, sw=2, sg=2)


def flat_adamw() -> Config:
    b = _ListBuilder()
    b.add("flat", 16384, 4096)
    return Config("flat_adamw", "one 64M-element fp32 shard, AdamW, bf16 grads; "
                  "MXFP8 requant as 16384x4096", "adamw", b.members, [], so=1, sw=1, sg=1)


def lm_layer() -> Config:
    b = _ListBuilder()
    _qkv(b, "", d=4096, hq=32, hkv=8, dh=128)
    b.add("gate", 14336, 4096)
    b.add("up", 14336, 4096)
    b.add("down", 4096, 14336)
    return Config("lm_layer", "hidden 4096, 32 q + 8 kv heads x 128 (48 per-head 128x4096 "
                  "units), MLP gate/up [14336][4096] and down [4096][14336] whole-matrix; "
                  "8 emulated ranks", "muon", b.members, b.units, so=8, sw=4, sg=4)


def ragged_shift(so: int, max_blocks: int, seed: int) -> List[int]:
    """A seeded ragged-edge shift: interior edges move by a nonzero multiple of
    32 elements, at most max_blocks * 32 either way; the end edges stay."""
    rng = np.random.default_rng(seed)
    mag = rng.integers(1, max_blocks + 1, so + 1)
    sign = np.where(rng.integers(0, 2, so + 1) == 0, -1, 1)
    sh = [int(32 * m * s) for m, s in zip(mag, sign)]
    sh[0] = sh[so] = 0
    return sh


def moe_layer(experts: int = 64) -> Config:
    b = _ListBuilder()
    for e in range(experts):
        b.add(f"gate{e}", 1408, 2048)
    for e in range(experts):
        b.add(f"up{e}", 1408, 2048)
    for e in range(experts):
        b.add(f"down{e}", 2048, 1408)
    # even edges would fall exactly on expert boundaries (12 matrices per rank);
    # ragged edges make every one of the 15 interior edges split a matrix
    name = "moe_layer" if experts == 64 else f"moe_layer_{experts}e"
    return Config(name, f"{experts} experts, gate/up [1408][2048], down [2048][1408]; "
                  f"{3 * experts} expert-matrix Muon units; 16 emulated ranks with ragged edges",
                  "muon", b.members, b.units, so=16, sw=8, sg=8,
                  edge_shift=ragged_shift(16, 2048 * experts // 64, seed=16))


def video_dit(layers: int = 8) -> Config:
    b = _ListBuilder()
    for l in range(layers):
        _qkv(b, f"l{l}.", d=5120, hq=40, hkv=40, dh=128)
        b.add(f"l{l}.fc1", 20480, 5120)
        b.add(f"l{l}.fc2", 5120, 20480)
    return Config("video_dit", f"{layers} layers, hidden 5120, 40 heads x 128 (120 per-head "
                  "128x5120 units per layer), MLP fc1 [20480][5120] + fc2 [5120][20480] "
                  "whole-matrix; 32 emulated ranks",
                  "muon", b.members, b.units, so=32, sw=16, sg=16)


def video_dit_layer() -> Config:
    """One Video-DiT layer (120 heads, fc1, fc2; 288 M parameters): the same
    shape classes at one eighth of the size, for profiling captures that must
    stay a few GB on the device."""
    c = video_dit(layers=1)
    return Config("video_dit_layer", "1 layer of video_dit: hidden 5120, 120 per-head 128x5120 units, "
                  "fc1 [20480][5120] + fc2 [5120][20480]; 32 emulated ranks",
                  "muon", c.members, c.units, so=c.so, sw=c.sw, sg=c.sg)


def scaled_muon(name: str, shapes: List[Tuple[int, int, Optional[int]]], so: int,
                sw: int, sg: int) -> Config:
    """A free-form Muon config for tests: (rows, cols, unit_rows or None)."""
    b = _ListBuilder()
    for i, (r, c, ur) in enumerate(shapes):
        b.add(f"t{i}", r, c, unit_rows=ur)
    return Config(name, "test config", "muon", b.members, b.units, so=so, sw=sw, sg=sg)


def class_subset(cfg: Config, m: int, n: int) -> Config:
    """The members of cfg whose update units have shape class (min, max) =
    (m, n), as a config of their own with the same rank degrees (for timing
    one Newton-Schulz shape class alone)."""
    b = _ListBuilder()
    for mem in cfg.members:
        us = [u for u in cfg.units if u.member == cfg.members.index(mem)]
        if us and (min(us[0].rows, us[0].cols), max(us[0].rows, us[0].cols)) == (m, n):
            b.add(mem.name, mem.rows, mem.cols, unit_rows=None if len(us) == 1 else us[0].rows)
    return Config(f"{cfg.name}_class_{m}x{n}", f"the {m}x{n} units of {cfg.name}", "muon", b.members, b.units,
                  so=cfg.so, sw=cfg.sw, sg=cfg.sg)


CONFIGS = {
    "tiny": tiny,
    "flat_adamw": flat_adamw,
    "lm_layer": lm_layer,
    "moe_layer": moe_layer,
    # a quarter of the MoE layer (48 units, about 3 GB on the device): the
    # same Newton-Schulz shape class, small enough for a multi-pass profiler capture
    "moe_layer_16e": lambda: moe_layer(16),
    "video_dit": video_dit,
    "video_dit_layer": video_dit_layer,
}


def get(name: str) -> Config:
    return CONFIGS[name]()


def generate(cfg: Config, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Seeded logical-order inputs: main weight w ~ N(0, w_std) and main
    gradient g ~ N(0, g_std), both float32, drawn from one
    numpy.random.default_rng(seed) stream in the order w then g.
    Optimizer states start at zero (step 1)."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    n = cfg.numel
    w = rng.standard_normal(n, dtype=np.float32) * np.float32(cfg.w_std)
    g = rng.standard_normal(n, dtype=np.float32) * np.float32(cfg.g_std)
    return {"w": w, "g": g}


def gaussian(shape, std: float, seed: int) -> np.ndarray:
    """A seeded float32 N(0, std) array."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)


def generate_device(cfg: Config, device, seed: Optional[int] = None):
    """Seeded inputs drawn on the GPU for the full-size workloads (the host
    generator would take minutes at 2.3 G elements): w ~ N(0, w_std) then
    g ~ N(0, g_std), float32, from one torch.Generator on `device`.  Tests
    that compare with the oracle copy the drawn values back."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed if seed is None else seed)
    n = cfg.numel
    w = torch.empty(n, dtype=torch.float32, device=device)
    w.normal_(0.0, cfg.w_std, generator=gen)
    g = torch.empty(n, dtype=torch.float32, device=device)
    g.normal_(0.0, cfg.g_std, generator=gen)
    return {"w": w, "g": g}


def mixed() -> Config:
    """A small config that exercises every path: per-head units, transposed
    and non-transposed whole matrices, a Gram size that is not a multiple of
    128, one that is a multiple of 128 but not of 256 (single-CTA 128 x 256
    tiles instead of CTA pairs), a width that is not a multiple of 64, and
    ragged edges over 8 ranks."""
    b = _ListBuilder()
    _qkv(b, "", d=512, hq=4, hkv=4, dh=64)       # 12 x (64 x 512)
    b.add("up", 1536, 512)                       # transposed, 512 x 1536
    b.add("down", 512, 1536)                     # 512 x 1536
    for e in range(3):
        b.add(f"e{e}", 192, 320)                 # m = 192 -> padded to 256
    b.add("odd", 96, 160)                        # n = 160 -> padded to 192
    b.add("mid0", 384, 640)                      # Gram 384: single-CTA kernel
    b.add("mid1", 640, 384)                      # the same class, transposed
    return Config("mixed", "test mix of unit shapes over 8 ragged ranks", "muon", b.members, b.units,
                  so=8, sw=4, sg=4, edge_shift=ragged_shift(8, 400, seed=8))


def tiny_ragged() -> Config:
    cfg = tiny()
    cfg.name = "tiny_ragged"
    cfg.edge_shift = ragged_shift(4, 200, seed=4)
    return cfg


CONFIGS["mixed"] = mixed
CONFIGS["tiny_ragged"] = tiny_ragged
