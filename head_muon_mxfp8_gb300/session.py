"""Device state for the C ABI: PyTorch allocates the roots and the workspace
and supplies the stream; every computation runs in libhm's kernels.

A MuonSession owns one tensor list's emulated ZeRO-1 layout: the seven field
roots (w, m, g, u, v, q, s), each holding `so` rank segments with canary gaps,
a shard chain, a Muon plan and its uploaded workspace.  Moving logical-order
host data into the segments and back (`load` / `fetch`) is test and bench
set-up, done with plain tensor copies."""
from __future__ import annotations

from typing import Dict, Optional, Sequence, Tuple

import numpy as np
import torch

from . import _abi as abi

CANARY = {"w": 0x7FC0DEAD, "m": 0x7FC0BEEF, "g": 0x7FC0CAFE, "v": 0x7FC0F00D}  # fp32 NaN payloads
CANARY_U16 = 0xFFB7   # a bf16 NaN pattern


def _s32(x: int) -> int:
    return x - (1 << 32) if x >= 1 << 31 else x


def _s16(x: int) -> int:
    return x - (1 << 16) if x >= 1 << 15 else x
CANARY_U8 = 0xA5


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def aligned_empty(nbytes: int, device, align: int = 1024) -> Tuple[torch.Tensor, int]:
    """A uint8 device buffer and the first `align`-aligned address in it."""
    buf = torch.empty(nbytes + align, dtype=torch.uint8, device=device)
    addr = buf.data_ptr()
    return buf, (addr + align - 1) // align * align


class MuonSession:
    def __init__(self, numel: int, units: Sequence[Tuple[int, int, int]], so: int, sw: int, sg: int,
                 device="cuda", edges: Optional[Sequence[int]] = None,
                 edge_shift: Optional[Sequence[int]] = None, canaries: bool = True):
        self.device = torch.device(device)
        self.so, self.sw, self.sg, self.numel = so, sw, sg, numel
        self.units = [tuple(u) for u in units]
        self.chain = abi.shard_chain(numel, so, sw, sg, list(edges) if edges is not None else None,
                                     list(edge_shift) if edge_shift is not None else None)
        self.total, self.bases, self.lens, self.chunk_of = abi.shard_chain_layout(self.chain, so)
        # logical start of every rank's chunk
        rank_of_chunk = {c: r for r, c in enumerate(self.chunk_of)}
        self.edges = [0]
        for c in range(so):
            self.edges.append(self.edges[-1] + self.lens[rank_of_chunk[c]])
        self.plan = abi.muon_plan(self.chain, self.units)
        self.info = abi.muon_plan_query(self.plan)
        t, dev = self.total, self.device
        self.w = torch.empty(t, dtype=torch.float32, device=dev)
        self.m = torch.empty(t, dtype=torch.float32, device=dev)
        self.g = torch.empty(t, dtype=torch.float32, device=dev)
        self.v = torch.empty(t, dtype=torch.float32, device=dev)
        self.u = torch.empty(t, dtype=torch.int16, device=dev)
        self.q = torch.empty(t, dtype=torch.uint8, device=dev)
        self.s = torch.empty(t // 32, dtype=torch.uint8, device=dev)
        if canaries:
            for k in ("w", "m", "g", "v"):
                getattr(self, k).view(torch.int32).fill_(_s32(CANARY[k]))
            self.u.fill_(_s16(CANARY_U16))
            self.q.fill_(CANARY_U8)
            self.s.fill_(CANARY_U8)
        self.ws_bytes = int(self.info.workspace_bytes)
        self._ws_buf, self.ws = aligned_empty(self.ws_bytes, dev)
        abi.muon_plan_upload(self.plan, self.ws, self.ws_bytes, _stream_handle(None))
        self.bufs = abi.hm_muon_bufs(self.w.data_ptr(), self.m.data_ptr(), self.g.data_ptr(), self.u.data_ptr(),
                                     self.v.data_ptr(), self.q.data_ptr(), self.s.data_ptr())

    @classmethod
    def from_config(cls, cfg, device="cuda", **kw) -> "MuonSession":
        kw.setdefault("edge_shift", cfg.edge_shift)
        return cls(cfg.numel, [(u.offset, u.rows, u.cols) for u in cfg.units], cfg.so, cfg.sw, cfg.sg,
                   device=device, **kw)

    # ---- placement (set-up only) -------------------------------------------
    def _root(self, field: str) -> torch.Tensor:
        return getattr(self, field)

    def load(self, field: str, logical) -> None:
        """Copy a logical-order array (numpy or tensor) into the segments."""
        root = self._root(field)
        if isinstance(logical, np.ndarray) and logical.dtype == np.uint16:
            logical = logical.view(np.int16)
        src = torch.as_tensor(logical)
        if src.dtype != root.dtype:
            src = src.view(root.dtype) if src.element_size() == root.element_size() else src.to(root.dtype)
        src = src.to(self.device)
        div = 32 if field == "s" else 1
        for r in range(self.so):
            c = self.chunk_of[r]
            b, ln, e = self.bases[r] // div, self.lens[r] // div, self.edges[c] // div
            if ln:
                root[b:b + ln].copy_(src[e:e + ln])

    def fetch(self, field: str) -> torch.Tensor:
        """Logical-order copy of a field (on the host)."""
        root = self._root(field)
        div = 32 if field == "s" else 1
        out = torch.empty(self.numel // div, dtype=root.dtype, device=self.device)
        for r in range(self.so):
            c = self.chunk_of[r]
            b, ln, e = self.bases[r] // div, self.lens[r] // div, self.edges[c] // div
            if ln:
                out[e:e + ln].copy_(root[b:b + ln])
        return out.cpu()

    def fetch_range(self, field: str, a: int, b: int) -> torch.Tensor:
        """Logical elements [a, b) of a field (on the host); for the scale
        field a and b count scales."""
        root = self._root(field)
        div = 32 if field == "s" else 1
        out = torch.empty(b - a, dtype=root.dtype, device=self.device)
        for r in range(self.so):
            c = self.chunk_of[r]
            e0, e1 = self.edges[c] // div, self.edges[c + 1] // div
            lo, hi = max(a, e0), min(b, e1)
            if lo < hi:
                base = self.bases[r] // div
                out[lo - a:hi - a].copy_(root[base + lo - e0:base + hi - e0])
        return out.cpu()

    def unit_v(self, unit: int) -> torch.Tensor:
        """The direction v of one unit in logical order (root or staging)."""
        o, r, c = self.units[unit]
        if abi.muon_plan_unit(self.plan, unit)["local"]:
            return self.fetch_range("v", o, o + r * c)
        return self.staging(unit)[1].cpu()

    def canary_intact(self) -> Dict[str, bool]:
        ok = {}
        mask = torch.ones(self.total, dtype=torch.bool, device=self.device)
        for r in range(self.so):
            mask[self.bases[r]:self.bases[r] + self.lens[r]] = False
        for k in ("w", "m", "g", "v"):
            x = getattr(self, k).view(torch.int32)[mask]
            ok[k] = bool((x == _s32(CANARY[k])).all())
        uu = self.u[mask].to(torch.int32) & 0xFFFF
        ok["u"] = bool((uu == CANARY_U16).all())
        ok["q"] = bool((self.q[mask] == CANARY_U8).all())
        smask = mask.view(-1, 32).all(dim=1)
        ok["s"] = bool((self.s[smask] == CANARY_U8).all())
        return ok

    # ---- the update --------------------------------------------------------
    def run(self, hp: "abi.hm_muon_hparams", stages: int = abi.HM_STAGE_ALL,
            stream: Optional[torch.cuda.Stream] = None) -> None:
        abi.muon_update_units(self.plan, self.bufs, hp, self.ws, self.ws_bytes, stages, _stream_handle(stream))

    def staging(self, unit: int):
        """Device views of a straddling unit's u / v staging."""
        u_addr, v_addr = abi.muon_plan_staging(self.plan, unit)
        o, r, c = self.units[unit]
        n = r * c
        base_u = u_addr - self._ws_buf.data_ptr()
        u = self._ws_buf[base_u:base_u + 2 * n].view(torch.int16)
        base_v = v_addr - self._ws_buf.data_ptr()
        v = self._ws_buf[base_v:base_v + 4 * n].view(torch.float32)
        return u, v

    def close(self) -> None:
        if self.plan:
            abi.muon_plan_destroy(self.plan)
            self.plan = 0
        if self.chain:
            abi.chain_destroy(self.chain)
            self.chain = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def muon_hparams(h) -> "abi.hm_muon_hparams":
    """From a workloads.MuonHparams-like object."""
    return abi.hm_muon_hparams(h.lr, h.momentum, h.weight_decay, h.eps, h.ns_a, h.ns_b, h.ns_c, h.ns_steps,
                               int(h.nesterov), h.alpha_mode)


def adamw_hparams(h, step: int) -> "abi.hm_adamw_hparams":
    return abi.hm_adamw_hparams(h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, step)
