"""Data tree, shard chain, fragments and the emulated rank-segment layout.

Follows "SS-HSDP" section 3.2:
  * Data Tree: a child is a view at a byte offset inside its parent; the
    child's shape and dtype fix its size; only the root owns storage and a
    node reaches it through its accumulated offset.
  * Shard Chain: the flat tensor list is cut into contiguous chunks,
    W -> W^z3 -> W^z2 -> W^z1; a member's local fragment at a level is the
    intersection of its range with the local chunk, or empty.
  * Distributed updates: the fragments of a unit are located at the ZeRO-1
    level; a unit with one fragment is local, otherwise an execution rank
    gathers the fragments, computes, and returns the modified fragments.
and section 4.2 (Fully Zero Copy, Figure 4): ZeRO-1 chunks are stored in
group-rank order, owners [0, 2, 1, 3] for so = 4, sw = sg = 2.

Readings where the paper is silent (listed in the design notes):
  * edges: E_c = 32 * floor(c * N / (32 * so)), c = 0..so (32-aligned, nearly
    even, not unit-aligned); N must be a multiple of 32; a workload may move
    the interior edges by a given 32-aligned shift (ragged edges);
  * owner of z1 chunk c = i*R + j (R = so/sw) is rank i + j*sw;
  * a level of degree s has chunk k = z1 chunks [k*so/s, (k+1)*so/s);
  * execution rank of a unit = owner of the chunk holding its first element
    (Head0 spans ranks 2 and 1 and rank 2 executes, section 3.4);
  * emulation: rank r's z1 chunk is stored as segment r of one allocation, in
    rank order, each segment starting on a multiple of ALIGN elements with a
    GAP-element canary region before the first segment, between segments and
    after the last.

Pins (tests/test_oracle_views.py): Figure 4 owners and the Head0 example
(tests/golden/fig4_shard_chain.txt), fragments against a brute-force
per-element owner map, gather/scatter inverse in both directions, data-tree
aliasing through the root, nesting of the three levels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence, Tuple

import numpy as np

ALIGN = 1024   # elements: segment base alignment (4 KiB for fp32)
GAP = 1024     # elements: canary region around every segment


# ----------------------------------------------------------------------------
# Data tree
# ----------------------------------------------------------------------------
class DataTree:
    """Root owns a byte buffer; every other node is (parent, byte offset,
    dtype, shape).  A node's data is the root storage at its accumulated
    offset."""

    def __init__(self, root_bytes: int):
        self.storage = np.zeros(root_bytes, dtype=np.uint8)
        self.nodes: List[Tuple[int, int, np.dtype, Tuple[int, ...]]] = [
            (-1, 0, np.dtype(np.uint8), (root_bytes,))]

    def nbytes(self, node: int) -> int:
        _, _, dt, shape = self.nodes[node]
        return int(np.prod(shape, dtype=np.int64)) * dt.itemsize

    def add_view(self, parent: int, byte_off: int, dtype, shape) -> int:
        dt = np.dtype(dtype)
        shape = tuple(int(s) for s in shape)
        size = int(np.prod(shape, dtype=np.int64)) * dt.itemsize
        if parent < 0 or parent >= len(self.nodes):
            raise ValueError("no such parent")
        if byte_off < 0 or byte_off + size > self.nbytes(parent):
            raise ValueError("view exceeds its parent")
        if (self.resolve(parent) + byte_off) % dt.itemsize:
            raise ValueError("view misaligned for its dtype")
        self.nodes.append((parent, byte_off, dt, shape))
        return len(self.nodes) - 1

    def resolve(self, node: int) -> int:
        """Accumulated byte offset of a node from the root."""
        off = 0
        while node > 0:
            parent, byte_off, _, _ = self.nodes[node]
            off += byte_off
            node = parent
        return off

    def view(self, node: int) -> np.ndarray:
        _, _, dt, shape = self.nodes[node]
        return np.ndarray(shape, dtype=dt, buffer=self.storage, offset=self.resolve(node))


# ----------------------------------------------------------------------------
# Shard chain
# ----------------------------------------------------------------------------
def z1_edges(n: int, so: int, shift: Sequence[int] = None) -> List[int]:
    """Default ZeRO-1 edges, optionally moved by a ragged 32-aligned shift
    (shift[0] = shift[so] = 0)."""
    if n % 32:
        raise ValueError("tensor-list length must be a multiple of 32")
    e = [32 * ((c * n) // (32 * so)) for c in range(so + 1)]
    if shift is not None:
        if shift[0] or shift[so] or any(x % 32 for x in shift):
            raise ValueError("edge shift must be 32-aligned and keep 0 and n")
        e = [a + b for a, b in zip(e, shift)]
        if any(b < a for a, b in zip(e[:-1], e[1:])):
            raise ValueError("shifted edges decrease")
    return e


def owner(c: int, so: int, sw: int) -> int:
    r = so // sw
    return (c // r) + (c % r) * sw


def chunk_of_rank(rank: int, so: int, sw: int) -> int:
    for c in range(so):
        if owner(c, so, sw) == rank:
            return c
    raise ValueError("rank out of range")


def check_degrees(so: int, sw: int, sg: int) -> None:
    if so < 1 or sw < 1 or sg < 1 or sg % sw or so % sg:
        raise ValueError("sharding degrees must nest: sw | sg | so")


def level_range(edges: Sequence[int], so: int, s: int, k: int) -> Tuple[int, int]:
    """Element range of chunk k at a level of degree s."""
    per = so // s
    return edges[k * per], edges[(k + 1) * per]


def rank_level_chunk(rank: int, so: int, sw: int, s: int) -> int:
    """Index of the level-s chunk that holds rank's z1 chunk."""
    return chunk_of_rank(rank, so, sw) // (so // s)


@dataclass(frozen=True)
class Fragment:
    chunk: int        # z1 chunk index
    rank: int         # owning rank (= segment index)
    seg_offset: int   # element offset inside the owner's segment
    unit_offset: int  # element offset inside the unit
    length: int
    root_offset: int  # element offset inside the emulated root allocation


def segment_layout(edges: Sequence[int], so: int, sw: int) -> Tuple[List[int], int]:
    """Base element offset of every rank's segment and the total length of the
    emulated root allocation (segments in rank order, ALIGN-aligned, GAP
    canary elements before, between and after them)."""
    bases = []
    pos = GAP
    for r in range(so):
        c = chunk_of_rank(r, so, sw)
        ln = edges[c + 1] - edges[c]
        bases.append(pos)
        pos += -(-ln // ALIGN) * ALIGN + GAP
    return bases, pos


def fragments(a: int, b: int, edges: Sequence[int], so: int, sw: int,
              bases: Sequence[int]) -> List[Fragment]:
    """z1 fragments of the logical range [a, b), in unit order."""
    out = []
    for c in range(so):
        lo, hi = max(a, edges[c]), min(b, edges[c + 1])
        if lo < hi:
            r = owner(c, so, sw)
            out.append(Fragment(c, r, lo - edges[c], lo - a, hi - lo,
                                bases[r] + lo - edges[c]))
    return out


def execution_rank(frags: Sequence[Fragment]) -> int:
    return frags[0].rank


def gather(root: np.ndarray, frags: Sequence[Fragment], numel: int) -> np.ndarray:
    out = np.empty(numel, dtype=root.dtype)
    for f in frags:
        out[f.unit_offset:f.unit_offset + f.length] = root[f.root_offset:f.root_offset + f.length]
    return out


def scatter(root: np.ndarray, frags: Sequence[Fragment], unit: np.ndarray) -> None:
    for f in frags:
        root[f.root_offset:f.root_offset + f.length] = unit[f.unit_offset:f.unit_offset + f.length]


def to_segments(logical: np.ndarray, edges, so, sw, fill=0) -> np.ndarray:
    """Place a logical-order field into the emulated root allocation."""
    bases, total = segment_layout(edges, so, sw)
    root = np.full(total, fill, dtype=logical.dtype)
    for r in range(so):
        c = chunk_of_rank(r, so, sw)
        root[bases[r]:bases[r] + edges[c + 1] - edges[c]] = logical[edges[c]:edges[c + 1]]
    return root


def from_segments(root: np.ndarray, edges, so, sw) -> np.ndarray:
    bases, _ = segment_layout(edges, so, sw)
    out = np.empty(edges[-1], dtype=root.dtype)
    for r in range(so):
        c = chunk_of_rank(r, so, sw)
        out[edges[c]:edges[c + 1]] = root[bases[r]:bases[r] + edges[c + 1] - edges[c]]
    return out


def canary_mask(edges, so, sw) -> np.ndarray:
    """True for every root element that lies outside all segments."""
    bases, total = segment_layout(edges, so, sw)
    mask = np.ones(total, dtype=bool)
    for r in range(so):
        c = chunk_of_rank(r, so, sw)
        mask[bases[r]:bases[r] + edges[c + 1] - edges[c]] = False
    return mask
