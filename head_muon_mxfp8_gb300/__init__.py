"""GB300-native update phase of runtime/update-decoupled sharded data
parallelism (SS-HSDP): data-tree / shard-chain views, Muon (momentum +
batched Newton-Schulz on tcgen05 tensor cores), AdamW and MXFP8 requant,
as the C-ABI library libhm with a thin ctypes binding.

    from head_muon_mxfp8_gb300 import abi          # the C ABI, same names
    from head_muon_mxfp8_gb300.session import MuonSession, AdamWSession

The library is built in-tree by `__graft_entry__.build()` (or
`python head_muon_mxfp8_gb300/build.py`); using it before it is built raises.
"""
from . import _abi as abi  # noqa: F401

__all__ = ["abi"]
