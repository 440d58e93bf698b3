"""ctypes binding of libhm (include/hm.h): the same names, argument
marshalling only.  Every step of the update path runs in the library's CUDA
kernels; there is no Python or CPU fallback.  Loading fails loudly when the
library has not been built."""
from __future__ import annotations

import ctypes as C
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhm.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "hm.h")

HM_OK = 0
HM_ERR_ARG = -1
HM_ERR_GEOMETRY = -2
HM_ERR_OVERLAP = -3
HM_ERR_ALIGN = -4
HM_ERR_DTYPE = -5
HM_ERR_UNITS = -6
HM_ERR_CUDA = -7
HM_ERR_ARCH = -8
HM_ERR_TIMEOUT = -9
HM_ERR_WORKSPACE = -10
HM_ERR_STATE = -11

HM_U8, HM_BF16, HM_F32, HM_E4M3 = 0, 1, 2, 3
HM_SEG_ALIGN = 1024
HM_SEG_GAP = 1024
HM_MX_BLOCK = 32
HM_NOALLOC_MAX_MIN_DIM = 128
HM_NOALLOC_MAX_MAX_DIM = 8192
HM_NOALLOC_SCRATCH_BYTES = 4262912

HM_STAGE_F0 = 1
HM_STAGE_GATHER = 2
HM_STAGE_NS = 4
HM_STAGE_F2 = 8
HM_STAGE_REQUANT = 16
HM_STAGE_ALL = 31
HM_STAGE_FUSED = 32
HM_STAGE_ALL_FUSED = 63
HM_STAGE_SCRATCH = 64
HM_STAGE_STEP = 127
HM_RS_FP32, HM_RS_BF16, HM_RS_BF16_SR = 0, 1, 2


class hm_fragment(C.Structure):
    _fields_ = [("chunk", C.c_int32), ("rank", C.c_int32), ("seg_offset", C.c_int64),
                ("unit_offset", C.c_int64), ("length", C.c_int64), ("root_offset", C.c_int64)]


class hm_unit_desc(C.Structure):
    _fields_ = [("offset", C.c_int64), ("rows", C.c_int32), ("cols", C.c_int32)]


class hm_muon_plan_info(C.Structure):
    _fields_ = [("n_units", C.c_int32), ("n_local", C.c_int32), ("n_straddling", C.c_int32),
                ("n_classes", C.c_int32), ("staging_elems", C.c_int64), ("workspace_bytes", C.c_int64),
                ("n_fragments", C.c_int32)]


class hm_muon_hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("momentum", C.c_float), ("weight_decay", C.c_float), ("eps", C.c_float),
                ("ns_a", C.c_float), ("ns_b", C.c_float), ("ns_c", C.c_float), ("ns_steps", C.c_int32),
                ("nesterov", C.c_int32), ("alpha_mode", C.c_int32)]


class hm_muon_bufs(C.Structure):
    _fields_ = [("w", C.c_void_p), ("m", C.c_void_p), ("g", C.c_void_p), ("u", C.c_void_p),
                ("v", C.c_void_p), ("q", C.c_void_p), ("s", C.c_void_p)]


class hm_adamw_hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float), ("step", C.c_int32)]


class hm_mx_tensor(C.Structure):
    _fields_ = [("src_offset", C.c_int64), ("dst_offset", C.c_int64), ("scale_offset", C.c_int64),
                ("rows", C.c_int64), ("k", C.c_int64)]


class hm_scale_relayout(C.Structure):
    _fields_ = [("src_offset", C.c_int64), ("dst_offset", C.c_int64), ("rows", C.c_int64), ("kb", C.c_int64),
                ("block_rows", C.c_int32), ("pad", C.c_int32)]


class HmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({status_str(status)})")
        self.status = status


_P = C.c_void_p
_I64P = C.POINTER(C.c_int64)
_I32P = C.POINTER(C.c_int32)
_SIGS = {
    "hm_status_str": (C.c_char_p, [C.c_int]),
    "hm_device_error": (C.c_int, [_I32P]),
    "hm_kernel_launches": (C.c_int, [C.POINTER(C.c_int64)]),
    "create_data_tree": (C.c_int, [C.POINTER(_P), _P, C.c_size_t]),
    "data_tree_add_view": (C.c_int, [_P, C.c_int, C.c_size_t, C.c_int, C.c_int, _I64P, _I32P]),
    "data_tree_resolve": (C.c_int, [_P, C.c_int, C.POINTER(_P), C.POINTER(C.c_size_t)]),
    "data_tree_check_disjoint": (C.c_int, [_P, _I32P, C.c_int]),
    "tree_destroy": (None, [_P]),
    "shard_chain": (C.c_int, [C.POINTER(_P), C.c_int64, C.c_int, C.c_int, C.c_int, _I64P, _I64P]),
    "shard_chain_layout": (C.c_int, [_P, _I64P, _I64P, _I64P, _I32P]),
    "shard_chain_fragments": (C.c_int, [_P, C.c_int64, C.c_int64, C.c_int, C.POINTER(hm_fragment), C.c_int,
                                        _I32P]),
    "shard_chain_segment_views": (C.c_int, [_P, _P, C.c_int, _I32P]),
    "chain_destroy": (None, [_P]),
    "muon_plan": (C.c_int, [C.POINTER(_P), _P, C.POINTER(hm_unit_desc), C.c_int]),
    "muon_plan_query": (C.c_int, [_P, C.POINTER(hm_muon_plan_info)]),
    "muon_plan_unit": (C.c_int, [_P, C.c_int, _I32P, _I32P, _I32P, _I32P]),
    "muon_plan_upload": (C.c_int, [_P, _P, C.c_size_t, _P]),
    "muon_update_units": (C.c_int, [_P, C.POINTER(hm_muon_bufs), C.POINTER(hm_muon_hparams), _P, C.c_size_t,
                                    C.c_int, _P]),
    "muon_plan_staging": (C.c_int, [_P, C.c_int, C.POINTER(_P), C.POINTER(_P)]),
    "muon_plan_destroy": (None, [_P]),
    "adamw_update_flat": (C.c_int, [_P, _P, C.c_int, _P, _P, C.c_int64, C.POINTER(hm_adamw_hparams), _P]),
    "mxfp8_requant_packed": (C.c_int, [_P, _P, _P, C.POINTER(hm_mx_tensor), C.c_int, _P]),
    "mxfp8_requant_32x32": (C.c_int, [_P, _P, _P, _P, C.POINTER(hm_mx_tensor), C.c_int, _P]),
    "mxfp8_scale_relayout": (C.c_int, [_P, _P, C.POINTER(hm_scale_relayout), C.c_int, _P]),
    "reduce_scatter_grad": (C.c_int, [_P, _P, C.c_int, C.c_int, _P, C.c_int, C.c_int, C.c_uint64, C.c_uint64,
                                      _P]),
    "newton_schulz_noalloc": (C.c_int, [_P, C.c_int32, C.c_int32, _P, C.POINTER(hm_muon_hparams), _P]),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libhm.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


def header_symbols() -> list:
    """Every function the C header declares (used by the export test)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                                 text, flags=re.M)))


def status_str(s: int) -> str:
    return lib().hm_status_str(s).decode()


def check(fn: str, status: int) -> None:
    if status != HM_OK:
        raise HmError(fn, status)


def _i64(vals):
    return (C.c_int64 * len(vals))(*vals) if vals is not None else None


# ---- thin wrappers: same names as the C ABI --------------------------------
def hm_kernel_launches() -> int:
    """Kernels this thread has launched through the library so far."""
    n = C.c_int64(0)
    check("hm_kernel_launches", lib().hm_kernel_launches(C.byref(n)))
    return n.value


def hm_device_error() -> int:
    code = C.c_int32(0)
    check("hm_device_error", lib().hm_device_error(C.byref(code)))
    return code.value


def create_data_tree(root: int, root_bytes: int) -> int:
    h = _P()
    check("create_data_tree", lib().create_data_tree(C.byref(h), _P(root), root_bytes))
    return h.value


def data_tree_add_view(tree: int, parent: int, byte_off: int, dtype: int, shape) -> int:
    node = C.c_int32(0)
    check("data_tree_add_view", lib().data_tree_add_view(_P(tree), parent, byte_off, dtype, len(shape),
                                                         _i64(list(shape)), C.byref(node)))
    return node.value


def data_tree_resolve(tree: int, node: int):
    ptr, off = _P(), C.c_size_t(0)
    check("data_tree_resolve", lib().data_tree_resolve(_P(tree), node, C.byref(ptr), C.byref(off)))
    return ptr.value or 0, off.value


def data_tree_check_disjoint(tree: int, nodes) -> int:
    arr = (C.c_int32 * len(nodes))(*nodes)
    return lib().data_tree_check_disjoint(_P(tree), arr, len(nodes))


def tree_destroy(tree: int) -> None:
    lib().tree_destroy(_P(tree))


def shard_chain(n: int, so: int, sw: int, sg: int, z1_edges=None, edge_shift=None) -> int:
    h = _P()
    check("shard_chain", lib().shard_chain(C.byref(h), n, so, sw, sg, _i64(z1_edges), _i64(edge_shift)))
    return h.value


def shard_chain_layout(chain: int, so: int):
    total = C.c_int64(0)
    bases, lens = (C.c_int64 * so)(), (C.c_int64 * so)()
    chunks = (C.c_int32 * so)()
    check("shard_chain_layout", lib().shard_chain_layout(_P(chain), C.byref(total), bases, lens, chunks))
    return total.value, list(bases), list(lens), list(chunks)


def shard_chain_fragments(chain: int, a: int, b: int, level: int = 1):
    n = C.c_int32(0)
    check("shard_chain_fragments", lib().shard_chain_fragments(_P(chain), a, b, level, None, 0, C.byref(n)))
    out = (hm_fragment * max(1, n.value))()
    check("shard_chain_fragments", lib().shard_chain_fragments(_P(chain), a, b, level, out, n.value, C.byref(n)))
    return [out[i] for i in range(n.value)]


def shard_chain_segment_views(chain: int, tree: int, dtype: int, so: int):
    nodes = (C.c_int32 * so)()
    check("shard_chain_segment_views", lib().shard_chain_segment_views(_P(chain), _P(tree), dtype, nodes))
    return list(nodes)


def chain_destroy(chain: int) -> None:
    lib().chain_destroy(_P(chain))


def muon_plan(chain: int, units) -> int:
    arr = (hm_unit_desc * max(1, len(units)))(*[hm_unit_desc(o, r, c) for (o, r, c) in units])
    h = _P()
    check("muon_plan", lib().muon_plan(C.byref(h), _P(chain), arr, len(units)))
    return h.value


def muon_plan_query(plan: int) -> hm_muon_plan_info:
    info = hm_muon_plan_info()
    check("muon_plan_query", lib().muon_plan_query(_P(plan), C.byref(info)))
    return info


def muon_plan_unit(plan: int, unit: int):
    e, n, c, l = C.c_int32(), C.c_int32(), C.c_int32(), C.c_int32()
    check("muon_plan_unit", lib().muon_plan_unit(_P(plan), unit, C.byref(e), C.byref(n), C.byref(c), C.byref(l)))
    return {"exec_rank": e.value, "n_frags": n.value, "cls": c.value, "local": bool(l.value)}


def muon_plan_upload(plan: int, workspace: int, workspace_bytes: int, stream: int = 0) -> None:
    check("muon_plan_upload", lib().muon_plan_upload(_P(plan), _P(workspace), workspace_bytes, _P(stream)))


def muon_update_units(plan: int, bufs: hm_muon_bufs, hp: hm_muon_hparams, workspace: int, workspace_bytes: int,
                      stages: int = HM_STAGE_ALL, stream: int = 0) -> None:
    check("muon_update_units", lib().muon_update_units(_P(plan), C.byref(bufs), C.byref(hp), _P(workspace),
                                                       workspace_bytes, stages, _P(stream)))


def muon_plan_staging(plan: int, unit: int):
    u, v = _P(), _P()
    check("muon_plan_staging", lib().muon_plan_staging(_P(plan), unit, C.byref(u), C.byref(v)))
    return u.value, v.value


def muon_plan_destroy(plan: int) -> None:
    lib().muon_plan_destroy(_P(plan))


def adamw_update_flat(w: int, g: int, g_dtype: int, m: int, v: int, n: int, hp: hm_adamw_hparams,
                      stream: int = 0) -> None:
    check("adamw_update_flat", lib().adamw_update_flat(_P(w), _P(g), g_dtype, _P(m), _P(v), n, C.byref(hp),
                                                       _P(stream)))


def mxfp8_requant_packed(w: int, q: int, scales: int, tensors, stream: int = 0) -> None:
    arr = (hm_mx_tensor * max(1, len(tensors)))(*[hm_mx_tensor(*t) for t in tensors])
    check("mxfp8_requant_packed", lib().mxfp8_requant_packed(_P(w), _P(q), _P(scales), arr, len(tensors),
                                                             _P(stream)))


def mxfp8_requant_32x32(chain: int, w: int, q: int, scales: int, tensors, stream: int = 0) -> None:
    arr = (hm_mx_tensor * max(1, len(tensors)))(*[hm_mx_tensor(*t) for t in tensors])
    check("mxfp8_requant_32x32", lib().mxfp8_requant_32x32(_P(chain), _P(w), _P(q), _P(scales), arr, len(tensors),
                                                           _P(stream)))


def mxfp8_scale_relayout(src: int, dst: int, items, stream: int = 0) -> None:
    """items: (src_offset, dst_offset, rows, kb, block_rows)."""
    arr = (hm_scale_relayout * max(1, len(items)))(*[hm_scale_relayout(*it, 0) for it in items])
    check("mxfp8_scale_relayout", lib().mxfp8_scale_relayout(_P(src), _P(dst), arr, len(items), _P(stream)))


def reduce_scatter_grad(chain: int, parts: int, n_parts: int, ranks_per_node: int, g: int, mode: int,
                        accumulate: bool, seed: int, offset: int, stream: int = 0) -> None:
    check("reduce_scatter_grad", lib().reduce_scatter_grad(_P(chain), _P(parts), n_parts, ranks_per_node, _P(g), mode,
                                                           int(accumulate), seed, offset, _P(stream)))


def newton_schulz_noalloc(u: int, rows: int, cols: int, v: int, hp: hm_muon_hparams, stream: int = 0) -> None:
    """One unit's Newton-Schulz on the library's built-in scratch: for callers
    that cannot allocate device memory (see include/hm.h)."""
    check("newton_schulz_noalloc", lib().newton_schulz_noalloc(_P(u), rows, cols, _P(v), C.byref(hp), _P(stream)))
