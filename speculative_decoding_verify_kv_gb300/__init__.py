"""Python binding of libverify_attn.so (GB300 speculative-decoding verify
attention).

Argument marshalling only: tensors' device pointers and sizes go into the
C structs of ``include/verify_attn.h`` and every step of the computation
runs in the library's CUDA kernels.  PyTorch supplies device memory and
streams.  There is no fallback: if the library is missing or cannot load,
importing this package raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

from . import _build

F32, BF16, Q8_0 = 0, 1, 2
MODE_CHAIN, MODE_TREE, MODE_MIXED = 0, 1, 2
FLAG_CUDA_CORES = 0x1
# Partial kernels (va_plan_info.kernel).
KERNEL_CUDA_CORES, KERNEL_TENSOR, KERNEL_TENSOR_Q8 = 0, 1, 2

DEV_BAD_PARENT = 0x1
DEV_BAD_BLOCK = 0x2
DEV_CTX_OVERFLOW = 0x4
DEV_BAD_ROWS = 0x8
DEV_TIMEOUT = 0x10

# Rows per sequence (chain / tree); see VA_MAX_ROWS_PER_SEQ in the header.
MAX_ROWS_PER_SEQ = 1024
MAX_TREE_ROWS = 32

STATUS_NAMES = {0: "VA_OK", 1: "VA_ERR_INVALID_ARG", 2: "VA_ERR_UNSUPPORTED",
                3: "VA_ERR_ALIGNMENT", 4: "VA_ERR_WORKSPACE_TOO_SMALL", 5: "VA_ERR_CUDA"}

DTYPE_CODES = {"f32": F32, "bf16": BF16, "q8_0": Q8_0}
MODE_CODES = {"chain": MODE_CHAIN, "tree": MODE_TREE, "mixed": MODE_MIXED}

EXPORTED = ["va_version", "va_status_string", "va_last_cuda_error", "va_workspace_size", "va_validate",
            "verify_attn_chain", "verify_attn_tree", "verify_attn_mixed",
            "va_debug_row_map", "va_debug_gather_index", "va_plan", "va_timing_enable",
            "va_timing_read", "verify_attn_noalloc", "verify_attn_promote", "va_debug_split_ranges"]


class VaKV(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("page_size", ctypes.c_int32), ("capacity", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("draft_k", ctypes.c_void_p),
                ("draft_v", ctypes.c_void_p)]


class VaProblem(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("q_dtype", ctypes.c_int), ("q", ctypes.c_void_p),
                ("cu_rows", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p),
                ("parent", ctypes.c_void_p), ("seq_kind", ctypes.c_void_p),
                ("total_rows", ctypes.c_int32), ("max_rows_per_seq", ctypes.c_int32),
                ("scale", ctypes.c_float), ("num_splits", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class VaPlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("sub_splits", ctypes.c_int32),
                ("slots", ctypes.c_int32), ("grid_x", ctypes.c_int32),
                ("grid_y", ctypes.c_int32), ("grid_z", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32)]


def _load():
    path = _build.lib_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.va_version.restype = ctypes.c_int32
    lib.va_status_string.restype = ctypes.c_char_p
    lib.va_status_string.argtypes = [ctypes.c_int]
    lib.va_last_cuda_error.restype = ctypes.c_char_p
    lib.va_workspace_size.restype = ctypes.c_size_t
    lib.va_workspace_size.argtypes = [P(VaProblem), P(VaKV)]
    lib.va_validate.restype = ctypes.c_int
    lib.va_validate.argtypes = [P(VaProblem), P(VaKV), ctypes.c_int32, ctypes.c_size_t]
    for name in ("verify_attn_chain", "verify_attn_tree", "verify_attn_mixed"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [P(VaProblem), P(VaKV), ctypes.c_void_p, ctypes.c_size_t,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.va_debug_row_map.restype = ctypes.c_int
    lib.va_debug_row_map.argtypes = [P(VaProblem), ctypes.c_int32, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.va_debug_gather_index.restype = ctypes.c_int
    lib.va_debug_gather_index.argtypes = [P(VaProblem), P(VaKV), ctypes.c_int32,
                                          ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p]
    lib.va_plan.restype = ctypes.c_int
    lib.va_plan.argtypes = [P(VaProblem), P(VaKV), ctypes.c_int32, P(VaPlanInfo)]
    lib.va_debug_split_ranges.restype = ctypes.c_int
    lib.va_debug_split_ranges.argtypes = [P(VaProblem), P(VaKV), ctypes.c_int32, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]
    lib.va_timing_enable.restype = ctypes.c_int
    lib.va_timing_enable.argtypes = [ctypes.c_int32]
    lib.verify_attn_noalloc.restype = ctypes.c_int
    lib.verify_attn_noalloc.argtypes = [P(VaProblem), P(VaKV), ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.va_timing_read.restype = ctypes.c_int
    lib.va_timing_read.argtypes = [ctypes.c_int32, P(ctypes.c_float), P(ctypes.c_float),
                                   P(ctypes.c_int32)]
    lib.verify_attn_promote.restype = ctypes.c_int
    lib.verify_attn_promote.argtypes = [P(VaProblem), P(VaKV), ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return lib


lib = _load()
LIB_PATH = _build.lib_path()


class VaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        extra = f": {lib.va_last_cuda_error().decode()}" if code == 5 else ""
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} "
                         f"({lib.va_status_string(code).decode()}{extra})")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return int(t.data_ptr())


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) or None


@dataclass
class KV:
    """Device KV cache (contiguous or paged).  ``k``/``v`` are uint8, uint16
    or float32 tensors holding the storage rows."""
    dtype: int
    num_kv_heads: int
    head_dim: int
    k: object
    v: object
    page_size: int = 0
    capacity: int = 0
    block_table: object = None
    max_blocks_per_seq: int = 0
    num_blocks: int = 0
    draft_k: object = None  # optional tree scratch KV [total_rows][KVH][row]
    draft_v: object = None

    def c(self) -> VaKV:
        return VaKV(self.dtype, self.num_kv_heads, self.head_dim, _ptr(self.k), _ptr(self.v),
                    self.page_size, self.capacity, _ptr(self.block_table),
                    self.max_blocks_per_seq, self.num_blocks, _ptr(self.draft_k),
                    _ptr(self.draft_v))


@dataclass
class Problem:
    """Device query side of a verify call."""
    num_seqs: int
    num_heads: int
    q_dtype: int
    q: object
    cu_rows: object
    ctx_len: object
    parent: object
    seq_kind: object
    total_rows: int
    max_rows_per_seq: int
    scale: float = 0.0
    num_splits: int = 1
    flags: int = 0

    def c(self) -> VaProblem:
        return VaProblem(self.num_seqs, self.num_heads, self.q_dtype, _ptr(self.q),
                         _ptr(self.cu_rows), _ptr(self.ctx_len), _ptr(self.parent),
                         _ptr(self.seq_kind), self.total_rows, self.max_rows_per_seq,
                         float(self.scale), self.num_splits, self.flags)


def workspace_size(p: Problem, kv: KV) -> int:
    return int(lib.va_workspace_size(ctypes.byref(p.c()), ctypes.byref(kv.c())))


def validate(p: Problem, kv: KV, mode: int, ws_bytes: int) -> int:
    return int(lib.va_validate(ctypes.byref(p.c()), ctypes.byref(kv.c()), mode, ws_bytes))


def plan(p: Problem, kv: KV, mode: int = MODE_CHAIN) -> dict:
    info = VaPlanInfo()
    st = lib.va_plan(ctypes.byref(p.c()), ctypes.byref(kv.c()), mode, ctypes.byref(info))
    if st:
        raise VaError(st, "va_plan")
    return {f: getattr(info, f) for f, _ in VaPlanInfo._fields_}


def alloc_workspace(p: Problem, kv: KV, device=None):
    import torch
    n = workspace_size(p, kv)
    dev = device if device is not None else p.q.device
    # 256-byte alignment holds for torch's caching allocator (512-byte blocks).
    return torch.empty(max(n, 256), dtype=torch.uint8, device=dev)


def _call(fname: str, p: Problem, kv: KV, ws=None, o=None, lse=None, status=None,
          stream=None, check: bool = True):
    import torch
    dev = p.q.device
    D = kv.head_dim
    if o is None:
        o = torch.empty((p.total_rows, p.num_heads, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((p.total_rows, p.num_heads), dtype=torch.float32, device=dev)
    if ws is None:
        ws = alloc_workspace(p, kv, dev)
    pc, kc = p.c(), kv.c()
    st = getattr(lib, fname)(ctypes.byref(pc), ctypes.byref(kc), _ptr(ws),
                             ws.numel() * ws.element_size(), _ptr(o), _ptr(lse), _ptr(status),
                             _stream_handle(stream))
    if st and check:
        raise VaError(st, fname)
    return o, lse


def verify_attn_chain(p: Problem, kv: KV, **kw):
    return _call("verify_attn_chain", p, kv, **kw)


def verify_attn_tree(p: Problem, kv: KV, **kw):
    return _call("verify_attn_tree", p, kv, **kw)


def verify_attn_mixed(p: Problem, kv: KV, **kw):
    return _call("verify_attn_mixed", p, kv, **kw)


def verify_attn(p: Problem, kv: KV, mode: int, **kw):
    return _call(("verify_attn_chain", "verify_attn_tree", "verify_attn_mixed")[mode], p, kv, **kw)


# Bytes of library-held scratch behind verify_attn_noalloc (one array per
# device, part of the library's device image).
STATIC_WORKSPACE_BYTES = 16 * 1024 * 1024


def verify_attn_noalloc(p: Problem, kv: KV, mode: int, o, lse, status=None, stream=None):
    """Verify call that uses the library's own scratch: no workspace
    argument and no allocation on the call path (``o`` and ``lse`` are the
    caller's preallocated outputs).  Raises VaError(VA_ERR_WORKSPACE_TOO_SMALL)
    for problems that need more than STATIC_WORKSPACE_BYTES of partials.
    Calls that may overlap in time on one device share the scratch and must
    not be issued; make the first call per device outside stream capture."""
    st = lib.verify_attn_noalloc(ctypes.byref(p.c()), ctypes.byref(kv.c()), mode, _ptr(o),
                                 _ptr(lse), _ptr(status), _stream_handle(stream))
    if st:
        raise VaError(st, "verify_attn_noalloc")
    return o, lse


def verify_attn_promote(p: Problem, kv: KV, mode: int, accepted_len, accepted_nodes, status,
                        stream=None):
    """Copy each tree sequence's accepted path from the tree scratch KV
    (``kv.draft_k/draft_v``) into the cache at positions ctx..ctx+m-1, as
    one device-checked transaction (nothing is written if the preflight
    flags any sequence).  ``accepted_len`` int32 [num_seqs] and
    ``accepted_nodes`` int32 [total_rows] are device tensors; ``status`` is a
    zeroed device int32 word that receives the VA_DEV_* bits."""
    st = lib.verify_attn_promote(ctypes.byref(p.c()), ctypes.byref(kv.c()), mode,
                                 _ptr(accepted_len), _ptr(accepted_nodes), _ptr(status),
                                 _stream_handle(stream))
    if st:
        raise VaError(st, "verify_attn_promote")


def debug_row_map(p: Problem, mode: int, status=None, stream=None):
    import torch
    dev = p.cu_rows.device
    row_seq = torch.full((max(p.total_rows, 1),), -1, dtype=torch.int32, device=dev)
    anc = torch.zeros((max(p.total_rows, 1),), dtype=torch.int32, device=dev)
    st = lib.va_debug_row_map(ctypes.byref(p.c()), mode, _ptr(row_seq), _ptr(anc),
                              _ptr(status), _stream_handle(stream))
    if st:
        raise VaError(st, "va_debug_row_map")
    return row_seq[:p.total_rows], anc[:p.total_rows]


def debug_gather_index(p: Problem, kv: KV, kv_head: int, max_len: int, status=None,
                       stream=None):
    import torch
    out = torch.empty((p.num_seqs, max_len), dtype=torch.int64, device=p.cu_rows.device)
    st = lib.va_debug_gather_index(ctypes.byref(p.c()), ctypes.byref(kv.c()), kv_head,
                                   max_len, _ptr(out), _ptr(status), _stream_handle(stream))
    if st:
        raise VaError(st, "va_debug_gather_index")
    return out


def debug_split_ranges(p: Problem, kv: KV, mode: int = MODE_CHAIN, status=None, stream=None):
    """Each sequence's KV chunks as the partial kernels cut them: an int32
    tensor [num_seqs][slots][2] of (lo, hi) positions."""
    import torch
    slots = plan(p, kv, mode)["slots"]
    out = torch.full((max(p.num_seqs, 1), slots, 2), -2, dtype=torch.int32, device=p.cu_rows.device)
    st = lib.va_debug_split_ranges(ctypes.byref(p.c()), ctypes.byref(kv.c()), mode, _ptr(out),
                                   _ptr(status), _stream_handle(stream))
    if st:
        raise VaError(st, "va_debug_split_ranges")
    return out[:p.num_seqs]


def upload(case, device="cuda", num_splits=None, flags: int = 0):
    """Copy a host-side case (numpy storage arrays with the fields of the
    synthetic generator) into device tensors and return (Problem, KV, mode)."""
    import numpy as np
    import torch

    def dev(a, dt=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dt is not None:
            t = t.to(dt)
        return t.to(device)

    q = dev(case.q.view(np.int16) if case.q.dtype == np.uint16 else case.q)
    k = dev(case.k.view(np.int16) if case.k.dtype == np.uint16 else case.k)
    v = dev(case.v.view(np.int16) if case.v.dtype == np.uint16 else case.v)
    bt = None if case.block_table is None else dev(case.block_table.astype(np.int32))
    dk = getattr(case, "draft_k", None)
    dv = getattr(case, "draft_v", None)
    kv = KV(DTYPE_CODES[case.kv_dtype], case.num_kv_heads, case.head_dim, k, v,
            page_size=case.page_size, capacity=case.capacity, block_table=bt,
            max_blocks_per_seq=0 if bt is None else int(case.block_table.shape[1]),
            num_blocks=0 if bt is None else int(case.k.shape[0]),
            draft_k=None if dk is None else dev(dk.view(np.int16) if dk.dtype == np.uint16 else dk),
            draft_v=None if dv is None else dev(dv.view(np.int16) if dv.dtype == np.uint16 else dv))
    p = Problem(num_seqs=case.num_seqs, num_heads=case.num_heads,
                q_dtype=DTYPE_CODES[case.q_dtype], q=q,
                cu_rows=dev(case.cu_rows.astype(np.int32)),
                ctx_len=dev(case.ctx_len.astype(np.int32)),
                parent=dev(case.parent.astype(np.int32)),
                seq_kind=dev(case.seq_kind.astype(np.uint8)),
                total_rows=case.total_rows, max_rows_per_seq=max(1, case.max_rows_per_seq),
                scale=float(case.scale),
                num_splits=int(num_splits if num_splits is not None else case.num_splits),
                flags=flags)
    return p, kv, MODE_CODES[case.mode]


def timing_enable(on: bool) -> None:
    lib.va_timing_enable(1 if on else 0)


def timing_read(max_calls: int = 4096):
    """Per-call (partial_ms, merge_ms) lists of the calls recorded since
    timing was last enabled."""
    a = (ctypes.c_float * max_calls)()
    b = (ctypes.c_float * max_calls)()
    n = ctypes.c_int32(0)
    st = lib.va_timing_read(max_calls, a, b, ctypes.byref(n))
    if st:
        raise VaError(st, "va_timing_read")
    return list(a[:n.value]), list(b[:n.value])
