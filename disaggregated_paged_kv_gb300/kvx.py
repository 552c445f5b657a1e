"""Thin Python binding of libkvx (include/kvx.h).

Argument marshalling only: every step of a move runs in libkvx's kernels.  Each function here
maps one to one onto the C entry point of the same name without the ``kvx_`` prefix
(``gather`` -> ``kvx_gather``).  Device buffers may be given as torch tensors (their
``data_ptr()`` is passed) or as plain integer addresses; ``stream=None`` means torch's current
stream.  A non-OK return code raises :class:`KvxError`; device-side results land in the status
tensor the caller passes.

There is no fallback: if ``libkvx.so`` is missing the first call raises, telling the user to
build it (``python -m disaggregated_paged_kv_gb300.build`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvx.so")

# ---- constants (kvx.h) ------------------------------------------------------------------
OK = 0
ERR_INVALID_ARG = 1
ERR_ALIGNMENT = 2
ERR_OUT_OF_RANGE = 3
ERR_DUPLICATE_DST = 4
ERR_OVERLAP = 5
ERR_CUDA = 6
ERR_NO_WORKSPACE = 7
ERR_TIMEOUT = 8
ERR_CANCELLED = 9

F16, BF16, F32, FP8 = 1, 2, 3, 4
NHD, HND_PAGED = 0, 1
OP_GATHER, OP_SCATTER, OP_TRANSFER, OP_BATCH = 0, 1, 2, 3

MAX_PLANES = 256
PLAN_TILE = 2048
MAX_TOKENS = PLAN_TILE * 4096
CHUNK_BYTES = 2048
NOALLOC_MAX_TOKENS = 16384
NOALLOC_MAX_DUP_TOKENS = 8192

ELEM_BYTES = {F16: 2, BF16: 2, F32: 4, FP8: 1}


class KvxError(RuntimeError):
    """A non-OK kvx_status: `code` is the status, the message names the call."""

    def __init__(self, code: int, where: str):
        self.code = code
        msg = status_str(code)
        if code == ERR_CUDA:
            msg += f" (cudaError {last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{code}]")


class LayoutDesc(ctypes.Structure):
    """kvx_layout_desc (kvx.h), as given to kvx_layout_create."""
    _fields_ = [
        ("num_layers", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("kind", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_slots", ctypes.c_int64),
        ("plane_ptrs", ctypes.POINTER(ctypes.c_void_p)),
        ("base", ctypes.c_void_p),
        ("plane_stride", ctypes.c_int64),
        ("slot_stride", ctypes.c_int64),
        ("kv_planes", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class Request(ctypes.Structure):
    """kvx_request (kvx.h): one request of a batch, 32 bytes."""
    _fields_ = [
        ("op", ctypes.c_int32),
        ("n_tokens", ctypes.c_int32),
        ("src_off", ctypes.c_int64),
        ("dst_off", ctypes.c_int64),
        ("buf_off", ctypes.c_int64),
    ]


assert ctypes.sizeof(Request) == 32

MAX_WAIT_NS = 10_000_000_000


class StreamCtl(ctypes.Structure):
    """kvx_stream_ctl: pointers are device or pinned host addresses (or None)."""
    _fields_ = [
        ("layer_ready", ctypes.c_void_p),
        ("ready_value", ctypes.c_int32),
        ("epoch_word", ctypes.c_void_p),
        ("epoch", ctypes.c_int32),
        ("wait_ns", ctypes.c_int64),
        ("max_ctas", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("host_done", ctypes.c_void_p),
        ("dst_page_epochs", ctypes.c_void_p),
        ("epoch_page", ctypes.c_int32),
        ("reserved2", ctypes.c_int32),
    ]

class HeadPart(ctypes.Structure):
    """kvx_head_part: heads [src_head0, src_head0 + n_heads) of srcs[src] -> heads from
    dst_head0 of dsts[dst]."""
    _fields_ = [
        ("src", ctypes.c_int32),
        ("dst", ctypes.c_int32),
        ("src_head0", ctypes.c_int32),
        ("dst_head0", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


assert ctypes.sizeof(HeadPart) == 24

RESHARD_MAX_LAYOUTS = 64
RESHARD_MAX_PARTS = 128
RESHARD_MAX_PLANE_TABLE = 3072

_lib: Optional[ctypes.CDLL] = None

_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_U32 = ctypes.c_uint32

_SIGS = {
    "kvx_layout_create": (_I32, [ctypes.POINTER(LayoutDesc), ctypes.POINTER(_VP)]),
    "kvx_layout_destroy": (_I32, [_VP]),
    "kvx_layout_row_bytes": (_I64, [_VP]),
    "kvx_layout_num_planes": (_I32, [_VP]),
    "kvx_workspace_size": (_SZ, [_I64, _I32]),
    "kvx_gather": (_I32, [_VP, _VP, _I32, _VP, _SZ, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_scatter": (_I32, [_VP, _VP, _I32, _VP, _SZ, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_transfer": (_I32, [_VP, _VP, _VP, _VP, _I32, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_transfer_noalloc": (_I32, [_VP, _VP, _VP, _VP, _I32, _VP, _U32, _VP]),
    "kvx_gather_runs": (_I32, [_VP, _VP, _I32, _I32, _VP, _SZ, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_scatter_runs": (_I32, [_VP, _VP, _I32, _I32, _VP, _SZ, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_transfer_runs": (_I32, [_VP, _VP, _VP, _I32, _I32, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_batch": (_I32, [_VP, _VP, _VP, _I32, _I64, _VP, _I64, _VP, _I64, _VP, _SZ, _VP, _SZ,
                         _VP, _U32, _VP]),
    "kvx_submit": (_I32, [_I32, _VP, _VP, _VP, _VP, _I32, _VP, _SZ, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_stream": (_I32, [_I32, _VP, _VP, _VP, _VP, _I32, _VP, _SZ, ctypes.POINTER(StreamCtl),
                          _VP, _SZ, _VP, _U32, _VP]),
    "kvx_tp_slice": (_I32, [_I32, _I32, _I32, _I32, _I32, ctypes.POINTER(_I32),
                            ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "kvx_move_heads": (_I32, [_I32, _VP, _VP, _I32, _VP, _VP, _I32, _I32, _I32, _VP, _SZ, _VP,
                              _SZ, _VP, _U32, _VP]),
    "kvx_tp_plan": (_I32, [_I32, _I32, _I32, ctypes.POINTER(HeadPart), _I32,
                           ctypes.POINTER(_I32)]),
    "kvx_reshard": (_I32, [ctypes.POINTER(_VP), _I32, _VP, ctypes.POINTER(_VP), _I32, _VP,
                           ctypes.POINTER(HeadPart), _I32, _I32, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_stream_reshard": (_I32, [ctypes.POINTER(_VP), _I32, _VP, ctypes.POINTER(_VP), _I32, _VP,
                                  ctypes.POINTER(HeadPart), _I32, _I32, ctypes.POINTER(StreamCtl),
                                  _VP, _SZ, _VP, _U32, _VP]),
    "kvx_plan": (_I32, [_I32, _VP, _VP, _VP, _VP, _I32, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_plan_runs": (_I32, [_I32, _VP, _VP, _VP, _I32, _I32, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_plan_batch": (_I32, [_VP, _VP, _VP, _I32, _I64, _VP, _I64, _VP, _I64, _SZ, _VP, _SZ,
                              _VP, _U32, _VP]),
    "kvx_execute": (_I32, [_I32, _VP, _VP, _VP, _I32, _I64, _VP, _SZ, _VP, _SZ, _VP, _U32, _VP]),
    "kvx_plan_export": (_I32, [_VP, _SZ, _I64, _VP, _I64, _VP, _VP]),
    "kvx_status_str": (ctypes.c_char_p, [_I32]),
    "kvx_last_cuda_error": (_I32, []),
    "kvx_version": (_I32, []),
    "kvx_set_copy_engine": (_I32, [_I32]),
    "kvx_get_copy_engine": (_I32, []),
    "kvx_set_fused_max_tokens": (_I32, [_I32]),
    "kvx_get_fused_max_tokens": (_I32, []),
    "kvx_set_check_duplicates": (_I32, [_I32]),
    "kvx_get_check_duplicates": (_I32, []),
}


def lib() -> ctypes.CDLL:
    """The loaded libkvx.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libkvx.so not found at {LIB_PATH}; build it with "
                "`python -m disaggregated_paged_kv_gb300.build`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def exported_names() -> Sequence[str]:
    """The C entry points this binding declares (every KVX_API function of kvx.h)."""
    return tuple(_SIGS)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _nbytes(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        raise TypeError("give the byte size explicitly for a raw address")
    return int(x.numel() * x.element_size())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) or None
    if isinstance(stream, int):
        return stream or None
    return int(stream.cuda_stream) or None


def _flags(flags) -> int:
    """A call's flags word: None means DEFAULTS (the process-wide settings)."""
    return DEFAULTS if flags is None else int(flags)


def _check(rc: int, where: str) -> None:
    if rc != OK:
        raise KvxError(rc, where)


def status_str(code: int) -> str:
    """kvx_status_str: the status code's name."""
    return lib().kvx_status_str(code).decode()


def last_cuda_error() -> int:
    """kvx_last_cuda_error: the cudaError_t behind this thread's last KVX_ERR_CUDA."""
    return int(lib().kvx_last_cuda_error())


def version() -> int:
    """kvx_version: major * 10000 + minor * 100 + patch."""
    return int(lib().kvx_version())


ENGINE_AUTO, ENGINE_REGISTERS, ENGINE_BULK = 0, 1, 2

# per-call options (the flags argument of every call that moves rows)
DEFAULTS = 0xFFFFFFFF
CHECK_DUP = 0x1
USE_REGISTERS = 0x2
USE_BULK = 0x4
ONE_LAUNCH = 0x8


def set_copy_engine(engine: int) -> None:
    """Process-wide default copy engine (ENGINE_AUTO / _REGISTERS / _BULK) for flags=None."""
    _check(lib().kvx_set_copy_engine(engine), "kvx_set_copy_engine")


def get_copy_engine() -> int:
    """The process-wide default copy engine."""
    return int(lib().kvx_get_copy_engine())


FUSED_MAX_TOKENS = 8192


def set_fused_max_tokens(max_tokens: int) -> None:
    """Process-wide default limit of the one-launch path (0: off) for flags=None."""
    _check(lib().kvx_set_fused_max_tokens(max_tokens), "kvx_set_fused_max_tokens")


def get_fused_max_tokens() -> int:
    """The process-wide default limit of the one-launch path."""
    return int(lib().kvx_get_fused_max_tokens())


def set_check_duplicates(on: bool) -> None:
    """Process-wide default of the duplicate-destination check for flags=None."""
    _check(lib().kvx_set_check_duplicates(1 if on else 0), "kvx_set_check_duplicates")


def get_check_duplicates() -> bool:
    """The process-wide default of the duplicate-destination check."""
    return bool(lib().kvx_get_check_duplicates())


def workspace_size(max_tokens: int, max_requests: int = 0) -> int:
    """kvx_workspace_size: bytes of workspace for calls of up to max_tokens rows per plane and
    max_requests requests (batches) or runs (run lists)."""
    return int(lib().kvx_workspace_size(max_tokens, max_requests))


class Layout:
    """Owns a kvx_layout_t.  Plane addresses come either from ``plane_ptrs`` (a sequence of
    tensors or integer addresses, one per plane) or from ``base`` + p * ``plane_stride``."""

    def __init__(self, num_layers: int, kv_heads: int, head_dim: int, dtype: int,
                 num_slots: int, kind: int = NHD, page_size: int = 1, plane_ptrs=None,
                 base=None, plane_stride: int = 0, slot_stride: int = 0, keepalive=None,
                 kv_planes: int = 2):
        d = LayoutDesc()
        d.kv_planes = kv_planes
        d.num_layers, d.kv_heads, d.head_dim, d.dtype = num_layers, kv_heads, head_dim, dtype
        d.kind, d.page_size, d.num_slots = kind, page_size, num_slots
        self._ptr_array = None
        if plane_ptrs is not None:
            arr = (ctypes.c_void_p * len(plane_ptrs))(*[_ptr(p) for p in plane_ptrs])
            self._ptr_array = arr
            d.plane_ptrs = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        d.base = _ptr(base)
        d.plane_stride, d.slot_stride = plane_stride, slot_stride
        h = ctypes.c_void_p()
        _check(lib().kvx_layout_create(ctypes.byref(d), ctypes.byref(h)), "kvx_layout_create")
        self.handle = h.value
        self.num_layers, self.kv_heads, self.head_dim = num_layers, kv_heads, head_dim
        self.dtype, self.kind, self.page_size, self.num_slots = dtype, kind, page_size, num_slots
        self.kv_planes = kv_planes
        self._keepalive = keepalive  # tensors whose memory the planes point into

    @property
    def row_bytes(self) -> int:
        return int(lib().kvx_layout_row_bytes(self.handle))

    @property
    def num_planes(self) -> int:
        return int(lib().kvx_layout_num_planes(self.handle))

    def close(self) -> None:
        if getattr(self, "handle", None):
            lib().kvx_layout_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _h(layout: Optional[Layout]) -> Optional[int]:
    return None if layout is None else layout.handle


def gather(src: Layout, src_slots, n: int, buf, ws, status, buf_bytes=None, ws_bytes=None,
           flags=None, stream=None) -> None:
    """kvx_gather: buf[p][i] = row(src, p, src_slots[i]) for i < n; the device status word
    (status) gets KVX_OK or KVX_ERR_OUT_OF_RANGE (nothing written)."""
    rc = lib().kvx_gather(_h(src), _ptr(src_slots), n, _ptr(buf),
                          _nbytes(buf) if buf_bytes is None else buf_bytes, _ptr(ws),
                          _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                          _flags(flags), _stream(stream))
    _check(rc, "kvx_gather")


def scatter(dst: Layout, dst_slots, n: int, buf, ws, status, buf_bytes=None, ws_bytes=None,
            flags=None, stream=None) -> None:
    """kvx_scatter: row(dst, p, dst_slots[i]) = buf[p][i]; rows of other slots keep their bytes."""
    rc = lib().kvx_scatter(_h(dst), _ptr(dst_slots), n, _ptr(buf),
                           _nbytes(buf) if buf_bytes is None else buf_bytes, _ptr(ws),
                           _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                           _flags(flags), _stream(stream))
    _check(rc, "kvx_scatter")


def transfer(src: Layout, src_slots, dst: Layout, dst_slots, n: int, ws, status,
             ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_transfer: row(dst, p, dst_slots[i]) = row(src, p, src_slots[i]) for i < n."""
    rc = lib().kvx_transfer(_h(src), _ptr(src_slots), _h(dst), _ptr(dst_slots), n, _ptr(ws),
                            _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                            _flags(flags), _stream(stream))
    _check(rc, "kvx_transfer")


def transfer_noalloc(src: Layout, src_slots, dst: Layout, dst_slots, n: int, status,
                     flags=None, stream=None) -> None:
    """kvx_transfer without a workspace, for callers that cannot allocate device memory when
    KV has to move (the planner's scratch is a fixed array inside libkvx; n is at most
    NOALLOC_MAX_TOKENS, and calls that overlap on the GPU must not share it)."""
    rc = lib().kvx_transfer_noalloc(_h(src), _ptr(src_slots), _h(dst), _ptr(dst_slots), n,
                                    _ptr(status), _flags(flags), _stream(stream))
    _check(rc, "kvx_transfer_noalloc")


def gather_runs(src: Layout, runs, n_runs: int, n_tokens: int, buf, ws, status, buf_bytes=None,
                ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_gather_runs: runs is a device int32[n_runs][3] of (src_start, dst_start, len);
    the buffer fills in run order (its start field ignored)."""
    rc = lib().kvx_gather_runs(_h(src), _ptr(runs), n_runs, n_tokens, _ptr(buf),
                               _nbytes(buf) if buf_bytes is None else buf_bytes, _ptr(ws),
                               _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                               _flags(flags), _stream(stream))
    _check(rc, "kvx_gather_runs")


def scatter_runs(dst: Layout, runs, n_runs: int, n_tokens: int, buf, ws, status,
                 buf_bytes=None, ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_scatter_runs: the runs' destination slots take consecutive buffer rows."""
    rc = lib().kvx_scatter_runs(_h(dst), _ptr(runs), n_runs, n_tokens, _ptr(buf),
                                _nbytes(buf) if buf_bytes is None else buf_bytes, _ptr(ws),
                                _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                                _flags(flags), _stream(stream))
    _check(rc, "kvx_scatter_runs")


def transfer_runs(src: Layout, dst: Layout, runs, n_runs: int, n_tokens: int, ws, status,
                  ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_transfer_runs: rows src_start.. of each run to dst_start.. of the same run."""
    rc = lib().kvx_transfer_runs(_h(src), _h(dst), _ptr(runs), n_runs, n_tokens, _ptr(ws),
                                 _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                                 _flags(flags), _stream(stream))
    _check(rc, "kvx_transfer_runs")


def batch(src: Optional[Layout], dst: Optional[Layout], reqs, n_reqs: int, total_tokens: int,
          src_slots, n_src_slots: int, dst_slots, n_dst_slots: int, buf, ws, status,
          buf_bytes=None, ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_batch: the requests (device array of Request) in one plan + one copy; status has
    n_reqs + 1 words (overall, then each request's own)."""
    rc = lib().kvx_batch(_h(src), _h(dst), _ptr(reqs), n_reqs, total_tokens, _ptr(src_slots),
                         n_src_slots, _ptr(dst_slots), n_dst_slots, _ptr(buf),
                         _nbytes(buf) if buf_bytes is None else buf_bytes, _ptr(ws),
                         _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                         _flags(flags), _stream(stream))
    _check(rc, "kvx_batch")


def submit(op: int, src: Optional[Layout], h_src_slots, dst: Optional[Layout], h_dst_slots,
           n: int, buf, ws, h_status, buf_bytes=None, ws_bytes=None, flags=None, stream=None) -> None:
    """Host slot lists (pinned tensors or numpy arrays) and a host status word."""
    rc = lib().kvx_submit(op, _h(src), _host_ptr(h_src_slots), _h(dst), _host_ptr(h_dst_slots),
                          n, _ptr(buf), _nbytes(buf) if buf_bytes is None else buf_bytes,
                          _ptr(ws), _nbytes(ws) if ws_bytes is None else ws_bytes,
                          _host_ptr(h_status), _flags(flags), _stream(stream))
    _check(rc, "kvx_submit")


def _host_ptr(x) -> Optional[int]:
    if x is None or isinstance(x, int):
        return x
    if hasattr(x, "ctypes"):  # numpy
        return int(x.ctypes.data)
    return int(x.data_ptr())


def plan(op: int, src: Optional[Layout], src_slots, dst: Optional[Layout], dst_slots, n: int,
         ws, status, ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_plan: validate and plan a slot-list move into ws (run it with execute)."""
    rc = lib().kvx_plan(op, _h(src), _ptr(src_slots), _h(dst), _ptr(dst_slots), n, _ptr(ws),
                        _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                        _flags(flags), _stream(stream))
    _check(rc, "kvx_plan")


def plan_runs(op: int, src: Optional[Layout], dst: Optional[Layout], runs, n_runs: int,
              n_tokens: int, ws, status, ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_plan_runs: the plan of a run-list move."""
    rc = lib().kvx_plan_runs(op, _h(src), _h(dst), _ptr(runs), n_runs, n_tokens, _ptr(ws),
                             _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                             _flags(flags), _stream(stream))
    _check(rc, "kvx_plan_runs")


def plan_batch(src: Optional[Layout], dst: Optional[Layout], reqs, n_reqs: int,
               total_tokens: int, src_slots, n_src_slots: int, dst_slots, n_dst_slots: int,
               buf_bytes: int, ws, status, ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_plan_batch: the plan of a batch (execute it with op OP_BATCH)."""
    rc = lib().kvx_plan_batch(_h(src), _h(dst), _ptr(reqs), n_reqs, total_tokens,
                              _ptr(src_slots), n_src_slots, _ptr(dst_slots), n_dst_slots,
                              buf_bytes, _ptr(ws), _nbytes(ws) if ws_bytes is None else ws_bytes,
                              _ptr(status), _flags(flags), _stream(stream))
    _check(rc, "kvx_plan_batch")


def execute(op: int, src: Optional[Layout], dst: Optional[Layout], reqs, n_reqs: int,
            n_tokens: int, buf, ws, status, buf_bytes=None, ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_execute: the copy of the plan in ws; sizes must match the plan's (else
    KVX_ERR_INVALID_ARG on the device)."""
    rc = lib().kvx_execute(op, _h(src), _h(dst), _ptr(reqs), n_reqs, n_tokens, _ptr(buf),
                           _nbytes(buf) if buf_bytes is None else buf_bytes, _ptr(ws),
                           _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                           _flags(flags), _stream(stream))
    _check(rc, "kvx_execute")


def plan_export(ws, n_tokens: int, out, max_chunks: int, count, ws_bytes=None,
                stream=None) -> None:
    """kvx_plan_export: the plan's chunks as int32[count][4] (request, source offset,
    destination offset, rows), for inspection."""
    rc = lib().kvx_plan_export(_ptr(ws), _nbytes(ws) if ws_bytes is None else ws_bytes,
                               n_tokens, _ptr(out), max_chunks, _ptr(count), _stream(stream))
    _check(rc, "kvx_plan_export")


def stream(op: int, src: Optional[Layout], src_slots, dst: Optional[Layout], dst_slots, n: int,
           buf, ws, status, layer_ready=None, ready_value: int = 1, epoch_word=None,
           epoch: int = 0, wait_ns: int = 100_000_000, max_ctas: int = 0, host_done=None,
           dst_page_epochs=None, epoch_page: int = 1, buf_bytes=None, ws_bytes=None,
           flags=None, stream=None) -> None:
    """kvx_stream: a gather / scatter / transfer that moves layer l once
    ``layer_ready[l] >= ready_value`` and stops when ``epoch_word`` no longer holds ``epoch``
    or a layer's wait exceeds ``wait_ns``.  ``status`` is a device int32[4] (verdict, layers
    pending, internal, done).  Control words may be device tensors or pinned host tensors."""
    ctl = _stream_ctl(layer_ready, ready_value, epoch_word, epoch, wait_ns, max_ctas, host_done,
                      dst_page_epochs, epoch_page)
    rc = lib().kvx_stream(op, _h(src), _ptr(src_slots), _h(dst), _ptr(dst_slots), n, _ptr(buf),
                          _nbytes(buf) if buf_bytes is None else buf_bytes, ctypes.byref(ctl),
                          _ptr(ws), _nbytes(ws) if ws_bytes is None else ws_bytes,
                          _ptr(status), _flags(flags), _stream(stream))
    _check(rc, "kvx_stream")


def _stream_ctl(layer_ready, ready_value, epoch_word, epoch, wait_ns, max_ctas, host_done,
                dst_page_epochs, epoch_page) -> StreamCtl:
    ctl = StreamCtl()
    ctl.layer_ready = _any_ptr(layer_ready)
    ctl.ready_value = ready_value
    ctl.epoch_word = _any_ptr(epoch_word)
    ctl.epoch = epoch
    ctl.wait_ns = wait_ns
    ctl.max_ctas = max_ctas
    ctl.reserved = 0
    ctl.host_done = _any_ptr(host_done)
    ctl.dst_page_epochs = _any_ptr(dst_page_epochs)
    ctl.epoch_page = epoch_page if dst_page_epochs is not None else 0
    ctl.reserved2 = 0
    return ctl


def stream_reshard(srcs: Sequence[Optional[Layout]], src_slots, dsts: Sequence[Optional[Layout]],
                   dst_slots, parts, n: int, ws, status, layer_ready=None, ready_value: int = 1,
                   epoch_word=None, epoch: int = 0, wait_ns: int = 100_000_000, host_done=None,
                   dst_page_epochs=None, epoch_page: int = 1, max_ctas: int = 0, ws_bytes=None,
                   flags=None, stream=None) -> None:
    """kvx_stream_reshard: kvx_reshard moving layer l once ``layer_ready[l] >= ready_value``,
    stopping on a changed epoch word or a wait past ``wait_ns``; ``status`` is a device
    int32[4] as for stream(); ``max_ctas`` > 0 caps the grid as for stream()."""
    ctl = _stream_ctl(layer_ready, ready_value, epoch_word, epoch, wait_ns, max_ctas, host_done,
                      dst_page_epochs, epoch_page)
    sa = (_VP * max(1, len(srcs)))(*[_h(x) for x in srcs])
    da = (_VP * max(1, len(dsts)))(*[_h(x) for x in dsts])
    pa = (HeadPart * max(1, len(parts)))()
    for k, q in enumerate(parts):
        vals = tuple(int(x) for x in q)
        pa[k] = HeadPart(*(vals + (0,) * (6 - len(vals))))
    rc = lib().kvx_stream_reshard(sa, len(srcs), _ptr(src_slots), da, len(dsts),
                                  _ptr(dst_slots), pa, len(parts), n, ctypes.byref(ctl),
                                  _ptr(ws), _nbytes(ws) if ws_bytes is None else ws_bytes,
                                  _ptr(status), _flags(flags), _stream(stream))
    _check(rc, "kvx_stream_reshard")


def _any_ptr(x) -> Optional[int]:
    """Address of a tensor (device or pinned host), a numpy array or an integer."""
    if x is None or isinstance(x, int):
        return x
    if hasattr(x, "ctypes"):
        return int(x.ctypes.data)
    return int(x.data_ptr())


def tp_slice(kv_heads: int, src_tp: int, src_rank: int, dst_tp: int, dst_rank: int):
    """kvx_tp_slice: (src_head0, dst_head0, n_heads) a source rank sends a destination rank."""
    a, b, c = _I32(0), _I32(0), _I32(0)
    _check(lib().kvx_tp_slice(kv_heads, src_tp, src_rank, dst_tp, dst_rank, ctypes.byref(a),
                              ctypes.byref(b), ctypes.byref(c)), "kvx_tp_slice")
    return a.value, b.value, c.value


def tp_plan(kv_heads: int, src_tp: int, dst_tp: int):
    """kvx_tp_plan: the whole reshard plan between TP groups of sizes src_tp and dst_tp, as a
    list of (src rank, dst rank, src_head0, dst_head0, n_heads)."""
    n = _I32(0)
    rc = lib().kvx_tp_plan(kv_heads, src_tp, dst_tp, None, 0, ctypes.byref(n))
    if rc != OK and n.value == 0:
        _check(rc, "kvx_tp_plan")
    arr = (HeadPart * max(1, n.value))()
    _check(lib().kvx_tp_plan(kv_heads, src_tp, dst_tp, arr, n.value, ctypes.byref(n)),
           "kvx_tp_plan")
    return [(q.src, q.dst, q.src_head0, q.dst_head0, q.n_heads) for q in arr[:n.value]]


def reshard(srcs: Sequence[Optional[Layout]], src_slots, dsts: Sequence[Optional[Layout]],
            dst_slots, parts, n: int, ws, status, ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_reshard: every part (src, dst, src_head0, dst_head0, n_heads) of a reshard between
    the pools of two TP groups, in one planner + one copy launch."""
    sa = (_VP * max(1, len(srcs)))(*[_h(x) for x in srcs])
    da = (_VP * max(1, len(dsts)))(*[_h(x) for x in dsts])
    pa = (HeadPart * max(1, len(parts)))()
    for k, q in enumerate(parts):
        vals = tuple(int(x) for x in q)
        pa[k] = HeadPart(*(vals + (0,) * (6 - len(vals))))
    rc = lib().kvx_reshard(sa, len(srcs), _ptr(src_slots), da, len(dsts), _ptr(dst_slots), pa,
                           len(parts), n, _ptr(ws), _nbytes(ws) if ws_bytes is None else ws_bytes,
                           _ptr(status), _flags(flags), _stream(stream))
    _check(rc, "kvx_reshard")


def move_heads(op: int, src: Optional[Layout], src_slots, src_head0: int, dst: Optional[Layout],
               dst_slots, dst_head0: int, n_heads: int, n: int, buf, ws, status, buf_bytes=None,
               ws_bytes=None, flags=None, stream=None) -> None:
    """kvx_move_heads: heads [src_head0, src_head0 + n_heads) of each source row to heads
    [dst_head0, ...) of each destination row (layouts may have different kv_heads)."""
    rc = lib().kvx_move_heads(op, _h(src), _ptr(src_slots), src_head0, _h(dst), _ptr(dst_slots),
                              dst_head0, n_heads, n, _ptr(buf),
                              _nbytes(buf) if buf_bytes is None else buf_bytes, _ptr(ws),
                              _nbytes(ws) if ws_bytes is None else ws_bytes, _ptr(status),
                              _flags(flags), _stream(stream))
    _check(rc, "kvx_move_heads")


# ---- checked calls -------------------------------------------------------------------------
# The one-shot moves in the short form: gather(layout, slots, buf) and its siblings with the
# workspace and the status word supplied here, the stream synchronised after the call, and a
# device-side error (an index out of range, a repeated destination under KVX_CHECK_DUP)
# raised as KvxError.  Each host thread keeps its own workspace and status word per device,
# grown as needed, so threads on different streams do not share them.  The caller's buffers
# and slot lists are torch tensors on the same device.


_scratch = threading.local()


def _scratch_for(device, n_tokens: int):
    import torch
    per = getattr(_scratch, "by_device", None)
    if per is None:
        per = _scratch.by_device = {}
    idx = device.index if device.index is not None else torch.cuda.current_device()
    need = workspace_size(max(1, n_tokens), 0)
    ws, st = per.get(idx, (None, None))
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=torch.device("cuda", idx))
        st = torch.empty(4, dtype=torch.int32, device=torch.device("cuda", idx))
        per[idx] = (ws, st)
    return ws, st


def _sync_and_raise(st, stream, where: str) -> None:
    import torch
    if stream is None:
        torch.cuda.current_stream(st.device).synchronize()
    elif isinstance(stream, int):
        torch.cuda.ExternalStream(stream, device=st.device).synchronize()
    else:
        stream.synchronize()
    code = int(st[0].item())
    if code != OK:
        raise KvxError(code, where + " (device status)")


def gather_sync(src: Layout, slots, buf, flags=None, stream=None) -> None:
    """buf[p][i] = row(src, p, slots[i]) for the n = slots.numel() tokens; raises KvxError if
    any slot is out of range (nothing is written then)."""
    n = int(slots.numel())
    ws, st = _scratch_for(slots.device, n)
    gather(src, slots, n, buf, ws, st, flags=flags, stream=stream)
    _sync_and_raise(st, stream, "kvx_gather")


def scatter_sync(dst: Layout, slots, buf, flags=None, stream=None) -> None:
    """row(dst, p, slots[i]) = buf[p][i]; raises KvxError on a bad slot (or, with CHECK_DUP, a
    repeated one), with nothing written."""
    n = int(slots.numel())
    ws, st = _scratch_for(slots.device, n)
    scatter(dst, slots, n, buf, ws, st, flags=flags, stream=stream)
    _sync_and_raise(st, stream, "kvx_scatter")


def transfer_sync(src: Layout, src_slots, dst: Layout, dst_slots, flags=None,
                  stream=None) -> None:
    """row(dst, p, dst_slots[i]) = row(src, p, src_slots[i]); raises KvxError on a bad slot
    (or, with CHECK_DUP, a repeated destination), with nothing written."""
    n = int(src_slots.numel())
    if int(dst_slots.numel()) != n:
        raise ValueError("the two slot lists differ in length")
    ws, st = _scratch_for(src_slots.device, n)
    transfer(src, src_slots, dst, dst_slots, n, ws, st, flags=flags, stream=stream)
    _sync_and_raise(st, stream, "kvx_transfer")
