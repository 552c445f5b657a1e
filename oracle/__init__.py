"""CPU oracle for paged-KV gather / scatter / transfer (ctypes wrapper of kvx_oracle.c).

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may load this module; the library path never does.  It shares no code
with the CUDA library: the C source computes every address on its own from the pages'
definitions (see the header comment of ``kvx_oracle.h`` for the passages followed).

Pools are described by numpy byte arrays: a :class:`Pool` holds one base array plus the byte
offset of every plane inside it (or one array per plane), so the same numpy memory can be
copied to the GPU and compared byte for byte afterwards.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvx_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkvx_oracle.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_OUT_OF_RANGE = 3
ERR_DUPLICATE_DST = 4

TOKEN_ROWS = 0
HND_PAGES = 1

OP_GATHER = 0
OP_SCATTER = 1
OP_TRANSFER = 2


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with the host C compiler (plain -O2, no vectorisation flags)."""
    cmd = ["gcc", "-O2", "-std=c99", "-Wall", "-Wextra", "-shared", "-fPIC", src, "-o", out]
    subprocess.run(cmd, check=True)
    return out


class _Pool(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("elem_bytes", ctypes.c_int32),
        ("kind", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_slots", ctypes.c_int64),
        ("planes", ctypes.POINTER(ctypes.c_void_p)),
        ("slot_stride", ctypes.c_int64),
        ("kv_planes", ctypes.c_int32),
    ]


class Request(ctypes.Structure):
    _fields_ = [
        ("op", ctypes.c_int32),
        ("n_tokens", ctypes.c_int32),
        ("src_off", ctypes.c_int64),
        ("dst_off", ctypes.c_int64),
        ("buf_off", ctypes.c_int64),
    ]


class Run(ctypes.Structure):
    _fields_ = [("req", ctypes.c_int32), ("src", ctypes.c_int32), ("dst", ctypes.c_int32),
                ("len", ctypes.c_int32)]


class Part(ctypes.Structure):
    """kvxo_part: heads [src_head0, src_head0 + n_heads) of srcs[src] -> heads from dst_head0
    of dsts[dst]."""
    _fields_ = [("src", ctypes.c_int32), ("dst", ctypes.c_int32), ("src_head0", ctypes.c_int32),
                ("dst_head0", ctypes.c_int32), ("n_heads", ctypes.c_int32)]


_lib_cache = {}


def load(path: str = _LIB_PATH) -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library at ``path``."""
    if path in _lib_cache:
        return _lib_cache[path]
    if not os.path.exists(path) or (path == _LIB_PATH and
                                    os.path.getmtime(path) < os.path.getmtime(_SRC)):
        build(out=path)
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    i32p, u8p = P(ctypes.c_int32), ctypes.c_void_p
    lib.kvxo_bytes_per_token.restype = ctypes.c_int64
    lib.kvxo_bytes_per_token.argtypes = [ctypes.c_int32] * 4
    lib.kvxo_mla_bytes_per_token.restype = ctypes.c_int64
    lib.kvxo_mla_bytes_per_token.argtypes = [ctypes.c_int32] * 4
    lib.kvxo_row_bytes.restype = ctypes.c_int64
    lib.kvxo_row_bytes.argtypes = [P(_Pool)]
    lib.kvxo_check_slots.argtypes = [P(_Pool), i32p, ctypes.c_int64]
    lib.kvxo_has_duplicate.argtypes = [i32p, ctypes.c_int64, ctypes.c_int64]
    lib.kvxo_gather.argtypes = [P(_Pool), i32p, ctypes.c_int64, u8p, P(ctypes.c_int64)]
    lib.kvxo_scatter.argtypes = [P(_Pool), i32p, ctypes.c_int64, u8p, ctypes.c_int,
                                 P(ctypes.c_int64)]
    lib.kvxo_transfer.argtypes = [P(_Pool), i32p, P(_Pool), i32p, ctypes.c_int64, ctypes.c_int,
                                  P(ctypes.c_int64)]
    lib.kvxo_transfer_layers.argtypes = [P(_Pool), i32p, P(_Pool), i32p, ctypes.c_int64,
                                         ctypes.c_int32, P(ctypes.c_int64)]
    lib.kvxo_transfer_owned.argtypes = [P(_Pool), i32p, P(_Pool), i32p, ctypes.c_int64,
                                        ctypes.c_int32, i32p, ctypes.c_int32, ctypes.c_int32,
                                        P(ctypes.c_int64)]
    lib.kvxo_move_heads.argtypes = [ctypes.c_int32, P(_Pool), i32p, ctypes.c_int32, P(_Pool),
                                    i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, u8p,
                                    P(ctypes.c_int64)]
    lib.kvxo_tp_slice.argtypes = [ctypes.c_int32] * 5 + [P(ctypes.c_int32)] * 3
    lib.kvxo_reshard.argtypes = [P(P(_Pool)), ctypes.c_int32, i32p, P(P(_Pool)), ctypes.c_int32,
                                 i32p, P(Part), ctypes.c_int32, ctypes.c_int64,
                                 P(ctypes.c_int64)]
    lib.kvxo_hnd_gather.argtypes = [P(_Pool), i32p, ctypes.c_int64, u8p]
    lib.kvxo_hnd_rebuild.argtypes = [P(_Pool), i32p, ctypes.c_int64, u8p]
    lib.kvxo_batch.argtypes = [P(_Pool), P(_Pool), P(Request), ctypes.c_int32, i32p,
                               ctypes.c_int64, i32p, ctypes.c_int64, u8p, ctypes.c_int64,
                               ctypes.c_int, i32p]
    lib.kvxo_runs.restype = ctypes.c_int64
    lib.kvxo_runs.argtypes = [i32p, i32p, ctypes.c_int64, P(ctypes.c_int64), ctypes.c_int32,
                              P(Run), ctypes.c_int64]
    _lib_cache[path] = lib
    return lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i32p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


@dataclass
class Pool:
    """A KV pool in host memory.

    ``planes`` holds, for every plane p = kv_planes*layer + kv, a pair (array, byte_offset):
    the plane starts ``byte_offset`` bytes into the uint8 view of ``array``.  ``kind`` is
    TOKEN_ROWS (slot s at ``slot_stride * s``) or HND_PAGES ([page][head][page_size][dim]).
    ``kv_planes`` is 2 (K and V) or 1 (one latent plane per layer, MLA).
    """

    num_layers: int
    kv_heads: int
    head_dim: int
    elem_bytes: int
    kind: int
    num_slots: int
    planes: List[tuple]
    slot_stride: int = 0
    page_size: int = 1
    kv_planes: int = 2
    _keep: list = field(default_factory=list, repr=False)

    @property
    def num_planes(self) -> int:
        return self.kv_planes * self.num_layers

    @property
    def row_bytes(self) -> int:
        return self.kv_heads * self.head_dim * self.elem_bytes

    def _struct(self) -> _Pool:
        ptrs = (ctypes.c_void_p * self.num_planes)()
        for p, (arr, off) in enumerate(self.planes):
            assert arr.flags["C_CONTIGUOUS"]
            ptrs[p] = arr.ctypes.data + int(off)
        s = _Pool(self.num_layers, self.kv_heads, self.head_dim, self.elem_bytes, self.kind,
                  self.page_size, self.num_slots, ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)),
                  self.slot_stride, self.kv_planes)
        self._keep = [ptrs]
        return s


def mla_bytes_per_token(num_layers: int, latent_dim: int, rope_dim: int, elem_bytes: int,
                        lib=None) -> int:
    return int((lib or load()).kvxo_mla_bytes_per_token(num_layers, latent_dim, rope_dim,
                                                         elem_bytes))


def bytes_per_token(num_layers: int, kv_heads: int, head_dim: int, elem_bytes: int,
                    lib: Optional[ctypes.CDLL] = None) -> int:
    return int((lib or load()).kvxo_bytes_per_token(num_layers, kv_heads, head_dim, elem_bytes))


def gather(pool: Pool, slots, lib=None):
    """Returns (status, buffer bytes [P*n*R] (None on error), bytes written)."""
    lib = lib or load()
    slots = _i32(slots)
    n = len(slots)
    buf = np.zeros(max(1, pool.num_planes * n * pool.row_bytes), dtype=np.uint8)
    written = ctypes.c_int64(0)
    ps = pool._struct()
    rc = lib.kvxo_gather(ctypes.byref(ps), _i32p(slots), n, buf.ctypes.data, ctypes.byref(written))
    if rc != OK:
        return rc, None, 0
    return rc, buf[: pool.num_planes * n * pool.row_bytes], written.value


def scatter(pool: Pool, slots, buf: np.ndarray, check_dup: bool = False, lib=None):
    lib = lib or load()
    slots = _i32(slots)
    buf = np.ascontiguousarray(buf).view(np.uint8)
    written = ctypes.c_int64(0)
    ps = pool._struct()
    rc = lib.kvxo_scatter(ctypes.byref(ps), _i32p(slots), len(slots), buf.ctypes.data,
                          int(check_dup), ctypes.byref(written))
    return rc, written.value


def transfer(src: Pool, src_slots, dst: Pool, dst_slots, check_dup: bool = False, lib=None):
    lib = lib or load()
    a, b = _i32(src_slots), _i32(dst_slots)
    assert len(a) == len(b)
    written = ctypes.c_int64(0)
    s1, s2 = src._struct(), dst._struct()
    rc = lib.kvxo_transfer(ctypes.byref(s1), _i32p(a), ctypes.byref(s2), _i32p(b), len(a),
                           int(check_dup), ctypes.byref(written))
    return rc, written.value


def transfer_layers(src: Pool, src_slots, dst: Pool, dst_slots, stop: int, lib=None):
    """kvxo_transfer_layers: the transfer of layers 0 .. stop-1 only."""
    lib = lib or load()
    a, b = _i32(src_slots), _i32(dst_slots)
    assert len(a) == len(b)
    written = ctypes.c_int64(0)
    s1, s2 = src._struct(), dst._struct()
    rc = lib.kvxo_transfer_layers(ctypes.byref(s1), _i32p(a), ctypes.byref(s2), _i32p(b), len(a),
                                  int(stop), ctypes.byref(written))
    return rc, written.value


def transfer_owned(src: Pool, src_slots, dst: Pool, dst_slots, stop: int, page_epochs,
                   epoch_page: int, epoch: int, lib=None):
    """kvxo_transfer_owned: rows of layers < stop whose destination page still holds epoch."""
    lib = lib or load()
    a, b, e = _i32(src_slots), _i32(dst_slots), _i32(page_epochs)
    assert len(a) == len(b)
    written = ctypes.c_int64(0)
    s1, s2 = src._struct(), dst._struct()
    rc = lib.kvxo_transfer_owned(ctypes.byref(s1), _i32p(a), ctypes.byref(s2), _i32p(b), len(a),
                                 int(stop), _i32p(e), int(epoch_page), int(epoch),
                                 ctypes.byref(written))
    return rc, written.value


def move_heads(op: int, src: Optional[Pool], src_slots, src_head0: int, dst: Optional[Pool],
               dst_slots, dst_head0: int, n_heads: int, n: int, buf: Optional[np.ndarray] = None,
               lib=None):
    """kvxo_move_heads.  op 0 gather returns (status, buffer bytes); 1 scatter reads ``buf``;
    2 transfer.  Returns (status, buffer or None, bytes written)."""
    lib = lib or load()
    a = _i32(src_slots if src_slots is not None else [])
    b = _i32(dst_slots if dst_slots is not None else [])
    shape = dst if op == 1 else src
    if op == 0:
        buf = np.zeros(max(1, shape.num_planes * n * n_heads * shape.head_dim * shape.elem_bytes),
                       dtype=np.uint8)
    written = ctypes.c_int64(0)
    s1 = src._struct() if src is not None else None
    s2 = dst._struct() if dst is not None else None
    bp = np.ascontiguousarray(buf).view(np.uint8) if buf is not None else None
    rc = lib.kvxo_move_heads(op, ctypes.byref(s1) if s1 is not None else None, _i32p(a),
                             src_head0, ctypes.byref(s2) if s2 is not None else None, _i32p(b),
                             dst_head0, n_heads, n, bp.ctypes.data if bp is not None else None,
                             ctypes.byref(written))
    return rc, (bp if op == 0 else None), written.value


def reshard(srcs: Sequence[Optional[Pool]], src_slots, dsts: Sequence[Optional[Pool]], dst_slots,
            parts, n: int, lib=None):
    """kvxo_reshard.  parts: sequence of (src, dst, src_head0, dst_head0, n_heads).  The
    destination pools are written in place.  Returns (status, bytes written)."""
    lib = lib or load()
    a = _i32(src_slots if src_slots is not None else [])
    b = _i32(dst_slots if dst_slots is not None else [])
    keep = [p._struct() if p is not None else None for p in list(srcs) + list(dsts)]
    ptr = lambda s: ctypes.pointer(s) if s is not None else ctypes.POINTER(_Pool)()
    sa = (ctypes.POINTER(_Pool) * max(1, len(srcs)))(*[ptr(s) for s in keep[:len(srcs)]])
    da = (ctypes.POINTER(_Pool) * max(1, len(dsts)))(*[ptr(s) for s in keep[len(srcs):]])
    pa = (Part * max(1, len(parts)))(*[Part(*map(int, q)) for q in parts])
    written = ctypes.c_int64(0)
    rc = lib.kvxo_reshard(sa, len(srcs), _i32p(a), da, len(dsts), _i32p(b), pa, len(parts), n,
                          ctypes.byref(written))
    return rc, written.value


def tp_slice(heads: int, p_tp: int, p_rank: int, d_tp: int, d_rank: int, lib=None):
    """kvxo_tp_slice: (status, src_head0, dst_head0, n_heads)."""
    lib = lib or load()
    a, b, c = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    rc = lib.kvxo_tp_slice(heads, p_tp, p_rank, d_tp, d_rank, ctypes.byref(a), ctypes.byref(b),
                           ctypes.byref(c))
    return rc, a.value, b.value, c.value


def hnd_gather(pool: Pool, page_table, seq_len: int, lib=None):
    lib = lib or load()
    pt = _i32(page_table)
    buf = np.zeros(max(1, pool.num_planes * seq_len * pool.row_bytes), dtype=np.uint8)
    ps = pool._struct()
    rc = lib.kvxo_hnd_gather(ctypes.byref(ps), _i32p(pt), seq_len, buf.ctypes.data)
    if rc != OK:
        return rc, None
    return rc, buf[: pool.num_planes * seq_len * pool.row_bytes]


def hnd_rebuild(pool: Pool, page_table, seq_len: int, buf: np.ndarray, lib=None):
    lib = lib or load()
    pt = _i32(page_table)
    buf = np.ascontiguousarray(buf).view(np.uint8)
    ps = pool._struct()
    return lib.kvxo_hnd_rebuild(ctypes.byref(ps), _i32p(pt), seq_len, buf.ctypes.data)


def batch(src: Optional[Pool], dst: Optional[Pool], reqs: Sequence[tuple], src_slots,
          dst_slots, buf: np.ndarray, check_dup: bool = False, lib=None) -> np.ndarray:
    """reqs: sequence of (op, n_tokens, src_off, dst_off, buf_off).  Returns status[n+1]."""
    lib = lib or load()
    arr = (Request * max(1, len(reqs)))(*[Request(*r) for r in reqs])
    a, b = _i32(src_slots), _i32(dst_slots)
    status = np.zeros(len(reqs) + 1, dtype=np.int32)
    s1 = src._struct() if src is not None else None
    s2 = dst._struct() if dst is not None else None
    buf = buf.view(np.uint8)
    lib.kvxo_batch(ctypes.byref(s1) if s1 else None, ctypes.byref(s2) if s2 else None, arr,
                   len(reqs), _i32p(a), len(a), _i32p(b), len(b), buf.ctypes.data, buf.nbytes,
                   int(check_dup), _i32p(status))
    return status


def runs(src_idx, dst_idx, req_start=(0,), lib=None) -> np.ndarray:
    """Run-length coalescing of two index lists (kvxo_runs); returns an int32 array
    [n_runs][4] = (req, src, dst, len) in token order."""
    lib = lib or load()
    a, b = _i32(src_idx), _i32(dst_idx)
    assert len(a) == len(b)
    rs = np.ascontiguousarray(np.asarray(req_start, dtype=np.int64))
    n = len(a)
    out = (Run * max(1, n))()
    cnt = lib.kvxo_runs(_i32p(a), _i32p(b), n, rs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                        len(rs), out, n)
    assert 0 <= cnt <= n
    return np.frombuffer(out, dtype=np.int32).reshape(-1, 4)[:cnt].copy()
