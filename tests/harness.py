"""Host/device mirrors of pools and buffers for parity tests.

A :class:`Mirror` holds one pool (or transfer buffer) twice: as a numpy byte array for the
oracle and as a CUDA tensor for libkvx, both wrapped in 64 KiB guard bands of quiet-NaN
sentinels.  After a libkvx call the device bytes -- guard bands included -- are read back and
compared with the oracle's bytes.  The oracle learns where the planes are from numpy views
(:func:`oracle_pool`); libkvx from an explicit layout description (:func:`kvx_layout`).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

import oracle
from tests import inputs

GUARD = 64 * 1024


def _shape(kind: str, L: int, H: int, D: int, num_slots: int, ps: int, kvp: int = 2):
    if kind in ("planes", "planes_separate", "planes_rotated"):
        return (kvp * L, num_slots, H, D)
    if kind == "slot_major":
        return (num_slots, L, kvp, H, D)
    if kind == "hnd":
        assert num_slots % ps == 0
        return (kvp * L, num_slots // ps, H, ps, D)
    raise ValueError(kind)


@dataclass
class Mirror:
    kind: str  # planes | planes_separate | planes_rotated | slot_major | hnd | buffer
    L: int
    H: int
    D: int
    dtype: str
    num_slots: int
    page_size: int
    host: np.ndarray       # uint8, guard + body + guard
    body: np.ndarray       # element view (uint16, or uint8 for fp8) with the layout's axes
    dev: object = None     # torch uint8 tensor mirroring host
    kvp: int = 2           # planes per layer: 2 (K, V) or 1 (MLA latent)

    @property
    def elem(self) -> int:
        return inputs.ELEM_BYTES[self.dtype]

    @property
    def R(self) -> int:
        return self.H * self.D * self.elem

    @property
    def P(self) -> int:
        return self.kvp * self.L

    def to_device(self):
        import torch
        self.dev = torch.from_numpy(self.host).to("cuda")
        return self

    def readback(self) -> np.ndarray:
        return self.dev.cpu().numpy()

    def dev_body_ptr(self) -> int:
        return int(self.dev.data_ptr()) + GUARD


def make_mirror(kind: str, L: int, H: int, D: int, dtype: str, num_slots: int = 0,
                page_size: int = 1, fill: str = "normal", g: Optional[np.random.Generator] = None,
                n_tokens: int = 0, salt: int = 0, kvp: int = 2) -> Mirror:
    """fill: 'normal' (N(0,1) values from g) or 'sentinel' (quiet-NaN payloads)."""
    if kind == "buffer":
        shape = (kvp * L, n_tokens, H, D)
    else:
        shape = _shape(kind, L, H, D, num_slots, page_size, kvp)
    e = inputs.ELEM_BYTES[dtype]
    n_el = int(np.prod(shape))
    host = np.empty(2 * GUARD + e * n_el, dtype=np.uint8)
    host[:GUARD] = inputs.sentinel_bits(GUARD // e, dtype, salt + 1).view(np.uint8)
    host[GUARD + e * n_el:] = inputs.sentinel_bits(GUARD // e, dtype, salt + 2).view(np.uint8)
    body = host[GUARD:GUARD + e * n_el].view(np.uint16 if e == 2 else np.uint8).reshape(shape)
    if fill == "normal":
        body.reshape(-1)[:] = inputs.normal_bits(g, n_el, dtype)
    else:
        body.reshape(-1)[:] = inputs.sentinel_bits(n_el, dtype, salt)
    return Mirror(kind, L, H, D, dtype, num_slots, page_size, host, body, kvp=kvp)


def oracle_pool(m: Mirror) -> oracle.Pool:
    """Plane addresses from numpy views of the body (numpy does the address arithmetic)."""
    base_addr = m.host.__array_interface__["data"][0]
    planes = []
    for layer in range(m.L):
        for kv in range(m.kvp):
            if m.kind == "slot_major":
                view = m.body[:, layer, kv]
            elif m.kind == "planes_separate":  # plane p stored in block P-1-p
                view = m.body[m.P - 1 - (m.kvp * layer + kv)]
            elif m.kind == "planes_rotated":  # plane p stored in block (p + P/2) % P
                view = m.body[(m.kvp * layer + kv + m.P // 2) % m.P]
            else:
                view = m.body[m.kvp * layer + kv]
            planes.append((m.host, view.__array_interface__["data"][0] - base_addr))
    if m.kind == "slot_major":
        return oracle.Pool(m.L, m.H, m.D, m.elem, oracle.TOKEN_ROWS, m.num_slots, planes,
                           m.body.strides[0], kv_planes=m.kvp)
    if m.kind == "hnd":
        return oracle.Pool(m.L, m.H, m.D, m.elem, oracle.HND_PAGES, m.num_slots, planes, 0,
                           m.page_size, kv_planes=m.kvp)
    return oracle.Pool(m.L, m.H, m.D, m.elem, oracle.TOKEN_ROWS, m.num_slots, planes,
                       m.body.strides[1], kv_planes=m.kvp)


KVX_DTYPE = {"fp16": 1, "bf16": 2, "fp8": 4}


def kvx_layout(m: Mirror):
    """libkvx layout handle for the device copy of m."""
    from disaggregated_paged_kv_gb300 import kvx
    base = m.dev_body_ptr()
    R, P = m.R, m.P
    dt = KVX_DTYPE[m.dtype]
    kvp = m.kvp
    if m.kind == "planes":
        return kvx.Layout(m.L, m.H, m.D, dt, m.num_slots, base=base,
                          plane_stride=m.num_slots * R, keepalive=m.dev, kv_planes=kvp)
    if m.kind == "planes_separate":
        ptrs = [base + (P - 1 - p) * m.num_slots * R for p in range(P)]
        return kvx.Layout(m.L, m.H, m.D, dt, m.num_slots, plane_ptrs=ptrs, keepalive=m.dev,
                          kv_planes=kvp)
    if m.kind == "planes_rotated":  # plane addresses not a constant stride apart
        ptrs = [base + ((p + P // 2) % P) * m.num_slots * R for p in range(P)]
        return kvx.Layout(m.L, m.H, m.D, dt, m.num_slots, plane_ptrs=ptrs, keepalive=m.dev,
                          kv_planes=kvp)
    if m.kind == "slot_major":
        return kvx.Layout(m.L, m.H, m.D, dt, m.num_slots, base=base, plane_stride=R,
                          slot_stride=P * R, keepalive=m.dev, kv_planes=kvp)
    if m.kind == "hnd":
        return kvx.Layout(m.L, m.H, m.D, dt, m.num_slots, kind=kvx.HND_PAGED,
                          page_size=m.page_size, base=base, plane_stride=m.num_slots * R,
                          keepalive=m.dev, kv_planes=kvp)
    raise ValueError(m.kind)


def buffer_body_bytes(m: Mirror) -> np.ndarray:
    return m.host[GUARD:len(m.host) - GUARD]


def first_mismatch(a: np.ndarray, b: np.ndarray) -> Optional[int]:
    if a.shape != b.shape:
        return -1
    d = np.flatnonzero(a != b)
    return int(d[0]) if len(d) else None


def assert_same_bytes(got: np.ndarray, want: np.ndarray, what: str) -> None:
    i = first_mismatch(got, want)
    assert i is None, f"{what}: bytes differ (first at {i} of {len(want)}; guard {GUARD})"


def workspace(max_tokens: int, max_requests: int = 0):
    import torch
    from disaggregated_paged_kv_gb300 import kvx
    n = kvx.workspace_size(max(1, max_tokens), max_requests)
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def status(n: int = 1):
    import torch
    return torch.full((n,), -1, dtype=torch.int32, device="cuda")


def dev_i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to("cuda")
