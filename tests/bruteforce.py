"""Element-by-element model of the KV moves, for tiny layouts only.

Independent of the oracle: no byte arithmetic and no memcpy.  A pool is a numpy array whose
axes name the multi-index of every element, and each element is moved on its own in Python
loops.  Layout axes:

  planes      [plane][slot][head][dim]            (plane = kvp*layer + kv)
  slot_major  [slot][layer][kv][head][dim]
  hnd         [plane][page][head][page_size][dim]

kvp is the number of planes per layer: 2 (K, V) or 1 (one latent vector per layer, MLA).
The transfer buffer is [layer][kv][token][head][dim].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle


@dataclass
class BFPool:
    layout: str
    L: int
    H: int
    D: int
    num_slots: int
    data: np.ndarray  # uint16 elements
    page_size: int = 1
    kvp: int = 2

    def copy(self) -> "BFPool":
        return BFPool(self.layout, self.L, self.H, self.D, self.num_slots, self.data.copy(),
                      self.page_size, self.kvp)

    def get(self, layer, kv, slot, h, d):
        if self.layout == "planes":
            return self.data[self.kvp * layer + kv, slot, h, d]
        if self.layout == "slot_major":
            return self.data[slot, layer, kv, h, d]
        return self.data[self.kvp * layer + kv, slot // self.page_size, h, slot % self.page_size, d]

    def set(self, layer, kv, slot, h, d, v):
        if self.layout == "planes":
            self.data[self.kvp * layer + kv, slot, h, d] = v
        elif self.layout == "slot_major":
            self.data[slot, layer, kv, h, d] = v
        else:
            self.data[self.kvp * layer + kv, slot // self.page_size, h, slot % self.page_size, d] = v


def make_pool(layout, L, H, D, num_slots, fill, page_size=1, kvp=2) -> BFPool:
    """fill: callable(n) -> uint16 values, used in C order of the layout's axes."""
    if layout == "planes":
        shape = (kvp * L, num_slots, H, D)
    elif layout == "slot_major":
        shape = (num_slots, L, kvp, H, D)
    else:
        assert num_slots % page_size == 0
        shape = (kvp * L, num_slots // page_size, H, page_size, D)
    n = int(np.prod(shape))
    return BFPool(layout, L, H, D, num_slots, np.asarray(fill(n), np.uint16).reshape(shape),
                  page_size, kvp)


def to_oracle(pool: BFPool) -> oracle.Pool:
    """Describe the numpy memory of a BFPool to the oracle.  Plane offsets and the slot
    stride are read off numpy's own strides, not computed by hand."""
    base = pool.data
    planes = []
    for layer in range(pool.L):
        for kv in range(pool.kvp):
            if pool.layout == "planes":
                view = base[pool.kvp * layer + kv]
            elif pool.layout == "slot_major":
                view = base[:, layer, kv]
            else:
                view = base[pool.kvp * layer + kv]
            off = view.__array_interface__["data"][0] - base.__array_interface__["data"][0]
            planes.append((base, off))
    if pool.layout == "planes":
        kind, stride = oracle.TOKEN_ROWS, base.strides[1]
    elif pool.layout == "slot_major":
        kind, stride = oracle.TOKEN_ROWS, base.strides[0]
    else:
        kind, stride = oracle.HND_PAGES, 0
    return oracle.Pool(pool.L, pool.H, pool.D, 2, kind, pool.num_slots, planes, stride,
                       pool.page_size, pool.kvp)


def gather(pool: BFPool, slots) -> np.ndarray:
    n = len(slots)
    out = np.zeros((pool.L, pool.kvp, n, pool.H, pool.D), np.uint16)
    for layer in range(pool.L):
        for kv in range(pool.kvp):
            for i in range(n):
                for h in range(pool.H):
                    for d in range(pool.D):
                        out[layer, kv, i, h, d] = pool.get(layer, kv, int(slots[i]), h, d)
    return out


def scatter(pool: BFPool, slots, buf: np.ndarray) -> BFPool:
    res = pool.copy()
    for layer in range(pool.L):
        for kv in range(pool.kvp):
            for i in range(len(slots)):
                for h in range(pool.H):
                    for d in range(pool.D):
                        res.set(layer, kv, int(slots[i]), h, d, buf[layer, kv, i, h, d])
    return res


def transfer(src: BFPool, src_slots, dst: BFPool, dst_slots) -> BFPool:
    res = dst.copy()
    for layer in range(src.L):
        for kv in range(src.kvp):
            for i in range(len(src_slots)):
                for h in range(src.H):
                    for d in range(src.D):
                        res.set(layer, kv, int(dst_slots[i]), h, d,
                                src.get(layer, kv, int(src_slots[i]), h, d))
    return res


def transfer_layers(src: BFPool, src_slots, dst: BFPool, dst_slots, stop: int) -> BFPool:
    """transfer() of the layers before `stop` only."""
    res = dst.copy()
    for layer in range(stop):
        for kv in range(src.kvp):
            for i in range(len(src_slots)):
                for h in range(src.H):
                    for d in range(src.D):
                        res.set(layer, kv, int(dst_slots[i]), h, d,
                                src.get(layer, kv, int(src_slots[i]), h, d))
    return res


def transfer_owned(src: BFPool, src_slots, dst: BFPool, dst_slots, stop: int, page_epochs,
                   epoch_page: int, epoch: int) -> BFPool:
    """transfer_layers() of the rows whose destination page still holds epoch."""
    res = dst.copy()
    for layer in range(stop):
        for kv in range(src.kvp):
            for i in range(len(src_slots)):
                if page_epochs[int(dst_slots[i]) // epoch_page] != epoch:
                    continue
                for h in range(src.H):
                    for d in range(src.D):
                        res.set(layer, kv, int(dst_slots[i]), h, d,
                                src.get(layer, kv, int(src_slots[i]), h, d))
    return res


def move_heads(op, src: BFPool, src_slots, h0, dst: BFPool, dst_slots, g0, nh, buf=None):
    """Head-range move, element by element.  op 0: returns the buffer [layer][kv][n][nh][D];
    op 1 (buffer -> dst) and op 2 (src -> dst): return the new destination pool."""
    shape = dst if op == 1 else src
    n = len(dst_slots) if op == 1 else len(src_slots)
    if op == 0:
        out = np.zeros((shape.L, shape.kvp, n, nh, shape.D), np.uint16)
    else:
        out = dst.copy()
    for layer in range(shape.L):
        for kv in range(shape.kvp):
            for i in range(n):
                for j in range(nh):
                    for d in range(shape.D):
                        if op == 0:
                            out[layer, kv, i, j, d] = src.get(layer, kv, int(src_slots[i]), h0 + j, d)
                        elif op == 1:
                            out.set(layer, kv, int(dst_slots[i]), g0 + j, d, buf[layer, kv, i, j, d])
                        else:
                            out.set(layer, kv, int(dst_slots[i]), g0 + j, d,
                                    src.get(layer, kv, int(src_slots[i]), h0 + j, d))
    return out


def reshard(srcs, src_slots, dsts, dst_slots, parts):
    """Every part (src, dst, h0, g0, nh) as its own element-by-element head transfer into a
    copy of its destination pool; returns the new destination pools."""
    out = [d.copy() for d in dsts]
    for si, di, h0, g0, nh in parts:
        src, res = srcs[si], out[di]
        for layer in range(src.L):
            for kv in range(src.kvp):
                for i in range(len(src_slots)):
                    for j in range(nh):
                        for d in range(src.D):
                            res.set(layer, kv, int(dst_slots[i]), g0 + j, d,
                                    src.get(layer, kv, int(src_slots[i]), h0 + j, d))
    return out


def hnd_gather(pool: BFPool, page_table, seq_len) -> np.ndarray:
    """[layer][kv][s][h][d] = element (h, s, d) of the page-table view."""
    out = np.zeros((pool.L, pool.kvp, seq_len, pool.H, pool.D), np.uint16)
    ps = pool.page_size
    for layer in range(pool.L):
        for kv in range(pool.kvp):
            for s in range(seq_len):
                slot = int(page_table[s // ps]) * ps + s % ps
                for h in range(pool.H):
                    for d in range(pool.D):
                        out[layer, kv, s, h, d] = pool.get(layer, kv, slot, h, d)
    return out
