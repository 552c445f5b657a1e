"""Whole-pool parity at full size.

Device pools of many GiB are read back into host memory in chunks of at most 1 GiB (through one
pinned staging buffer), the CPU oracle runs over those host copies with the request's real slot
lists and page tables, and every byte of the device's destination is then compared, chunk by
chunk, with the oracle's.  Nothing here computes an expected value: it only moves bytes between
the device and host memory, fills host memory with a sentinel, and compares.  Host-side copies,
fills and comparisons are split over the host's cores (numpy releases the GIL for them).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 30
_THREADS = max(1, min(16, os.cpu_count() or 1))
_pool = ThreadPoolExecutor(_THREADS)


def mem_available() -> int:
    """MemAvailable of this host, in bytes."""
    with open("/proc/meminfo") as f:
        for ln in f:
            if ln.startswith("MemAvailable:"):
                return int(ln.split()[1]) * 1024
    return 0


def require_host_bytes(nbytes: int):
    """Skips the calling test, saying why, when the host cannot hold nbytes (+ 8 GiB spare)."""
    import pytest

    have = mem_available()
    if have < nbytes + (8 << 30):
        pytest.skip(f"whole-pool parity needs {nbytes / 2**30:.1f} GiB of host memory; "
                    f"{have / 2**30:.1f} GiB available")


def _parts(n: int):
    step = -(-n // _THREADS)
    step = (step + 4095) & ~4095
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def par_copy(dst: np.ndarray, src: np.ndarray):
    """dst[:] = src for flat uint8 arrays of equal length, over the host's cores."""
    list(_pool.map(lambda ab: np.copyto(dst[ab[0]:ab[1]], src[ab[0]:ab[1]]), _parts(len(dst))))


def par_equal(a: np.ndarray, b: np.ndarray) -> bool:
    return all(_pool.map(lambda ab: np.array_equal(a[ab[0]:ab[1]], b[ab[0]:ab[1]]),
                         _parts(len(a))))


def filled(nbytes: int, sentinel16: int) -> np.ndarray:
    """A host uint8 array of nbytes holding the 16-bit sentinel in every element."""
    out = np.empty(nbytes, dtype=np.uint8)
    v = out.view(np.uint16)
    list(_pool.map(lambda ab: v[ab[0]:ab[1]].fill(sentinel16), _parts(len(v))))
    return out


class Stager:
    """One pinned host buffer of CHUNK bytes through which device bytes are read back."""

    def __init__(self):
        import torch

        self.torch = torch
        self.pinned = torch.empty(CHUNK, dtype=torch.uint8, pin_memory=True)
        self.np = self.pinned.numpy()

    def flat(self, t):
        assert t.is_contiguous()
        return t.reshape(-1).view(self.torch.uint8)

    def chunks(self, t):
        """Yields (offset, host view) for every chunk of device tensor t, read back in turn."""
        f = self.flat(t)
        n = f.numel()
        for a in range(0, n, CHUNK):
            b = min(n, a + CHUNK)
            self.pinned[: b - a].copy_(f[a:b])
            yield a, self.np[: b - a]

    def to_host(self, t, out: np.ndarray = None, at: int = 0) -> np.ndarray:
        """The bytes of device tensor t in host memory (into out[at:] if given)."""
        n = self.flat(t).numel()
        if out is None:
            out, at = np.empty(n, dtype=np.uint8), 0
        for a, h in self.chunks(t):
            par_copy(out[at + a: at + a + len(h)], h)
        return out

    def assert_equal(self, t, want: np.ndarray, what: str, row_bytes: int = 0):
        """Every byte of device tensor t equals want (flat uint8); on a mismatch, names the
        first differing byte (and its row, given row_bytes)."""
        n = self.flat(t).numel()
        assert want.size == n, f"{what}: {n} device bytes against {want.size} expected"
        for a, h in self.chunks(t):
            w = want[a: a + len(h)]
            if not par_equal(h, w):
                i = a + int(np.flatnonzero(h != w)[0])
                where = f" (row {i // row_bytes}, byte {i % row_bytes})" if row_bytes else ""
                raise AssertionError(f"{what}: first difference at byte {i}{where}: device "
                                     f"{int(h[i - a])}, oracle {int(want[i])}")


GUARD = 64 * 1024


def guarded(shape, dtype, fill: str, sentinel16: int, seed: int = 0):
    """A device tensor of `shape` and torch `dtype` between two 64 KiB guard bands holding the
    16-bit sentinel: returns (the whole uint8 tensor, the tensor).  fill is "normal" (seeded
    N(0,1)), "bytes" (seeded uniform bytes, for uint8 tensors) or "sentinel"."""
    import torch

    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    whole = torch.empty(n + 2 * GUARD, dtype=torch.uint8, device="cuda")
    whole.view(torch.int16).fill_(sentinel16 - 65536 if sentinel16 >= 32768 else sentinel16)
    body = whole[GUARD: GUARD + n].view(dtype).view(shape)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    if fill == "normal":
        torch.randn(shape, dtype=dtype, device="cuda", generator=g, out=body)
    elif fill == "bytes":
        torch.randint(0, 256, shape, dtype=dtype, device="cuda", generator=g, out=body)
    else:
        assert fill == "sentinel", fill
    return whole, body
