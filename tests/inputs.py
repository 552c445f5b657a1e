"""Seeded synthetic inputs for paged-KV gather / scatter / transfer.

This module is shared by the oracle side and the GPU side as *data only*: it draws slot
lists, page tables, run layouts and pool contents.  It holds none of the method's arithmetic
(no gather, no scatter, no address computation of a pool).

The pages' workloads are production TTS traffic and public prompts, which are not used here;
these shapes stand in for them (WORKLOADS, by name):

  small_gather_scatter  Qwen2.5-1.5B-shaped KV (28 layers, 2 kv heads, head_dim 128, fp16),
         slot-major pool of 4096 slots, one request of 128 distinct random slots: gather,
         then scatter back (3.5 MiB).
  transfer  36 layers x 8 kv heads x 128 bf16 (144 KiB/token), two pools of 65,536 slots,
         2048 + 2048 distinct random slots: pool-to-pool transfer (288 MiB each way).
  fragmented  the transfer shape on per-plane pools of 131,072 slots; one request of 1536
         tokens in runs of length ~Geometric(mean 1.6) placed at random non-overlapping starts
         with a free slot between runs, in shuffled address order: gather, then scatter into a
         fresh run layout.
  batch  64 requests of U{1000..2000} tokens, the transfer shape, token-paged pools of 262,144
         slots with page size 16 (distinct random pages, last page partial): one batch launch.
  hnd_permute  Qwen2.5-7B-shaped KV (28 layers, 4 kv heads, 128, bf16), seq 32,768, HND pages
         of 16 tokens in a 65,536-page pool with a random page table: fused permute gather,
         then the inverse rebuild into a second pool under an independent page table.

Values: elements ~N(0,1) (numpy PCG64, float64 draws rounded to float32 and then to the
KV dtype with round-to-nearest-even).  Destinations and guard bands hold quiet-NaN payload
patterns that N(0,1) never produces.  Seeds: 20261202 + 1000 * group + role, the group
being a workload's seed_id (1 to 5 in the order above) or a test's own number.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Tuple

import numpy as np

SEED_BASE = 20261202

# roles
ROLE_VALUES = 0
ROLE_SRC_SLOTS = 1
ROLE_DST_SLOTS = 2
ROLE_LENGTHS = 3
ROLE_DST_VALUES = 4


def seed(group: int, role: int) -> int:
    return SEED_BASE + 1000 * group + role


def rng(group: int, role: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed(group, role)))


ELEM_BYTES = {"fp16": 2, "bf16": 2, "fp8": 1}


def _e4m3_table() -> np.ndarray:
    """Every finite fp8 E4M3 value by code (NaN codes 0x7F / 0xFF excluded): sign, 4 exponent
    bits with bias 7, 3 mantissa bits, subnormals at exponent 0."""
    vals = np.full(256, np.nan)
    for code in range(256):
        if code & 0x7F == 0x7F:
            continue
        s, e, m = code >> 7, (code >> 3) & 0xF, code & 0x7
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals[code] = -mag if s else mag
    return vals


# ---------------------------------------------------------------------------------------
# values
# ---------------------------------------------------------------------------------------

def normal_bits(g: np.random.Generator, n_elems: int, dtype: str) -> np.ndarray:
    """n_elems N(0,1) values as raw bit patterns: uint16 of fp16 or bf16, uint8 of fp8 E4M3
    (nearest code, ties to the even code)."""
    x = g.standard_normal(n_elems).astype(np.float32)
    if dtype == "fp8":
        table = _e4m3_table()
        codes = np.flatnonzero(~np.isnan(table))
        order = codes[np.argsort(table[codes], kind="stable")]
        vals = table[order]
        xd = np.clip(x.astype(np.float64), vals[0], vals[-1])
        hi = np.clip(np.searchsorted(vals, xd), 1, len(vals) - 1)
        lo = hi - 1
        dlo, dhi = xd - vals[lo], vals[hi] - xd
        pick = np.where(dhi < dlo, hi, np.where(dlo < dhi, lo,
                        np.where(order[lo] % 2 == 0, lo, hi)))
        return order[pick].astype(np.uint8)
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16  # round to nearest even (no NaNs here)
        return rounded.astype(np.uint16)
    raise ValueError(dtype)


def sentinel_bits(n_elems: int, dtype: str, salt: int = 0) -> np.ndarray:
    """Quiet-NaN payload patterns: fp16 0x7E00 | 9-bit payload, bf16 0x7FC0 | 6-bit payload;
    fp8 E4M3 has two NaN codes only, 0x7F and 0xFF."""
    e = np.arange(n_elems, dtype=np.uint64) + np.uint64(salt) * np.uint64(0x9E3779B1)
    h = (e * np.uint64(0x9E3779B97F4A7C15)) >> np.uint64(40)
    if dtype == "fp8":
        return (np.uint8(0x7F) | ((h & np.uint64(1)) << np.uint64(7)).astype(np.uint8)).astype(np.uint8)
    if dtype == "fp16":
        return (np.uint16(0x7E00) | (h & np.uint64(0x1FF)).astype(np.uint16)).astype(np.uint16)
    if dtype == "bf16":
        return (np.uint16(0x7FC0) | (h & np.uint64(0x3F)).astype(np.uint16)).astype(np.uint16)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------------------
# index lists
# ---------------------------------------------------------------------------------------

def distinct_slots(g: np.random.Generator, n: int, num_slots: int) -> np.ndarray:
    """n distinct uniformly random slots in [0, num_slots)."""
    return g.choice(num_slots, size=n, replace=False).astype(np.int32)


def geometric_run_lengths(g: np.random.Generator, n_tokens: int, mean: float) -> List[int]:
    """Run lengths ~Geometric(p = 1/mean) on {1, 2, ...}, drawn until they cover n_tokens;
    the last one is truncated."""
    p = 1.0 / mean
    lens: List[int] = []
    total = 0
    while total < n_tokens:
        L = int(g.geometric(p))
        L = min(L, n_tokens - total)
        lens.append(L)
        total += L
    return lens


def fragmented_slots(g: np.random.Generator, n_tokens: int, num_slots: int,
                     mean_run: float = 1.6) -> Tuple[np.ndarray, List[int]]:
    """Slot list of n_tokens tokens in runs ~Geometric(mean_run).  Runs sit at random
    non-overlapping starts with at least one free slot between two runs (so neighbouring runs
    never merge), and are assigned to the request's token order in shuffled address order.
    Returns (slots, run_lengths in token order)."""
    lens = geometric_run_lengths(g, n_tokens, mean_run)
    k = len(lens)
    free = num_slots - n_tokens - (k - 1)
    assert free >= 0, "pool too small for this many runs"
    # random composition of the free slots into k + 1 gaps
    cuts = np.sort(g.integers(0, free + 1, size=k))
    gaps = np.diff(np.concatenate([[0], cuts]))
    # address-ordered run starts
    starts = []
    pos = 0
    for r in range(k):
        pos += int(gaps[r]) + (1 if r > 0 else 0)
        starts.append(pos)
        pos += lens[r]
    order = g.permutation(k)  # token order visits the runs in shuffled address order
    slots = np.empty(n_tokens, dtype=np.int32)
    t = 0
    run_lens_token_order = []
    for r in order:
        L = lens[r]
        slots[t:t + L] = np.arange(starts[r], starts[r] + L, dtype=np.int32)
        run_lens_token_order.append(L)
        t += L
    return slots, run_lens_token_order


def random_pages(g: np.random.Generator, n_pages: int, pool_pages: int) -> np.ndarray:
    """n_pages distinct random pages of a pool with pool_pages pages (a page table)."""
    return g.choice(pool_pages, size=n_pages, replace=False).astype(np.int32)


def paged_request_slots(g: np.random.Generator, lengths: List[int], page_size: int,
                        pool_slots: int) -> Tuple[np.ndarray, np.ndarray]:
    """Token-paged slot lists for several requests: request q takes ceil(len_q / page_size)
    distinct random pages (distinct across all requests); token t of a request sits at
    page[t // page_size] * page_size + t % page_size.  Returns (concatenated slots, offsets)."""
    pool_pages = pool_slots // page_size
    n_pages = [(L + page_size - 1) // page_size for L in lengths]
    pages = g.choice(pool_pages, size=sum(n_pages), replace=False).astype(np.int64)
    out = []
    offs = [0]
    pi = 0
    for L, npg in zip(lengths, n_pages):
        pt = pages[pi:pi + npg]
        pi += npg
        t = np.arange(L, dtype=np.int64)
        out.append((pt[t // page_size] * page_size + t % page_size).astype(np.int32))
        offs.append(offs[-1] + L)
    return np.concatenate(out) if out else np.zeros(0, np.int32), np.asarray(offs, np.int64)


def page_table_slots(page_table: np.ndarray, seq_len: int, page_size: int) -> np.ndarray:
    """The slot of every token of a sequence stored under a page table (test convenience for
    expressing a page-table gather as a slot-list gather)."""
    t = np.arange(seq_len, dtype=np.int64)
    return (page_table.astype(np.int64)[t // page_size] * page_size + t % page_size).astype(np.int32)


# ---------------------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    seed_id: int  # seed group of its inputs
    name: str
    num_layers: int
    kv_heads: int
    head_dim: int
    dtype: str
    layout: str  # "slot_major" | "planes" | "hnd"
    num_slots: int
    n_tokens: int
    page_size: int = 1
    n_requests: int = 1

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def planes(self) -> int:
        return 2 * self.num_layers

    @property
    def row_bytes(self) -> int:
        return self.kv_heads * self.head_dim * self.elem_bytes

    @property
    def bytes_per_token(self) -> int:
        return self.planes * self.row_bytes

    @property
    def payload_bytes(self) -> int:
        return self.n_tokens * self.bytes_per_token


WORKLOADS = {
    "small_gather_scatter": Workload(
        1, "qwen2.5-1.5b gather+scatter-back, slot-major pool, 128 tokens", 28, 2, 128, "fp16",
        "slot_major", 4096, 128),
    "transfer": Workload(
        2, "pool-to-pool transfer, 2048 random rows, 36x8x128 bf16 (288 MiB)", 36, 8, 128, "bf16",
        "planes", 65536, 2048),
    "fragmented": Workload(
        3, "fragmented gather+scatter, 1536 tokens in Geometric(1.6) runs", 36, 8, 128, "bf16",
        "planes", 131072, 1536),
    "batch": Workload(
        4, "batch of 64 requests U{1000..2000}, token-paged pools, page 16", 36, 8, 128, "bf16",
        "planes", 262144, 0, page_size=16, n_requests=64),
    "hnd_permute": Workload(
        5, "qwen2.5-7b fused HND->[S,H,D] gather + rebuild, seq 32768", 28, 4, 128, "bf16", "hnd",
        65536 * 16, 32768, page_size=16),
}


def batch_lengths(group: int = 4, n_requests: int = 64, lo: int = 1000,
                  hi: int = 2000) -> List[int]:
    """Prompt lengths U{lo..hi} inclusive (the batch workload's by default)."""
    g = rng(group, ROLE_LENGTHS)
    return [int(x) for x in g.integers(lo, hi + 1, size=n_requests)]
