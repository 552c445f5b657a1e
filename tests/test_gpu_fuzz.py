"""Randomised parity sweep: many small random cases over the cross product of layouts, element
widths, row shapes, calls, per-call options, sizes and planted errors, each compared byte for
byte with the oracle over the whole destination (pool or buffer, guard bands included), with
the source checked unchanged and the status word(s) compared.

The parametrised tests elsewhere vary one axis at a time; here they mix: a narrow HND
destination behind the bulk engine, a duplicate check on a run list into a slot-major pool, a
batch of fp8 rows with a planted bad index, the one-launch option on 2 KiB rows, ...  Every
case comes from its own seeded generator (the case number is its test id), so a failure reruns
alone; `test_fuzz_cases_draw` (no GPU) draws every case and checks that it is well formed.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

N_CASES = 600
POOL_CAP = 24 << 20  # bytes per pool
KINDS = ["planes", "planes_rotated", "slot_major", "hnd"]
# oneshot: kvx_gather / kvx_scatter / kvx_transfer by the case's op
CALLS = ["oneshot", "gather_runs", "scatter_runs", "transfer_runs", "batch", "plan_execute",
         "submit", "noalloc"]
CALL_P = [0.40, 0.07, 0.07, 0.08, 0.14, 0.10, 0.07, 0.07]
# per-call option words (None: KVX_DEFAULTS with random process-wide defaults)
FLAG_CHOICES = [None, 0, 1, 2, 4, 8, 1 | 2, 1 | 4, 1 | 8, 2 | 8, 4 | 8]
CHECK_DUP = 1
OP = {"gather": 0, "scatter": 1, "transfer": 2}
NOALLOC_MAX, NOALLOC_MAX_DUP = 16384, 8192


@dataclass
class Side:
    kind: str
    num: int
    ps: int


@dataclass
class Case:
    k: int
    dtype: str
    L: int
    H: int
    D: int
    kvp: int
    call: str
    op: str                  # gather / scatter / transfer (a batch's requests have their own)
    flags: Optional[int]
    defaults: tuple          # (check_dup, engine, fused_max) when flags is None
    src: Optional[Side]
    dst: Optional[Side]
    s: np.ndarray            # source slots (gather / transfer)
    d: np.ndarray            # destination slots (scatter / transfer)
    plant: str               # none / oor / dup
    reqs: List[tuple] = field(default_factory=list)  # batch: (op, n, src_off, dst_off, buf_off)
    buf_bytes: int = 0

    @property
    def R(self) -> int:
        return self.H * self.D * inputs.ELEM_BYTES[self.dtype]

    @property
    def P(self) -> int:
        return self.kvp * self.L

    @property
    def n(self) -> int:
        return len(self.s) if self.op != "scatter" else len(self.d)

    @property
    def check_dup(self) -> bool:
        return bool(self.defaults[0]) if self.flags is None else bool(self.flags & CHECK_DUP)


def _side(g, kind, n, cap_slots):
    ps = int(g.choice([1, 4, 16])) if kind == "hnd" else 1
    num = int(min(cap_slots, max(64, int(n * g.uniform(2.0, 4.0)) + 16)))
    num -= num % ps
    return Side(kind, num, ps)


def _slots(g, n, num, distinct=True):
    """A slot list of n tokens in [0, num): contiguous runs of random lengths, or uniformly
    random distinct slots, or (distinct=False) draws with repeats."""
    if n == 0:
        return np.zeros(0, np.int32)
    if not distinct:
        return g.integers(0, num, n).astype(np.int32)
    mean = float(g.choice([1.0, 1.6, 8.0, 64.0]))
    if mean == 1.0 or num < 2 * n + 2:
        return inputs.distinct_slots(g, n, num)
    return inputs.fragmented_slots(g, n, num, mean)[0]


def _plant(g, c: Case):
    """Plants the case's error into its slot lists (none / out of range / duplicate)."""
    if c.plant == "oor":
        reads = c.op != "scatter"
        writes = c.op != "gather"
        side = "s" if reads and (not writes or g.random() < 0.5) else "d"
        lst = c.s if side == "s" else c.d
        num = (c.src if side == "s" else c.dst).num
        lst[int(g.integers(0, len(lst)))] = int(g.choice([num, num + 7, -1, 2 ** 31 - 1]))
    elif c.plant == "dup":
        i, j = g.choice(len(c.d), 2, replace=False)
        c.d[j] = c.d[i]


def draw(k: int) -> Case:
    g = np.random.Generator(np.random.PCG64(31000 + k))
    dtype = str(g.choice(["fp8", "fp16", "bf16"]))
    H = int(g.choice([1, 2, 3, 4, 8]))
    D = int(g.choice([1, 3, 8, 16, 24, 36, 64, 100, 128]))  # rows of 1 byte to 2 KiB
    L = int(g.choice([1, 2, 3, 5]))
    kvp = 1 if g.random() < 0.25 else 2
    call = str(g.choice(CALLS, p=CALL_P))
    op = {"gather_runs": "gather", "scatter_runs": "scatter", "transfer_runs": "transfer",
          "noalloc": "transfer", "batch": "transfer"}.get(call)
    if op is None:
        op = str(g.choice(["gather", "scatter", "transfer"]))
    flags = FLAG_CHOICES[int(g.integers(0, len(FLAG_CHOICES)))]
    defaults = (int(g.integers(0, 2)), int(g.integers(0, 3)), int(g.choice([0, 512])))
    e = inputs.ELEM_BYTES[dtype]
    R = H * D * e
    cap_slots = max(64, POOL_CAP // (kvp * L * R))
    bucket = g.choice(["zero", "tiny", "small", "mid", "large"], p=[0.03, 0.17, 0.3, 0.3, 0.2])
    n = {"zero": 0, "tiny": int(g.integers(1, 17)), "small": int(g.integers(17, 513)),
         "mid": int(g.integers(513, 2100)), "large": int(g.integers(2100, 5000))}[bucket]
    n = min(n, cap_slots // 2 - 8)
    if call == "noalloc":
        n = min(n, NOALLOC_MAX)
    src = _side(g, str(g.choice(KINDS)), n, cap_slots) if op != "scatter" else None
    dst = _side(g, str(g.choice(KINDS)), n, cap_slots) if op != "gather" else None
    c = Case(k, dtype, L, H, D, kvp, call, op, flags, defaults, src, dst,
             np.zeros(0, np.int32), np.zeros(0, np.int32), "none")
    if call == "noalloc" and c.check_dup:
        n = min(n, NOALLOC_MAX_DUP)
    if src is not None:
        c.s = _slots(g, n, src.num, distinct=g.random() < 0.85)
    if dst is not None:
        c.d = _slots(g, n, dst.num)
    if n > 0:
        u = g.random()
        if u < 0.15:
            c.plant = "oor"
        elif u < 0.55 and c.check_dup and dst is not None and n >= 2:
            c.plant = "dup"
    if call == "batch":
        _draw_batch(g, c)
    else:
        _plant(g, c)
    return c


def _draw_batch(g, c: Case):
    """Splits the n tokens into requests of random ops over the concatenated slot lists; one
    request may carry a planted error (a bad index, or a destination slot another request or
    itself names again)."""
    n = len(c.s)
    cuts = np.sort(g.choice(np.arange(1, n), min(int(g.integers(0, 8)), max(0, n - 1)),
                            replace=False)) if n > 1 else np.zeros(0, int)
    bounds = np.concatenate([[0], cuts, [n]]).astype(int)
    bo = 0
    for a, b in zip(bounds[:-1], bounds[1:]):
        op = int(g.choice([0, 1, 2]))
        ln = int(b - a)
        boff = 0
        if op != 2:
            boff = bo
            bo += -(-c.P * ln * c.R // 16) * 16  # regions start on 16 bytes
        c.reqs.append((op, ln, int(a), int(a), boff))
    c.buf_bytes = max(16, bo)
    if c.plant == "oor":
        q = int(g.integers(0, len(c.reqs)))
        op, ln, so, do, _ = c.reqs[q]
        if ln > 0:
            if op == 1:
                c.d[do + int(g.integers(0, ln))] = c.dst.num
            else:
                c.s[so + int(g.integers(0, ln))] = int(g.choice([c.src.num, -3]))
    elif c.plant == "dup":
        writers = [r for r in c.reqs if r[0] != 0 and r[1] > 0]
        if writers:
            a = writers[int(g.integers(0, len(writers)))]
            b = writers[int(g.integers(0, len(writers)))]
            i = a[3] + int(g.integers(0, a[1]))
            j = b[3] + int(g.integers(0, b[1]))
            if i != j:
                c.d[j] = c.d[i]


# ---------------------------------------------------------------------------------------
# no GPU: the draws themselves
# ---------------------------------------------------------------------------------------

def test_fuzz_cases_draw():
    """Every case draws without error, fits the pool cap, and keeps its destination slots
    distinct unless a duplicate is planted under the check (the result of a repeat without
    the check is unspecified, so it is never compared)."""
    calls, plants = set(), set()
    for k in range(N_CASES):
        c = draw(k)
        calls.add(c.call)
        plants.add(c.plant)
        for side in (c.src, c.dst):
            if side is not None:
                assert side.num * c.P * c.R <= POOL_CAP + 64 * c.P * c.R
                assert side.num % side.ps == 0
        if c.dst is not None and c.plant != "dup":
            writes = c.d if c.call != "batch" else np.concatenate(
                [c.d[r[3]:r[3] + r[1]] for r in c.reqs if r[0] != 0] or [np.zeros(0, np.int32)])
            inr = writes[(writes >= 0) & (writes < c.dst.num)]
            assert len(np.unique(inr)) == len(inr), k
        if c.call == "batch":
            assert all(r[4] % 16 == 0 for r in c.reqs)
            assert sum(r[1] for r in c.reqs) == len(c.s)
        if c.call == "noalloc":
            assert c.n <= (NOALLOC_MAX_DUP if c.check_dup else NOALLOC_MAX)
    assert calls == set(CALLS)
    assert plants == {"none", "oor", "dup"}


# ---------------------------------------------------------------------------------------
# GPU
# ---------------------------------------------------------------------------------------

def _runs(s, d):
    """Maximal runs (src_start, dst_start, len) of two index lists, then some cut in two and a
    zero-length run added, as a caller's own run list might be."""
    runs, i, n = [], 0, len(s)
    while i < n:
        j = i + 1
        while j < n and int(s[j]) == int(s[j - 1]) + 1 and int(d[j]) == int(d[j - 1]) + 1:
            j += 1
        runs.append((int(s[i]), int(d[i]), j - i))
        i = j
    out = []
    for r, (a, b, ln) in enumerate(runs):
        if ln > 3 and r % 3 == 0:
            h = ln // 2
            out += [(a, b, h), (a + h, b + h, ln - h)]
        else:
            out.append((a, b, ln))
    out.insert(len(out) // 2, (0, 0, 0))
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("k", range(N_CASES))
def test_fuzz_case(k):
    torch = pytest.importorskip("torch")
    from disaggregated_paged_kv_gb300 import kvx

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    c = draw(k)
    g = np.random.Generator(np.random.PCG64(41000 + k))
    n, P, R = c.n, c.P, c.R

    def mirror(side, fill, salt):
        return hz.make_mirror(side.kind, c.L, c.H, c.D, c.dtype, side.num, side.ps, fill,
                              g if fill == "normal" else None, salt=salt, kvp=c.kvp)

    src = mirror(c.src, "normal", 0).to_device() if c.src else None
    dst = mirror(c.dst, "sentinel", 5).to_device() if c.dst else None
    exp_dst = mirror(c.dst, "sentinel", 5) if c.dst else None
    uses_buf = c.call == "batch" or c.op != "transfer"
    buf_n = c.buf_bytes if c.call == "batch" else P * n * R if uses_buf else 0
    buf = exp_buf = bufp = None
    if uses_buf:  # (a gather or scatter names a buffer even when it moves nothing)
        raw = g.integers(0, 256, 2 * hz.GUARD + max(16, buf_n), dtype=np.uint8)
        buf = torch.from_numpy(raw).cuda()
        exp_buf = raw.copy()
        bufp = hz.GUARD + buf.data_ptr()

    # the oracle's result
    dup = c.check_dup
    if c.call == "batch":
        want_status = list(oracle.batch(hz.oracle_pool(src), hz.oracle_pool(exp_dst), c.reqs, c.s,
                                        c.d, exp_buf[hz.GUARD:hz.GUARD + buf_n], check_dup=dup))
    elif c.op == "gather":
        rc, out, _ = oracle.gather(hz.oracle_pool(src), c.s)
        if rc == oracle.OK and n:
            exp_buf[hz.GUARD:hz.GUARD + buf_n] = out
        want_status = [rc]
    elif c.op == "scatter":
        body = exp_buf[hz.GUARD:hz.GUARD + max(16, buf_n)]
        want_status = [oracle.scatter(hz.oracle_pool(exp_dst), c.d, body, check_dup=dup)[0]]
    else:
        want_status = [oracle.transfer(hz.oracle_pool(src), c.s, hz.oracle_pool(exp_dst), c.d,
                                       check_dup=dup)[0]]

    # the same call through libkvx
    if c.flags is None:
        kvx.set_check_duplicates(bool(c.defaults[0]))
        kvx.set_copy_engine(c.defaults[1])
        kvx.set_fused_max_tokens(c.defaults[2])
    try:
        sl = hz.kvx_layout(src) if src else None
        dl = hz.kvx_layout(dst) if dst else None
        s_d = hz.dev_i32(c.s) if len(c.s) else None
        d_d = hz.dev_i32(c.d) if len(c.d) else None
        nst = len(c.reqs) + 1 if c.call == "batch" else 1
        st = hz.status(nst)
        f = c.flags
        if c.call == "oneshot":
            ws = hz.workspace(n)
            if c.op == "gather":
                kvx.gather(sl, s_d, n, bufp, ws, st, buf_bytes=buf_n, flags=f)
            elif c.op == "scatter":
                kvx.scatter(dl, d_d, n, bufp, ws, st, buf_bytes=buf_n, flags=f)
            else:
                kvx.transfer(sl, s_d, dl, d_d, n, ws, st, flags=f)
        elif c.call.endswith("_runs"):
            runs = _runs(c.s if len(c.s) else np.arange(n), c.d if len(c.d) else np.arange(n))
            rt = hz.dev_i32(np.asarray(runs, np.int32).reshape(-1))
            ws = hz.workspace(n, len(runs))
            if c.op == "gather":
                kvx.gather_runs(sl, rt, len(runs), n, bufp, ws, st, buf_bytes=buf_n, flags=f)
            elif c.op == "scatter":
                kvx.scatter_runs(dl, rt, len(runs), n, bufp, ws, st, buf_bytes=buf_n, flags=f)
            else:
                kvx.transfer_runs(sl, dl, rt, len(runs), n, ws, st, flags=f)
        elif c.call == "batch":
            dreq = torch.from_numpy(np.frombuffer(
                b"".join(bytes(kvx.Request(*r)) for r in c.reqs) or bytes(32),
                dtype=np.uint8).copy()).cuda()
            ws = hz.workspace(n, len(c.reqs))
            if k % 2 == 0:
                kvx.batch(sl, dl, dreq, len(c.reqs), n, s_d, len(c.s), d_d, len(c.d), bufp, ws,
                          st, buf_bytes=buf_n, flags=f)
            else:  # the same batch as plan + execute
                kvx.plan_batch(sl, dl, dreq, len(c.reqs), n, s_d, len(c.s), d_d, len(c.d), buf_n,
                               ws, st, flags=f)
                kvx.execute(kvx.OP_BATCH, sl, dl, dreq, len(c.reqs), n, bufp, ws, st,
                            buf_bytes=buf_n, flags=f)
        elif c.call == "plan_execute":
            ws = hz.workspace(n)
            kvx.plan(OP[c.op], sl, s_d, dl, d_d, n, ws, st, flags=f)
            kvx.execute(OP[c.op], sl, dl, None, 0, n, bufp, ws, st, buf_bytes=buf_n, flags=f)
        elif c.call == "submit":
            ws = hz.workspace(n)
            if k % 3:  # pinned lists and status word, read in place by the kernels
                hs = torch.from_numpy(c.s.copy()).pin_memory() if len(c.s) else None
                hd = torch.from_numpy(c.d.copy()).pin_memory() if len(c.d) else None
                hst = torch.full((1,), -1, dtype=torch.int32).pin_memory()
            else:  # pageable ones, staged by the call
                hs = c.s.copy() if len(c.s) else None
                hd = c.d.copy() if len(c.d) else None
                hst = np.full(1, -1, dtype=np.int32)
            kvx.submit(OP[c.op], sl, hs, dl, hd, n, bufp, ws, hst, buf_bytes=buf_n, flags=f)
        else:  # noalloc
            kvx.transfer_noalloc(sl, s_d, dl, d_d, n, st, flags=f)
        torch.cuda.synchronize()
        got_status = [int(hst[0])] if c.call == "submit" else st.cpu().numpy().tolist()
    finally:
        kvx.set_check_duplicates(False)
        kvx.set_copy_engine(kvx.ENGINE_AUTO)
        kvx.set_fused_max_tokens(0)

    what = f"case {k}: {c.call} {c.op} {c.dtype} L{c.L} H{c.H} D{c.D} kvp{c.kvp} n{n} " \
           f"flags {c.flags} plant {c.plant} src {c.src} dst {c.dst}"
    if n == 0 and c.call != "batch":
        want_status = [kvx.OK]
    assert got_status == want_status, what
    if dst is not None:
        hz.assert_same_bytes(dst.readback(), exp_dst.host, what + ": destination pool")
    if src is not None:
        hz.assert_same_bytes(src.readback(), src.host, what + ": source pool")
    if uses_buf:
        hz.assert_same_bytes(buf.cpu().numpy(), exp_buf, what + ": buffer")


# ---------------------------------------------------------------------------------------
# the layer-streamed and head-range calls
# ---------------------------------------------------------------------------------------
# kvx_stream and kvx_stream_reshard with every layer ready (ready words already raised in
# device or pinned host memory, or none), live epoch words and owned pages, on the row grid or
# a persistent grid capped at 1 ... 152 CTAs; kvx_move_heads between layouts of different head
# counts (narrow head slices included); kvx_reshard between random TP groups.  A call that
# waits on nothing unraised is deterministic, so it is compared like the one-shot calls.

N_LAYERED = 240
LCALLS = ["stream", "move_heads", "reshard", "stream_reshard"]
LCALL_P = [0.4, 0.25, 0.2, 0.15]
GRIDS = [0, 0, 1, 3, 19, 76, 152]
TPS = [1, 2, 4, 8]


@dataclass
class LCase:
    k: int
    dtype: str
    L: int
    D: int
    kvp: int
    call: str
    op: str
    flags: Optional[int]
    defaults: tuple
    heads: tuple             # (source kv_heads, destination kv_heads) of every pool
    src: Optional[Side]      # a kind and slot count shared by every source pool
    dst: Optional[Side]
    s: np.ndarray
    d: np.ndarray
    plant: str
    h0: int = 0              # move_heads: the head range
    g0: int = 0
    nh: int = 0
    tp: tuple = (1, 1)       # reshard: (P group size, D group size)
    H: int = 0               # reshard: the kv heads the TP groups shard
    ctl: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return len(self.s) if self.op != "scatter" else len(self.d)

    @property
    def check_dup(self) -> bool:
        return bool(self.defaults[0]) if self.flags is None else bool(self.flags & CHECK_DUP)


def _shard_heads(heads, t):
    return heads // t if t <= heads else 1


def draw_layered(k: int) -> LCase:
    g = np.random.Generator(np.random.PCG64(51000 + k))
    dtype = str(g.choice(["fp8", "fp16", "bf16"]))
    e = inputs.ELEM_BYTES[dtype]
    call = str(g.choice(LCALLS, p=LCALL_P))
    # whole 16-byte head vectors, except for the head-range move, which also takes narrow ones
    Ds = [8, 16, 24, 36, 64, 100, 128] if call == "move_heads" else \
        [d for d in (8, 16, 24, 32, 64, 128) if d * e % 16 == 0]
    D = int(g.choice(Ds))
    L = int(g.choice([1, 2, 3, 5]))
    kvp = 1 if g.random() < 0.25 else 2
    op = str(g.choice(["gather", "scatter", "transfer"])) if call in ("stream", "move_heads") \
        else "transfer"
    flags = [None, 0, 1, 2, 4, 1 | 2, 1 | 4][int(g.integers(0, 7))]
    defaults = (int(g.integers(0, 2)), int(g.integers(0, 3)), 0)
    tp = (1, 1)
    h0 = g0 = nh = 0
    if call in ("reshard", "stream_reshard"):
        H = int(g.choice([1, 2, 4, 8]))
        tp = (int(g.choice(TPS)), int(g.choice(TPS)))
        heads = (_shard_heads(H, tp[0]), _shard_heads(H, tp[1]))
        pools = tp[0] + tp[1]
    elif call == "move_heads":
        heads = (int(g.integers(1, 9)), int(g.integers(1, 9)))
        nh = int(g.integers(1, min(heads) + 1)) if op == "transfer" else \
            int(g.integers(1, (heads[0] if op == "gather" else heads[1]) + 1))
        h0 = int(g.integers(0, heads[0] - nh + 1)) if op != "scatter" else 0
        g0 = int(g.integers(0, heads[1] - nh + 1)) if op != "gather" else 0
        pools = 2
    else:
        H = int(g.choice([1, 2, 4, 8]))
        heads = (H, H)
        pools = 2
    R = max(heads) * D * e
    cap_slots = max(64, (POOL_CAP // pools) // (kvp * L * R))
    bucket = g.choice(["zero", "tiny", "small", "mid", "large"], p=[0.03, 0.17, 0.3, 0.3, 0.2])
    n = {"zero": 0, "tiny": int(g.integers(1, 17)), "small": int(g.integers(17, 513)),
         "mid": int(g.integers(513, 2100)), "large": int(g.integers(2100, 5000))}[bucket]
    n = min(n, cap_slots // 2 - 8)
    num = int(min(cap_slots, max(64, int(n * g.uniform(2.0, 4.0)) + 16)))
    num -= num % 16
    src = Side(str(g.choice(KINDS)), num, 16) if op != "scatter" else None
    dst = Side(str(g.choice(KINDS)), num, int(g.choice([1, 4, 16]))) if op != "gather" else None
    if src is not None and src.kind != "hnd":
        src.ps = 1
    if dst is not None and dst.kind != "hnd":
        dst.ps = 1
    c = LCase(k, dtype, L, D, kvp, call, op, flags, defaults, heads, src, dst,
              np.zeros(0, np.int32), np.zeros(0, np.int32), "none", h0, g0, nh, tp,
              H if call in ("reshard", "stream_reshard") else 0)
    if src is not None:
        c.s = _slots(g, n, num, distinct=g.random() < 0.85)
    if dst is not None:
        c.d = _slots(g, n, num)
    if call in ("stream", "stream_reshard"):
        c.ctl = dict(ready=str(g.choice(["none", "device", "pinned"])),
                     ready_value=int(g.integers(1, 6)),
                     epoch=str(g.choice(["none", "device", "pinned"])),
                     epoch_value=int(g.integers(0, 1000)),
                     owners=str(g.choice(["none", "device"])) if dst is not None else "none",
                     epoch_page=int(g.choice([1, 16, 64])),
                     done=bool(g.random() < 0.5),
                     max_ctas=int(g.choice(GRIDS)))
    if n > 0:
        u = g.random()
        if u < 0.15:
            c.plant = "oor"
        elif u < 0.5 and c.check_dup and dst is not None and n >= 2:
            c.plant = "dup"
    _plant(g, c)
    return c


def test_fuzz_layered_cases_draw():
    """Every layered case draws well formed: streamed and reshard cases on whole 16-byte head
    vectors, head ranges inside both layouts, distinct destination slots unless a duplicate is
    planted under the check."""
    calls = set()
    for k in range(N_LAYERED):
        c = draw_layered(k)
        calls.add(c.call)
        e = inputs.ELEM_BYTES[c.dtype]
        if c.call != "move_heads":
            assert c.D * e % 16 == 0
        else:
            if c.op != "scatter":
                assert 0 <= c.h0 and c.h0 + c.nh <= c.heads[0]
            if c.op != "gather":
                assert 0 <= c.g0 and c.g0 + c.nh <= c.heads[1]
        if c.dst is not None and c.plant != "dup":
            inr = c.d[(c.d >= 0) & (c.d < c.dst.num)]
            assert len(np.unique(inr)) == len(inr), k
        for side in (c.src, c.dst):
            if side is not None:
                assert side.num % side.ps == 0
    assert calls == set(LCALLS)


@pytest.mark.gpu
@pytest.mark.parametrize("k", range(N_LAYERED))
def test_fuzz_layered_case(k):
    torch = pytest.importorskip("torch")
    from disaggregated_paged_kv_gb300 import kvx

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    c = draw_layered(k)
    g = np.random.Generator(np.random.PCG64(61000 + k))
    n, e = c.n, inputs.ELEM_BYTES[c.dtype]
    P = c.kvp * c.L

    def mirror(side, H, fill, salt):
        return hz.make_mirror(side.kind, c.L, H, c.D, c.dtype, side.num, side.ps, fill,
                              g if fill == "normal" else None, salt=salt, kvp=c.kvp)

    resh = c.call in ("reshard", "stream_reshard")
    n_src = c.tp[0] if resh else (1 if c.src else 0)
    n_dst = c.tp[1] if resh else (1 if c.dst else 0)
    srcs = [mirror(c.src, c.heads[0], "normal", 0).to_device() for _ in range(n_src)]
    dsts = [mirror(c.dst, c.heads[1], "sentinel", 5 + r).to_device() for r in range(n_dst)]
    exps = [mirror(c.dst, c.heads[1], "sentinel", 5 + r) for r in range(n_dst)]
    rows = c.nh if c.call == "move_heads" else c.heads[0] if c.op != "scatter" else c.heads[1]
    uses_buf = c.op != "transfer"
    buf_n = P * n * rows * c.D * e if uses_buf else 0
    buf = exp_buf = bufp = None
    if uses_buf:
        raw = g.integers(0, 256, 2 * hz.GUARD + max(16, buf_n), dtype=np.uint8)
        buf = torch.from_numpy(raw).cuda()
        exp_buf = raw.copy()
        bufp = hz.GUARD + buf.data_ptr()
    body = exp_buf[hz.GUARD:hz.GUARD + max(16, buf_n)] if uses_buf else None
    parts = kvx.tp_plan(c.H, c.tp[0], c.tp[1]) if resh else []

    # the oracle's result.  A planted repeat (always under the check) must fail with nothing
    # moved: the oracle's head-range and reshard moves have no duplicate check, so that case
    # expects untouched destinations without running them.
    op_code = OP[c.op]
    if c.plant == "dup":
        rc = kvx.ERR_DUPLICATE_DST
    elif resh:
        rc = oracle.reshard([hz.oracle_pool(m) for m in srcs], c.s,
                            [hz.oracle_pool(m) for m in exps], c.d, parts, n)[0]
    elif c.call == "move_heads":
        sp = hz.oracle_pool(srcs[0]) if srcs else None
        dp = hz.oracle_pool(exps[0]) if dsts else None
        rc, out, _ = oracle.move_heads(op_code, sp, c.s if len(c.s) else None, c.h0, dp,
                                       c.d if len(c.d) else None, c.g0, c.nh, n,
                                       buf=body if c.op == "scatter" else None)
        if c.op == "gather" and rc == oracle.OK and n:
            exp_buf[hz.GUARD:hz.GUARD + buf_n] = out[:buf_n]
    elif c.op == "gather":
        rc, out, _ = oracle.gather(hz.oracle_pool(srcs[0]), c.s)
        if rc == oracle.OK and n:
            exp_buf[hz.GUARD:hz.GUARD + buf_n] = out
    elif c.op == "scatter":
        rc = oracle.scatter(hz.oracle_pool(exps[0]), c.d, body)[0]
    else:
        rc = oracle.transfer(hz.oracle_pool(srcs[0]), c.s, hz.oracle_pool(exps[0]), c.d)[0]
    if n == 0:
        rc = kvx.OK

    if c.flags is None:
        kvx.set_check_duplicates(bool(c.defaults[0]))
        kvx.set_copy_engine(c.defaults[1])
    keep = []
    try:
        sls = [hz.kvx_layout(m) for m in srcs]
        dls = [hz.kvx_layout(m) for m in dsts]
        s_d = hz.dev_i32(c.s) if len(c.s) else None
        d_d = hz.dev_i32(c.d) if len(c.d) else None
        ws = hz.workspace(n)
        f = c.flags
        streamed = c.call in ("stream", "stream_reshard")
        st = hz.status(4 if streamed else 1)
        kw = {}
        if streamed:
            ct = c.ctl

            def word(where, values):
                t = torch.tensor(values, dtype=torch.int32)
                t = t.cuda() if where == "device" else t.pin_memory()
                keep.append(t)
                return t

            if ct["ready"] != "none":
                kw["layer_ready"] = word(ct["ready"], [ct["ready_value"]] * c.L)
                kw["ready_value"] = ct["ready_value"]
            if ct["epoch"] != "none":
                kw["epoch_word"] = word(ct["epoch"], [ct["epoch_value"]])
            kw["epoch"] = ct["epoch_value"]
            if ct["owners"] != "none":
                pages = -(-c.dst.num // ct["epoch_page"])
                kw["dst_page_epochs"] = word("device", [ct["epoch_value"]] * pages)
                kw["epoch_page"] = ct["epoch_page"]
            if ct["done"]:
                kw["host_done"] = word("pinned", [0])
            kw["max_ctas"] = ct["max_ctas"]
            kw["wait_ns"] = 2_000_000_000
        if c.call == "stream":
            kvx.stream(op_code, sls[0] if sls else None, s_d, dls[0] if dls else None, d_d, n,
                       bufp, ws, st, buf_bytes=buf_n, flags=f, **kw)
        elif c.call == "stream_reshard":
            kvx.stream_reshard(sls, s_d, dls, d_d, parts, n, ws, st, flags=f, **kw)
        elif c.call == "reshard":
            kvx.reshard(sls, s_d, dls, d_d, parts, n, ws, st, flags=f)
        else:
            kvx.move_heads(op_code, sls[0] if sls else None, s_d, c.h0, dls[0] if dls else None,
                           d_d, c.g0, c.nh, n, bufp, ws, st, buf_bytes=buf_n, flags=f)
        torch.cuda.synchronize()
        got = st.cpu().numpy().tolist()
    finally:
        kvx.set_check_duplicates(False)
        kvx.set_copy_engine(kvx.ENGINE_AUTO)

    what = f"case {k}: {c.call} {c.op} {c.dtype} L{c.L} D{c.D} heads {c.heads} kvp{c.kvp} " \
           f"n{n} flags {c.flags} plant {c.plant} tp {c.tp} heads {c.h0}/{c.g0}/{c.nh} " \
           f"src {c.src} dst {c.dst} ctl {c.ctl}"
    if streamed:
        assert got[0] == rc and got[3] == 1, (got, rc, what)
        assert got[1] == (0 if rc == kvx.OK else c.L), (got, rc, what)
        if c.ctl.get("done"):
            assert int(kw["host_done"][0]) == 1, what
    else:
        assert got == [rc], (got, rc, what)
    for r, (m, x) in enumerate(zip(dsts, exps)):
        hz.assert_same_bytes(m.readback(), x.host, f"{what}: destination pool {r}")
    for r, m in enumerate(srcs):
        hz.assert_same_bytes(m.readback(), m.host, f"{what}: source pool {r}")
    if uses_buf:
        hz.assert_same_bytes(buf.cpu().numpy(), exp_buf, what + ": buffer")
