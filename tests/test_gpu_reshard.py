"""kvx_reshard / kvx_tp_plan -- a whole reshard between the pools of two tensor-parallel groups
in one call -- against the oracle's kvxo_reshard, through the C ABI (GPU).

Every case compares every destination pool (guard bands included) byte for byte with the
oracle on the same seeded inputs, and checks that no source pool changed.  Plans come from
kvx_tp_plan (checked against the oracle's tp_slice on the CPU); the cases cover merges
(several P shards into one D shard), splits, replicated heads, the layout kinds on either
side, rows over 2 KiB, layouts whose planes are not evenly spaced, one- and multi-tile slot
lists, grids of several rows, and the refusals that leave every pool untouched.
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


def _rng(k):
    return np.random.Generator(np.random.PCG64(9100 + k))


def _shard(heads, t, r):
    return heads // t if t <= heads else 1


class Groups:
    """The P group's pools (filled) and the D group's pools (sentinel), device and host."""

    def __init__(self, heads, p_tp, d_tp, src_kind="hnd", dst_kind="planes", layers=2, d=128,
                 dt="bf16", num_slots=2048, kvp=2, seed=0):
        g = _rng(seed)
        ps = lambda kind: 16 if kind == "hnd" else 1
        self.p = [hz.make_mirror(src_kind, layers, _shard(heads, p_tp, r), d, dt, num_slots,
                                 ps(src_kind), "normal", g, kvp=kvp).to_device()
                  for r in range(p_tp)]
        self.d = [hz.make_mirror(dst_kind, layers, _shard(heads, d_tp, r), d, dt, num_slots,
                                 ps(dst_kind), "sentinel", salt=r, kvp=kvp).to_device()
                  for r in range(d_tp)]
        self.d_exp = [hz.make_mirror(dst_kind, layers, _shard(heads, d_tp, r), d, dt, num_slots,
                                     ps(dst_kind), "sentinel", salt=r, kvp=kvp)
                      for r in range(d_tp)]
        self.parts = kvx.tp_plan(heads, p_tp, d_tp)
        self.num_slots = num_slots

    def expect(self, s, d, n, parts=None):
        rc, _ = oracle.reshard([hz.oracle_pool(m) for m in self.p], s,
                               [hz.oracle_pool(m) for m in self.d_exp], d,
                               parts if parts is not None else self.parts, n)
        return rc

    def run(self, s, d, n, parts=None, ws_tokens=None):
        st = hz.status()
        kvx.reshard([hz.kvx_layout(m) for m in self.p], hz.dev_i32(s),
                    [hz.kvx_layout(m) for m in self.d], hz.dev_i32(d),
                    parts if parts is not None else self.parts, n,
                    hz.workspace(ws_tokens or n), st)
        torch.cuda.synchronize()
        return int(st.item())

    def check(self, what):
        for r, (m, e) in enumerate(zip(self.d, self.d_exp)):
            hz.assert_same_bytes(m.readback(), e.host, f"{what}: D rank {r}")
        for r, m in enumerate(self.p):
            hz.assert_same_bytes(m.readback(), m.host, f"{what}: P rank {r} (source)")


def _slots(k, n, num):
    return inputs.distinct_slots(_rng(k), n, num)


PLANS = [(1, 2), (2, 1), (4, 2), (2, 4), (8, 1), (1, 8), (8, 8), (16, 2), (2, 16)]


@pytest.mark.parametrize("p_tp,d_tp", PLANS)
def test_reshard_tp_plans(p_tp, d_tp):
    """8 kv heads x 128 bf16: HND P pools (page 16) -> per-plane token-row D pools, 1500
    random tokens."""
    gr = Groups(8, p_tp, d_tp, seed=p_tp * 100 + d_tp)
    n = 1500
    s, d = _slots(1, n, gr.num_slots), _slots(2, n, gr.num_slots)
    assert gr.expect(s, d, n) == oracle.OK
    assert gr.run(s, d, n) == kvx.OK
    gr.check(f"P TP {p_tp} -> D TP {d_tp}")


KINDS = ["planes", "slot_major", "hnd", "planes_separate", "planes_rotated"]


@pytest.mark.parametrize("src_kind", KINDS)
@pytest.mark.parametrize("dst_kind", KINDS)
def test_reshard_layout_kinds(src_kind, dst_kind):
    """P TP 4 -> D TP 2 (merges of 512-byte pieces) between every pair of layout kinds,
    including per-plane pointer tables that are not a constant stride apart."""
    gr = Groups(8, 4, 2, src_kind, dst_kind, layers=3, seed=len(src_kind) * 10 + len(dst_kind))
    n = 999
    s, d = _slots(3, n, gr.num_slots), _slots(4, n, gr.num_slots)
    assert gr.expect(s, d, n) == oracle.OK
    assert gr.run(s, d, n) == kvx.OK
    gr.check(f"{src_kind} -> {dst_kind}")


@pytest.mark.parametrize("n", [1, 2, 31, 2048, 2049, 4100])
def test_reshard_token_counts(n):
    """One token, a ragged warp, exactly one planner tile, and two or three tiles."""
    gr = Groups(8, 8, 2, "planes", "hnd", num_slots=8192, seed=n)
    s, d = _slots(5 + n, n, gr.num_slots), _slots(6 + n, n, gr.num_slots)
    assert gr.expect(s, d, n) == oracle.OK
    assert gr.run(s, d, n) == kvx.OK
    gr.check(f"n={n}")


def test_reshard_zero_tokens():
    gr = Groups(8, 2, 1, seed=77)
    st = hz.status()
    kvx.reshard([hz.kvx_layout(m) for m in gr.p], None, [hz.kvx_layout(m) for m in gr.d], None,
                gr.parts, 0, None, st, ws_bytes=0)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    gr.check("n=0")


def test_reshard_long_rows():
    """Pieces over 2 KiB (4 heads of 1 KiB: fp16 head_dim 512) take the multi-pass instance."""
    gr = Groups(8, 1, 2, "slot_major", "planes", layers=2, d=512, dt="fp16", num_slots=1024,
                seed=5)
    n = 700
    s, d = _slots(7, n, gr.num_slots), _slots(8, n, gr.num_slots)
    assert gr.expect(s, d, n) == oracle.OK
    assert gr.run(s, d, n) == kvx.OK
    gr.check("4 KiB pieces")


def test_reshard_several_grid_rows():
    """40,000 tokens of 256-byte pieces: 5,000 token groups, so the grid has two rows."""
    gr = Groups(2, 2, 1, "planes", "planes", layers=1, d=128, num_slots=40960, seed=6)
    n = 40000
    s, d = _slots(9, n, gr.num_slots), _slots(10, n, gr.num_slots)
    assert gr.expect(s, d, n) == oracle.OK
    assert gr.run(s, d, n) == kvx.OK
    gr.check("two grid rows")


def test_reshard_mla_latent():
    """MLA (one latent plane per layer, one kv head replicated on every rank): P TP 2 -> D TP 4
    gives every D rank the latent rows from P rank 0."""
    gr = Groups(1, 2, 4, "planes", "hnd", layers=3, d=576, dt="bf16", kvp=1, seed=8)
    assert gr.parts == [(0, r, 0, 0, 1) for r in range(4)]
    n = 500
    s, d = _slots(11, n, gr.num_slots), _slots(12, n, gr.num_slots)
    assert gr.expect(s, d, n) == oracle.OK
    assert gr.run(s, d, n) == kvx.OK
    gr.check("MLA latent")


def test_reshard_fp8():
    gr = Groups(8, 2, 4, "hnd", "slot_major", dt="fp8", seed=9)
    n = 1200
    s, d = _slots(13, n, gr.num_slots), _slots(14, n, gr.num_slots)
    assert gr.expect(s, d, n) == oracle.OK
    assert gr.run(s, d, n) == kvx.OK
    gr.check("fp8")


def test_reshard_partial_plan_touches_only_its_heads():
    """A hand-made plan that fills only some heads of the D shards: the other heads keep their
    bytes (the oracle's expected pools are the sentinel pools with those parts applied)."""
    gr = Groups(8, 4, 1, "planes", "planes", seed=10)
    parts = [(2, 0, 0, 4, 2), (0, 0, 0, 1, 2)]
    n = 800
    s, d = _slots(15, n, gr.num_slots), _slots(16, n, gr.num_slots)
    assert gr.expect(s, d, n, parts) == oracle.OK
    assert gr.run(s, d, n, parts) == kvx.OK
    gr.check("partial plan")


@pytest.mark.parametrize("where", ["src", "dst", "negative"])
@pytest.mark.parametrize("n", [600, 3000])
def test_reshard_out_of_range_moves_nothing(where, n):
    gr = Groups(8, 4, 2, num_slots=4096, seed=11)
    s, d = _slots(17, n, gr.num_slots), _slots(18, n, gr.num_slots)
    if where == "src":
        s[n // 3] = gr.num_slots
    elif where == "dst":
        d[n - 1] = gr.num_slots + 5
    else:
        d[0] = -1
    assert gr.expect(s, d, n) == oracle.ERR_OUT_OF_RANGE
    assert gr.run(s, d, n) == kvx.ERR_OUT_OF_RANGE
    gr.check(f"out of range ({where})")


def test_reshard_duplicate_destination_refused():
    gr = Groups(8, 2, 2, seed=12)
    n = 900
    s, d = _slots(19, n, gr.num_slots), _slots(20, n, gr.num_slots)
    d[700] = d[3]
    kvx.set_check_duplicates(1)
    try:
        assert gr.run(s, d, n) == kvx.ERR_DUPLICATE_DST
    finally:
        kvx.set_check_duplicates(0)
    gr.check("duplicate destination")


def test_reshard_equals_pairwise_move_heads():
    """The one-call reshard leaves the D pools exactly as the pair-by-pair kvx_move_heads
    transfers of the same plan do (both on the GPU, then both against the oracle)."""
    gr = Groups(8, 8, 1, seed=13)
    n = 1000
    s, d = _slots(21, n, gr.num_slots), _slots(22, n, gr.num_slots)
    assert gr.run(s, d, n) == kvx.OK
    one_call = [m.readback() for m in gr.d]
    for m in gr.d:
        m.dev.copy_(torch.from_numpy(m.host))
    s_d, d_d, ws = hz.dev_i32(s), hz.dev_i32(d), hz.workspace(n)
    for pr, dr, h0, g0, nh in gr.parts:
        st = hz.status()
        kvx.move_heads(kvx.OP_TRANSFER, hz.kvx_layout(gr.p[pr]), s_d, h0, hz.kvx_layout(gr.d[dr]),
                       d_d, g0, nh, n, None, ws, st, buf_bytes=0)
        torch.cuda.synchronize()
        assert int(st.item()) == kvx.OK
    for a, m in zip(one_call, gr.d):
        hz.assert_same_bytes(a, m.readback(), "one call vs pair by pair")
    assert gr.expect(s, d, n) == oracle.OK
    for a, e in zip(one_call, gr.d_exp):
        hz.assert_same_bytes(a, e.host, "one call vs oracle")
