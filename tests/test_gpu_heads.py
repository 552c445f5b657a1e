"""kvx_move_heads / kvx_tp_slice -- moves of kv-head ranges between layouts whose kv_heads
differ (heterogeneous tensor parallelism) -- against the oracle, through the C ABI (GPU).

Every case compares the whole destination (pool or buffer, guard bands included) byte for
byte with the oracle's kvxo_move_heads on the same seeded inputs, on the three copy paths
(planner + row kernel, one-launch fused, planner + bulk engine).  The resharding cases move a
model's KV between TP groups of different sizes with the plan kvx_tp_slice computes.
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

L, D, DT = 3, 64, "fp16"  # 128-byte head vectors
KINDS = ["planes", "slot_major", "hnd"]
OPS = {"gather": kvx.OP_GATHER, "scatter": kvx.OP_SCATTER, "transfer": kvx.OP_TRANSFER}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


@pytest.fixture(params=["default", "fused", "planned_bulk"])
def path(request):
    fused, engine = {"default": (0, kvx.ENGINE_AUTO), "fused": (8192, kvx.ENGINE_AUTO),
                     "planned_bulk": (0, kvx.ENGINE_BULK)}[request.param]
    kvx.set_fused_max_tokens(fused)
    kvx.set_copy_engine(engine)
    yield request.param
    kvx.set_fused_max_tokens(0)
    kvx.set_copy_engine(kvx.ENGINE_AUTO)


def _rng(k):
    return np.random.Generator(np.random.PCG64(7000 + k))


def _pool(kind, heads, fill, g=None, num_slots=4096, salt=0, d=D, dt=DT, layers=L):
    return hz.make_mirror(kind, layers, heads, d, dt, num_slots, 16 if kind == "hnd" else 1, fill,
                          g, salt=salt).to_device()


def _host_pool(kind, heads, salt, num_slots=4096, d=D, dt=DT, layers=L):
    return hz.make_mirror(kind, layers, heads, d, dt, num_slots, 16 if kind == "hnd" else 1,
                          "sentinel", salt=salt)


def _slots(k, n, num_slots):
    return inputs.distinct_slots(_rng(k), n, num_slots)


CASES = [  # (src heads, dst heads, src_head0, dst_head0, n_heads)
    (8, 4, 2, 0, 4),
    (4, 8, 0, 4, 4),
    (8, 4, 6, 3, 1),
    (2, 2, 0, 0, 2),
]


@pytest.mark.parametrize("src_kind", KINDS)
@pytest.mark.parametrize("dst_kind", KINDS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: "h%d-%d_%d+%d_%d" % c)
def test_transfer_heads(src_kind, dst_kind, case, path):
    hs, hd, h0, g0, nh = case
    n = 777
    g = _rng(hs * 10 + hd + h0)
    src = _pool(src_kind, hs, "normal", g)
    dst = _pool(dst_kind, hd, "sentinel", salt=3)
    s, d = _slots(1 + h0, n, src.num_slots), _slots(2 + g0, n, dst.num_slots)
    exp = _host_pool(dst_kind, hd, 3)
    rc, _, _ = oracle.move_heads(2, hz.oracle_pool(src), s, h0, hz.oracle_pool(exp), d, g0, nh, n)
    assert rc == oracle.OK
    st = hz.status()
    kvx.move_heads(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), h0, hz.kvx_layout(dst),
                   hz.dev_i32(d), g0, nh, n, None, hz.workspace(n), st, buf_bytes=0)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"heads {case} {src_kind}->{dst_kind}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [1, 2048, 2500])
def test_gather_scatter_heads(kind, n, path):
    g = _rng(n)
    src = _pool(kind, 8, "normal", g)
    s = _slots(10 + n, n, src.num_slots)
    h0, nh = 4, 4
    rc, want, w = oracle.move_heads(0, hz.oracle_pool(src), s, h0, None, None, 0, nh, n)
    assert rc == oracle.OK and w == n * 2 * L * nh * D * 2
    want = want[:w]
    buf = hz.make_mirror("buffer", L, nh, D, DT, n_tokens=n, fill="sentinel").to_device()
    st = hz.status()
    kvx.move_heads(kvx.OP_GATHER, hz.kvx_layout(src), hz.dev_i32(s), h0, None, None, 0, nh, n,
                   hz.GUARD + buf.dev.data_ptr(), hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    exp_buf = buf.host.copy()
    exp_buf[hz.GUARD:hz.GUARD + w] = want
    hz.assert_same_bytes(buf.readback(), exp_buf, f"gather heads {kind} n={n}")

    # scatter those heads into heads [1, 5) of a 6-head pool
    dst = _pool(kind, 6, "sentinel", salt=4)
    d = _slots(20 + n, n, dst.num_slots)
    exp = _host_pool(kind, 6, 4)
    rc, _, _ = oracle.move_heads(1, None, None, 0, hz.oracle_pool(exp), d, 1, nh, n, buf=want)
    assert rc == oracle.OK
    st = hz.status()
    kvx.move_heads(kvx.OP_SCATTER, None, None, 0, hz.kvx_layout(dst), hz.dev_i32(d), 1, nh, n,
                   hz.GUARD + buf.dev.data_ptr(), hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"scatter heads {kind} n={n}")


def test_heads_out_of_range_moves_nothing(path):
    n = 600
    g = _rng(99)
    src = _pool("planes", 8, "normal", g)
    dst = _pool("hnd", 4, "sentinel", salt=6)
    s, d = _slots(31, n, src.num_slots), _slots(32, n, dst.num_slots)
    d[n // 2] = dst.num_slots
    before = dst.readback()
    st = hz.status()
    kvx.move_heads(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), 4, hz.kvx_layout(dst),
                   hz.dev_i32(d), 0, 4, n, None, hz.workspace(n), st, buf_bytes=0)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(dst.readback(), before, "nothing moved")


@pytest.mark.parametrize("p_tp,d_tp", [(1, 2), (2, 1), (4, 2), (2, 4), (8, 8), (16, 4)])
def test_tp_reshard(p_tp, d_tp, path):
    """A model with 8 kv heads (bf16, head_dim 128: 256-byte heads) whose KV sits in the pools
    of a TP group of size p_tp is moved into the pools of a TP group of size d_tp, every
    (P rank, D rank) pair moving the heads kvx_tp_slice assigns it.  Every D pool must equal the
    oracle's result of the same plan, and every D rank must have received each of its heads."""
    heads, dh, dt, layers, n, num = 8, 128, "bf16", 2, 1500, 2048
    per = lambda t: max(1, heads // t)
    g = _rng(p_tp * 100 + d_tp)
    p_pools = [_pool("hnd", per(p_tp), "normal", g, num_slots=num, d=dh, dt=dt, layers=layers)
               for _ in range(p_tp)]
    d_pools = [_pool("planes", per(d_tp), "sentinel", num_slots=num, salt=r, d=dh, dt=dt,
                     layers=layers) for r in range(d_tp)]
    d_exp = [_host_pool("planes", per(d_tp), r, num_slots=num, d=dh, dt=dt, layers=layers)
             for r in range(d_tp)]
    s = _slots(41, n, num)
    d = _slots(42, n, num)
    s_d, d_d, ws = hz.dev_i32(s), hz.dev_i32(d), hz.workspace(n)
    received = [0] * d_tp
    for dr in range(d_tp):
        for pr in range(p_tp):
            sh0, dh0, nh = kvx.tp_slice(heads, p_tp, pr, d_tp, dr)
            assert (oracle.OK, sh0, dh0, nh) == oracle.tp_slice(heads, p_tp, pr, d_tp, dr)
            if nh == 0:
                continue
            received[dr] += nh
            rc, _, _ = oracle.move_heads(2, hz.oracle_pool(p_pools[pr]), s, sh0,
                                         hz.oracle_pool(d_exp[dr]), d, dh0, nh, n)
            assert rc == oracle.OK
            st = hz.status()
            kvx.move_heads(kvx.OP_TRANSFER, hz.kvx_layout(p_pools[pr]), s_d, sh0,
                           hz.kvx_layout(d_pools[dr]), d_d, dh0, nh, n, None, ws, st, buf_bytes=0)
            torch.cuda.synchronize()
            assert int(st.item()) == kvx.OK
    assert received == [per(d_tp)] * d_tp
    for dr in range(d_tp):
        hz.assert_same_bytes(d_pools[dr].readback(), d_exp[dr].host, f"D rank {dr}")
