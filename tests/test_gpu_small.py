"""One-shot requests of up to 512 tokens (the one-launch path whose every CTA checks every
index), against the oracle (GPU).

Token counts on both sides of the 512-token boundary (the planner path takes over at 513), all
three ops between token-row and HND layouts, a bad index at the first, a middle and the last
position of either list (nothing may move, whichever CTA holds the bad token's rows), the
status word and kvx_submit's pinned host status, and two requests back to back on one stream
(the second reads what the first wrote).
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SH = dict(L=3, H=2, D=64, dtype="fp16")  # 256-byte rows


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


def _rng(k):
    return np.random.Generator(np.random.PCG64(14000 + k))


def _pool(kind, fill, g=None, num=2048, salt=0, D=SH["D"]):
    return hz.make_mirror(kind, SH["L"], SH["H"], D, SH["dtype"], num, 16 if kind == "hnd" else 1,
                          fill, g, salt=salt)


@pytest.mark.parametrize("n", [1, 100, 511, 512, 513, 700])
@pytest.mark.parametrize("kinds", [("planes", "hnd"), ("hnd", "slot_major")])
def test_transfer_around_the_boundary(n, kinds):
    g = _rng(n + len(kinds[0]))
    src = _pool(kinds[0], "normal", g).to_device()
    dst = _pool(kinds[1], "sentinel", salt=3).to_device()
    exp = _pool(kinds[1], "sentinel", salt=3)
    s = inputs.distinct_slots(g, n, src.num_slots)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == oracle.OK
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"n={n} {kinds}")
    hz.assert_same_bytes(src.readback(), src.host, "source")


@pytest.mark.parametrize("D", [64, 576, 1024])  # 256 B, 2304 B (two passes) and 4 KiB rows
@pytest.mark.parametrize("n", [37, 512])
def test_gather_scatter_small(D, n):
    g = _rng(D + n)
    src = _pool("hnd", "normal", g, D=D).to_device()
    s = inputs.distinct_slots(g, n, src.num_slots)
    rc, want, w = oracle.gather(hz.oracle_pool(src), s)
    assert rc == oracle.OK
    buf = hz.make_mirror("buffer", SH["L"], SH["H"], D, SH["dtype"], n_tokens=n,
                         fill="sentinel").to_device()
    st = hz.status()
    kvx.gather(hz.kvx_layout(src), hz.dev_i32(s), n, hz.GUARD + buf.dev.data_ptr(),
               hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    exp = buf.host.copy()
    exp[hz.GUARD:hz.GUARD + w] = want[:w]
    hz.assert_same_bytes(buf.readback(), exp, f"gather D={D} n={n}")
    dst = _pool("planes", "sentinel", salt=5, D=D).to_device()
    exp_d = _pool("planes", "sentinel", salt=5, D=D)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    assert oracle.scatter(hz.oracle_pool(exp_d), d, want[:w])[0] == oracle.OK
    st = hz.status()
    kvx.scatter(hz.kvx_layout(dst), hz.dev_i32(d), n, hz.GUARD + buf.dev.data_ptr(),
                hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp_d.host, f"scatter D={D} n={n}")


@pytest.mark.parametrize("where", [0, 250, 511])
@pytest.mark.parametrize("side", ["src", "dst"])
@pytest.mark.parametrize("bad", [-1, 2048, 2 ** 31 - 1])
def test_bad_index_moves_nothing(where, side, bad):
    n = 512
    g = _rng(where + len(side))
    src = _pool("planes", "normal", g).to_device()
    dst = _pool("planes", "sentinel", salt=7).to_device()
    s = inputs.distinct_slots(g, n, src.num_slots)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    (s if side == "src" else d)[where] = bad
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(dst), d)[0] == oracle.ERR_OUT_OF_RANGE
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(dst.readback(), dst.host, "nothing moved")


@pytest.mark.parametrize("bad", [False, True])
def test_submit_small(bad):
    n = 300
    g = _rng(31 + bad)
    src = _pool("planes", "normal", g).to_device()
    dst = _pool("planes", "sentinel", salt=9).to_device()
    exp = _pool("planes", "sentinel", salt=9)
    s = inputs.distinct_slots(g, n, src.num_slots)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    if bad:
        d[123] = -5
    rc = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0]
    hs = torch.from_numpy(s).pin_memory()
    hd = torch.from_numpy(d).pin_memory()
    hst = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    kvx.submit(kvx.OP_TRANSFER, hz.kvx_layout(src), hs, hz.kvx_layout(dst), hd, n, None,
               hz.workspace(n), hst, buf_bytes=0)
    torch.cuda.synchronize()
    assert int(hst[0]) == (kvx.ERR_OUT_OF_RANGE if bad else kvx.OK)
    assert rc == (oracle.ERR_OUT_OF_RANGE if bad else oracle.OK)
    hz.assert_same_bytes(dst.readback(), exp.host, "submit")


def test_back_to_back_reads_what_the_last_call_wrote():
    """Scatter into a pool, then gather the same slots from it on the same stream with no
    synchronisation in between: the gather must see the scattered rows."""
    n = 400
    g = _rng(55)
    pool = _pool("planes", "sentinel", salt=11).to_device()
    R, P = pool.R, pool.P
    data = torch.from_numpy(inputs.normal_bits(g, P * n * R // 2, "fp16").view(np.uint8)).cuda()
    slots = hz.dev_i32(inputs.distinct_slots(g, n, pool.num_slots))
    out = torch.empty_like(data)
    lay = hz.kvx_layout(pool)
    st1, st2 = hz.status(), hz.status()
    for _ in range(20):
        out.fill_(0)
        kvx.scatter(lay, slots, n, data, hz.workspace(n), st1)
        kvx.gather(lay, slots, n, out, hz.workspace(n), st2)
    torch.cuda.synchronize()
    assert int(st1.item()) == kvx.OK and int(st2.item()) == kvx.OK
    assert torch.equal(out, data)
