"""8-byte-aligned rows of every length, against the oracle (GPU).

Rows that start on 8-byte but not always 16-byte boundaries -- R = 8 mod 16 (so the phase of a
row changes from slot to slot), or plane bases 8 bytes off a 16-byte boundary -- move with
8-byte accesses (the narrow row kernel).  Row lengths of 3 to 259 words, buffers on either
side, token-row layouts of both kinds, offset planes on either or both sides, and a bad slot
that must stop the whole request; every case compares the whole destination, guard bands
included, with the oracle.
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


# row bytes: 3, 5, 7, 9, 15, 25 (head_dim 100 fp16), 33, 129, 257 and 259 words
ROWS = [24, 40, 56, 72, 120, 200, 264, 1032, 2056, 2072]
L = 2


def _rng(k):
    return np.random.Generator(np.random.PCG64(12000 + k))


def _mirror(kind, R, fill, g=None, num=1024, salt=0, n_tokens=0, dt="fp16"):
    e = 2 if dt == "fp16" else 1
    return hz.make_mirror(kind, L, 1, R // e, dt, num, 1, fill, g, salt=salt, n_tokens=n_tokens)


@pytest.mark.parametrize("R", ROWS)
@pytest.mark.parametrize("kinds", [("planes", "planes"), ("planes", "slot_major"),
                                   ("slot_major", "planes")])
def test_transfer_rows(R, kinds):
    n = 700
    g = _rng(R + len(kinds[0]) + 3 * len(kinds[1]))
    src = _mirror(kinds[0], R, "normal", g).to_device()
    dst = _mirror(kinds[1], R, "sentinel", salt=4).to_device()
    exp = _mirror(kinds[1], R, "sentinel", salt=4)
    s = inputs.distinct_slots(g, n, src.num_slots)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == oracle.OK
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"R={R} {kinds}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


@pytest.mark.parametrize("R", ROWS)
@pytest.mark.parametrize("dt", ["fp16", "fp8"])
def test_gather_scatter_rows(R, dt):
    n = 333
    g = _rng(7 * R + len(dt))
    src = _mirror("planes", R, "normal", g, dt=dt).to_device()
    s = inputs.distinct_slots(g, n, src.num_slots)
    rc, want, w = oracle.gather(hz.oracle_pool(src), s)
    assert rc == oracle.OK
    buf = _mirror("buffer", R, "sentinel", n_tokens=n, dt=dt).to_device()
    st = hz.status()
    kvx.gather(hz.kvx_layout(src), hz.dev_i32(s), n, hz.GUARD + buf.dev.data_ptr(),
               hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    exp = buf.host.copy()
    exp[hz.GUARD:hz.GUARD + w] = want[:w]
    hz.assert_same_bytes(buf.readback(), exp, f"gather R={R}")

    dst = _mirror("slot_major", R, "sentinel", salt=6, dt=dt).to_device()
    exp_dst = _mirror("slot_major", R, "sentinel", salt=6, dt=dt)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    assert oracle.scatter(hz.oracle_pool(exp_dst), d, want[:w])[0] == oracle.OK
    st = hz.status()
    kvx.scatter(hz.kvx_layout(dst), hz.dev_i32(d), n, hz.GUARD + buf.dev.data_ptr(),
                hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp_dst.host, f"scatter R={R}")


class OffsetPool:
    """A per-plane token-row pool whose planes start 8 bytes past a 16-byte boundary, so every
    row of a 16-byte-multiple R is on phase 1: host bytes (guard bands included) and device
    copy, described alike to the oracle and to libkvx."""

    def __init__(self, R, num, fill, g=None, salt=0):
        self.R, self.num, self.P = R, num, 2 * L
        body = self.P * num * R
        self.host = np.empty(2 * hz.GUARD + 8 + body, dtype=np.uint8)
        self.host[:] = inputs.sentinel_bits(len(self.host) // 2, "fp16", salt).view(np.uint8)
        if fill == "normal":
            self.host[hz.GUARD + 8:hz.GUARD + 8 + body] = \
                inputs.normal_bits(g, body // 2, "fp16").view(np.uint8)
        self.dev = torch.from_numpy(self.host).to("cuda")

    def oracle_pool(self):
        planes = [(self.host, hz.GUARD + 8 + p * self.num * self.R) for p in range(self.P)]
        return oracle.Pool(L, 1, self.R // 2, 2, oracle.TOKEN_ROWS, self.num, planes, self.R)

    def layout(self):
        return kvx.Layout(L, 1, self.R // 2, kvx.F16, self.num,
                          base=int(self.dev.data_ptr()) + hz.GUARD + 8,
                          plane_stride=self.num * self.R, keepalive=self.dev)


@pytest.mark.parametrize("R", [32, 64, 200, 1024])
@pytest.mark.parametrize("which", ["src", "dst", "both"])
def test_offset_planes(R, which):
    """Plane bases 8 bytes off: with R a multiple of 16 every row of that side is on phase 1
    (against a phase-0 side), and 200-byte rows mix both phases."""
    n, num = 500, 1024
    g = _rng(R + len(which))
    if which in ("src", "both"):
        src = OffsetPool(R, num, "normal", g)
        s_or, s_l, s_host, s_dev = src.oracle_pool(), src.layout(), src.host, src.dev
    else:
        m = _mirror("planes", R, "normal", g, num=num).to_device()
        s_or, s_l, s_host, s_dev = hz.oracle_pool(m), hz.kvx_layout(m), m.host, m.dev
    if which in ("dst", "both"):
        dst = OffsetPool(R, num, "sentinel", salt=3)
        exp = OffsetPool(R, num, "sentinel", salt=3)
        d_l, d_dev, e_or, e_host = dst.layout(), dst.dev, exp.oracle_pool(), exp.host
    else:
        dm = _mirror("planes", R, "sentinel", num=num, salt=3).to_device()
        em = _mirror("planes", R, "sentinel", num=num, salt=3)
        d_l, d_dev, e_or, e_host = hz.kvx_layout(dm), dm.dev, hz.oracle_pool(em), em.host
    s = inputs.distinct_slots(g, n, num)
    d = inputs.distinct_slots(g, n, num)
    assert oracle.transfer(s_or, s, e_or, d)[0] == oracle.OK
    st = hz.status()
    kvx.transfer(s_l, hz.dev_i32(s), d_l, hz.dev_i32(d), n, hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(d_dev.cpu().numpy(), e_host, f"offset {which} R={R}")
    hz.assert_same_bytes(s_dev.cpu().numpy(), s_host, "source")


@pytest.mark.parametrize("where", ["src", "dst"])
def test_rows_out_of_range_moves_nothing(where):
    n = 900
    g = _rng(99)
    src = _mirror("planes", 200, "normal", g).to_device()
    dst = _mirror("planes", 200, "sentinel", salt=8).to_device()
    s = inputs.distinct_slots(g, n, src.num_slots)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    (s if where == "src" else d)[n // 2] = -3
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(dst.readback(), dst.host, "nothing moved")
