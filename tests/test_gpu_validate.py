"""One-shot requests of more than one planner tile (2049 tokens and up), against the oracle (GPU).

Up to 8192 tokens one CTA validates the slot lists before the copy: it reads each list's
16-byte-aligned body with vector loads and the up to three elements before and after it one by
one, so the tests shift the lists off 16-byte alignment by 0 to 3 elements and put a bad index
(negative, or one past the pool) at the first element, the last scalar element before the body,
the middle of the body, and the last two elements, on either list: the status must say
KVX_ERR_OUT_OF_RANGE and nothing may move.  Larger requests (32,768 tokens) take the multi-tile
planner.  Valid requests must give the oracle's bytes for every op, including the gather whose
destination is a buffer (no list).
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SH = dict(L=2, H=1, D=64, dtype="fp16")  # 128-byte rows, 4 planes
NUM = 40960


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


def _rng(k):
    return np.random.Generator(np.random.PCG64(15000 + k))


def _pool(kind, fill, g=None, salt=0):
    return hz.make_mirror(kind, SH["L"], SH["H"], SH["D"], SH["dtype"], NUM,
                          16 if kind == "hnd" else 1, fill, g, salt=salt)


def _shifted(a, off):
    """a on the device, starting `off` int32 elements past a 16-byte boundary."""
    t = torch.zeros(len(a) + 4, dtype=torch.int32, device="cuda")
    assert t.data_ptr() % 16 == 0
    t[off: off + len(a)] = torch.from_numpy(np.asarray(a, dtype=np.int32)).cuda()
    return t[off: off + len(a)]


def _run(op, src, s, dst, d, n, buf=None, st=None):
    ws = hz.workspace(n)
    if op == "gather":
        kvx.gather(hz.kvx_layout(src), s, n, hz.GUARD + buf.dev.data_ptr(), ws, st,
                   buf_bytes=n * src.P * src.R)
    elif op == "scatter":
        kvx.scatter(hz.kvx_layout(dst), d, n, hz.GUARD + buf.dev.data_ptr(), ws, st,
                    buf_bytes=n * dst.P * dst.R)
    else:
        kvx.transfer(hz.kvx_layout(src), s, hz.kvx_layout(dst), d, n, ws, st)
    torch.cuda.synchronize()
    return int(st.item())


@pytest.mark.parametrize("offs", [(0, 0), (1, 3), (2, 1), (3, 2)])
@pytest.mark.parametrize("op", ["gather", "scatter", "transfer"])
@pytest.mark.parametrize("n", [2049, 5000, 8192, 32768])
def test_validated_request_matches_oracle(n, op, offs):
    g = _rng(n + 7 * offs[0] + offs[1])
    src = _pool("planes", "normal", g).to_device()
    dst = _pool("hnd", "sentinel", salt=2).to_device()
    exp_dst = _pool("hnd", "sentinel", salt=2)
    s = inputs.distinct_slots(g, n, NUM)
    d = inputs.distinct_slots(g, n, NUM)
    buf = hz.make_mirror("buffer", SH["L"], SH["H"], SH["D"], SH["dtype"], n_tokens=n,
                         fill="normal" if op == "scatter" else "sentinel", g=g).to_device()
    st = hz.status()
    assert _run(op, src, _shifted(s, offs[0]), dst, _shifted(d, offs[1]), n, buf, st) == kvx.OK
    if op == "gather":
        rc, want, w = oracle.gather(hz.oracle_pool(src), s)
        assert rc == oracle.OK
        exp = buf.host.copy()
        exp[hz.GUARD: hz.GUARD + w] = want[:w]
        hz.assert_same_bytes(buf.readback(), exp, f"gather n={n}")
        return
    if op == "scatter":
        body = buf.host[hz.GUARD: hz.GUARD + n * dst.P * dst.R]
        assert oracle.scatter(hz.oracle_pool(exp_dst), d, body)[0] == oracle.OK
    else:
        assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp_dst), d)[0] == oracle.OK
    hz.assert_same_bytes(dst.readback(), exp_dst.host, f"{op} n={n} offs={offs}")


@pytest.mark.parametrize("bad", [-1, NUM])
@pytest.mark.parametrize("side", ["src", "dst"])
@pytest.mark.parametrize("where", ["first", "before_body", "body", "next_to_last", "last"])
@pytest.mark.parametrize("off", [0, 1, 3])
def test_bad_index_moves_nothing(where, side, bad, off):
    n = 5000
    g = _rng(100 + off)
    src = _pool("planes", "normal", g).to_device()
    dst = _pool("planes", "sentinel", salt=4).to_device()
    s = inputs.distinct_slots(g, n, NUM)
    d = inputs.distinct_slots(g, n, NUM)
    head = (4 - off) % 4  # elements before the first 16-byte boundary
    pos = {"first": 0, "before_body": max(0, head - 1), "body": n // 2, "next_to_last": n - 2,
           "last": n - 1}[where]
    (s if side == "src" else d)[pos] = bad
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(dst), d)[0] == oracle.ERR_OUT_OF_RANGE
    st = hz.status()
    assert _run("transfer", src, _shifted(s, off), dst, _shifted(d, off), n, st=st) == \
        kvx.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(dst.readback(), dst.host, f"nothing moved ({where}, {side}, {bad})")


@pytest.mark.parametrize("n", [8192, 32768])
def test_bad_index_in_gather(n):
    g = _rng(200 + n)
    src = _pool("hnd", "normal", g).to_device()
    s = inputs.distinct_slots(g, n, NUM)
    s[n - 3] = NUM
    buf = hz.make_mirror("buffer", SH["L"], SH["H"], SH["D"], SH["dtype"], n_tokens=n,
                         fill="sentinel").to_device()
    st = hz.status()
    assert _run("gather", src, _shifted(s, 2), None, None, n, buf, st) == kvx.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(buf.readback(), buf.host, "buffer untouched")
