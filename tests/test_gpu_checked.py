"""The checked short-form calls of the binding (gather_sync / scatter_sync / transfer_sync:
workspace and status supplied by the binding, the stream synchronised, device errors raised),
against the oracle (GPU)."""
import threading

import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SH = dict(L=3, H=2, D=64, dtype="fp16")
NUM = 6000


def _rng(k):
    return np.random.Generator(np.random.PCG64(17000 + k))


def _pool(kind, fill, g=None, salt=0):
    return hz.make_mirror(kind, SH["L"], SH["H"], SH["D"], SH["dtype"], NUM,
                          16 if kind == "hnd" else 1, fill, g, salt=salt)


def test_checked_calls_match_the_oracle_and_raise_device_errors():
    assert torch.cuda.is_available()
    g = _rng(1)
    n = 3000
    src = _pool("planes", "normal", g).to_device()
    dst = _pool("hnd", "sentinel", salt=3).to_device()
    exp = _pool("hnd", "sentinel", salt=3)
    s_np = inputs.distinct_slots(g, n, NUM)
    d_np = inputs.distinct_slots(g, n, NUM)
    s, d = hz.dev_i32(s_np), hz.dev_i32(d_np)
    # gather into a torch buffer of the [plane][token][head][dim] shape
    buf = torch.empty((2 * SH["L"], n, SH["H"], SH["D"]), dtype=torch.float16, device="cuda")
    kvx.gather_sync(hz.kvx_layout(src), s, buf)
    rc, want, _ = oracle.gather(hz.oracle_pool(src), s_np)
    assert rc == oracle.OK
    assert np.array_equal(buf.cpu().numpy().view(np.uint8).reshape(-1), want)
    # transfer on an explicit stream
    side = torch.cuda.Stream()
    kvx.transfer_sync(hz.kvx_layout(src), s, hz.kvx_layout(dst), d, stream=side)
    assert oracle.transfer(hz.oracle_pool(src), s_np, hz.oracle_pool(exp), d_np)[0] == oracle.OK
    hz.assert_same_bytes(dst.readback(), exp.host, "transfer_sync")
    # scatter the gathered buffer back into a second pool
    dst2 = _pool("slot_major", "sentinel", salt=4).to_device()
    exp2 = _pool("slot_major", "sentinel", salt=4)
    kvx.scatter_sync(hz.kvx_layout(dst2), d, buf)
    assert oracle.scatter(hz.oracle_pool(exp2), d_np, want)[0] == oracle.OK
    hz.assert_same_bytes(dst2.readback(), exp2.host, "scatter_sync")
    # a slot out of range: KvxError with the device's code, nothing written
    bad = d_np.copy()
    bad[n - 1] = NUM
    before = dst2.readback()
    with pytest.raises(kvx.KvxError) as e:
        kvx.scatter_sync(hz.kvx_layout(dst2), hz.dev_i32(bad), buf)
    assert e.value.code == kvx.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(dst2.readback(), before, "nothing written")
    # a repeated destination under the duplicate check
    rep = d_np.copy()
    rep[7] = rep[1000]
    with pytest.raises(kvx.KvxError) as e:
        kvx.transfer_sync(hz.kvx_layout(src), s, hz.kvx_layout(dst2), hz.dev_i32(rep),
                          flags=kvx.CHECK_DUP)
    assert e.value.code == kvx.ERR_DUPLICATE_DST
    hz.assert_same_bytes(dst2.readback(), before, "nothing written")
    with pytest.raises(ValueError):
        kvx.transfer_sync(hz.kvx_layout(src), s, hz.kvx_layout(dst2), d[:-1])


def test_checked_calls_from_two_threads():
    """Two host threads, each on its own stream and with its own workspace, move different
    requests into different pools at the same time; both match the oracle."""
    g = _rng(2)
    n = 2500
    src = _pool("planes", "normal", g).to_device()
    outs, exps, lists = [], [], []
    for k in range(2):
        outs.append(_pool("planes", "sentinel", salt=10 + k).to_device())
        exps.append(_pool("planes", "sentinel", salt=10 + k))
        lists.append((inputs.distinct_slots(g, n, NUM), inputs.distinct_slots(g, n, NUM)))
    errors = []

    def work(k):
        try:
            st = torch.cuda.Stream()
            s_np, d_np = lists[k]
            for _ in range(20):
                kvx.transfer_sync(hz.kvx_layout(src), hz.dev_i32(s_np), hz.kvx_layout(outs[k]),
                                  hz.dev_i32(d_np), stream=st)
        except Exception as ex:  # reported below
            errors.append(ex)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k in range(2):
        s_np, d_np = lists[k]
        assert oracle.transfer(hz.oracle_pool(src), s_np, hz.oracle_pool(exps[k]), d_np)[0] == 0
        hz.assert_same_bytes(outs[k].readback(), exps[k].host, f"thread {k}")
