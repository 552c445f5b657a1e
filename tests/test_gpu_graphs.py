"""libkvx calls captured into a CUDA graph and replayed (GPU).

A captured kvx_transfer / kvx_gather / kvx_scatter replays its planner and copy on every
launch of the graph, so new slot lists written in place into the captured index buffers move
new rows.  Each replay is compared byte for byte with the oracle.
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
    return np.random.Generator(np.random.PCG64(15000 + k))


@pytest.mark.parametrize("shape", [(28, 2, 128, "fp16", "slot_major"), (4, 8, 128, "bf16", "planes")])
def test_transfer_graph_replays_new_slots(shape):
    L, H, D, dt, kind = shape
    n, num = 128, 4096
    src = hz.make_mirror(kind, L, H, D, dt, num, 1, "normal", _rng(1)).to_device()
    dst = hz.make_mirror("planes", L, H, D, dt, num, 1, "sentinel", salt=2).to_device()
    s_dev = torch.zeros(n, dtype=torch.int32, device="cuda")
    d_dev = torch.zeros(n, dtype=torch.int32, device="cuda")
    ws, st = hz.workspace(n), hz.status()
    sl, dl = hz.kvx_layout(src), hz.kvx_layout(dst)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):  # warm up outside the capture (library and device setup)
        s_dev.copy_(torch.arange(n, dtype=torch.int32, device="cuda"))
        d_dev.copy_(torch.arange(n, dtype=torch.int32, device="cuda"))
        kvx.transfer(sl, s_dev, dl, d_dev, n, ws, st)
    torch.cuda.synchronize()
    dst.dev.copy_(torch.from_numpy(dst.host).cuda())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvx.transfer(sl, s_dev, dl, d_dev, n, ws, st)
    exp = hz.make_mirror("planes", L, H, D, dt, num, 1, "sentinel", salt=2)
    for rep in range(3):
        s = inputs.distinct_slots(_rng(10 + rep), n, num)
        d = inputs.distinct_slots(_rng(20 + rep), n, num)
        s_dev.copy_(torch.from_numpy(s).cuda())
        d_dev.copy_(torch.from_numpy(d).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == kvx.OK
        assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == oracle.OK
        hz.assert_same_bytes(dst.readback(), exp.host, f"replay {rep}")


def test_gather_scatter_graph_and_bad_index():
    L, H, D, dt = 28, 2, 128, "fp16"
    n, num = 128, 4096
    pool = hz.make_mirror("slot_major", L, H, D, dt, num, 1, "normal", _rng(3)).to_device()
    buf = torch.zeros(2 * L * n * H * D, dtype=torch.float16, device="cuda")
    slots = torch.zeros(n, dtype=torch.int32, device="cuda")
    ws1, ws2, st1, st2 = hz.workspace(n), hz.workspace(n), hz.status(), hz.status()
    lay = hz.kvx_layout(pool)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        slots.copy_(torch.arange(n, dtype=torch.int32, device="cuda"))
        kvx.gather(lay, slots, n, buf, ws1, st1)
        kvx.scatter(lay, slots, n, buf, ws2, st2)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvx.gather(lay, slots, n, buf, ws1, st1)
        kvx.scatter(lay, slots, n, buf, ws2, st2)  # scatter back in place: pool unchanged
    s = inputs.distinct_slots(_rng(4), n, num)
    slots.copy_(torch.from_numpy(s).cuda())
    g.replay()
    torch.cuda.synchronize()
    assert int(st1.item()) == kvx.OK and int(st2.item()) == kvx.OK
    rc, want, _ = oracle.gather(hz.oracle_pool(pool), s)
    assert rc == oracle.OK
    assert np.array_equal(buf.cpu().numpy().view(np.uint8), want)
    hz.assert_same_bytes(pool.readback(), pool.host, "scatter back in place")
    # a replay with an index out of range: both legs refuse, nothing written
    bad = s.copy()
    bad[5] = num
    slots.copy_(torch.from_numpy(bad).cuda())
    buf_before = buf.clone()
    g.replay()
    torch.cuda.synchronize()
    assert int(st1.item()) == kvx.ERR_OUT_OF_RANGE and int(st2.item()) == kvx.ERR_OUT_OF_RANGE
    assert torch.equal(buf, buf_before)
    hz.assert_same_bytes(pool.readback(), pool.host, "nothing moved")
