"""Calls on several streams at once, and the streamed and resharding calls captured into CUDA
graphs and replayed, against the oracle (GPU).

- Four transfers from one source pool into four destination pools, each on its own stream
  with its own workspace and status, all enqueued before any synchronisation (planner path,
  small-request path and narrow rows mixed).
- kvx_reshard, kvx_stream and kvx_stream_reshard captured once into a graph and replayed with
  new slot lists written in place into the captured index buffers (and, for the streamed
  calls, ready words already raised): every replay equals the oracle's move of those slots.
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
    return np.random.Generator(np.random.PCG64(16000 + k))


def test_four_streams_at_once():
    L, H, D, num = 3, 2, 64, 8192
    g = _rng(1)
    src = hz.make_mirror("planes", L, H, D, "fp16", num, 1, "normal", g).to_device()
    ns = [300, 3000, 512, 2049]  # small path, planner path, boundary, two planner tiles
    dsts = [hz.make_mirror("hnd" if k % 2 else "planes", L, H, D, "fp16", num,
                           16 if k % 2 else 1, "sentinel", salt=k).to_device() for k in range(4)]
    exps = [hz.make_mirror("hnd" if k % 2 else "planes", L, H, D, "fp16", num,
                           16 if k % 2 else 1, "sentinel", salt=k) for k in range(4)]
    streams = [torch.cuda.Stream() for _ in range(4)]
    lists, stats, wss = [], [], []
    for k, n in enumerate(ns):
        s = inputs.distinct_slots(g, n, num)
        d = inputs.distinct_slots(g, n, num)
        lists.append((s, d, hz.dev_i32(s), hz.dev_i32(d)))
        stats.append(hz.status())
        wss.append(hz.workspace(n))
    torch.cuda.synchronize()
    for k, n in enumerate(ns):
        s, d, sd, dd = lists[k]
        kvx.transfer(hz.kvx_layout(src), sd, hz.kvx_layout(dsts[k]), dd, n, wss[k], stats[k],
                     stream=int(streams[k].cuda_stream))
    torch.cuda.synchronize()
    for k, n in enumerate(ns):
        s, d, _, _ = lists[k]
        assert int(stats[k].item()) == kvx.OK
        assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exps[k]), d)[0] == oracle.OK
        hz.assert_same_bytes(dsts[k].readback(), exps[k].host, f"stream {k} (n={n})")


def _capture(fn):
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):  # warm up outside the capture
        fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


@pytest.mark.parametrize("streamed", [False, True])
def test_reshard_graph_replays_new_slots(streamed):
    L, D, num, n = 3, 64, 4096, 1000
    g = _rng(2 + streamed)
    p = [hz.make_mirror("hnd", L, 2, D, "fp16", num, 16, "normal", g).to_device() for _ in range(4)]
    d = [hz.make_mirror("planes", L, 4, D, "fp16", num, 1, "sentinel", salt=r).to_device()
         for r in range(2)]
    parts = kvx.tp_plan(8, 4, 2)
    s_dev = torch.zeros(n, dtype=torch.int32, device="cuda")
    d_dev = torch.zeros(n, dtype=torch.int32, device="cuda")
    s_dev.copy_(torch.arange(n, dtype=torch.int32, device="cuda"))
    d_dev.copy_(torch.arange(n, dtype=torch.int32, device="cuda"))
    ws = hz.workspace(n)
    st = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    words = torch.ones(L, dtype=torch.int32, device="cuda")
    pl, dl = [hz.kvx_layout(m) for m in p], [hz.kvx_layout(m) for m in d]

    def call():
        if streamed:
            kvx.stream_reshard(pl, s_dev, dl, d_dev, parts, n, ws, st, layer_ready=words,
                               ready_value=1)
        else:
            kvx.reshard(pl, s_dev, dl, d_dev, parts, n, ws, st[:1])

    graph = _capture(call)
    for rep in range(3):
        for m in d:
            m.dev.copy_(torch.from_numpy(m.host))
        exp = [hz.make_mirror("planes", L, 4, D, "fp16", num, 1, "sentinel", salt=r)
               for r in range(2)]
        s = inputs.distinct_slots(_rng(10 + rep), n, num)
        dd = inputs.distinct_slots(_rng(20 + rep), n, num)
        s_dev.copy_(torch.from_numpy(s).cuda())
        d_dev.copy_(torch.from_numpy(dd).cuda())
        graph.replay()
        torch.cuda.synchronize()
        v = st.cpu().tolist()
        assert v[0] == kvx.OK and (not streamed or v[1:] == [0, 0, 1]), v
        rc, _ = oracle.reshard([hz.oracle_pool(m) for m in p], s, [hz.oracle_pool(m) for m in exp],
                               dd, parts, n)
        assert rc == oracle.OK
        for r in range(2):
            hz.assert_same_bytes(d[r].readback(), exp[r].host, f"replay {rep}, D rank {r}")


def test_stream_graph_replays_new_slots():
    L, H, D, num, n = 4, 8, 128, 4096, 1500
    g = _rng(5)
    src = hz.make_mirror("planes", L, H, D, "bf16", num, 1, "normal", g).to_device()
    dst = hz.make_mirror("slot_major", L, H, D, "bf16", num, 1, "sentinel", salt=3).to_device()
    s_dev = torch.arange(n, dtype=torch.int32, device="cuda")
    d_dev = torch.arange(n, dtype=torch.int32, device="cuda")
    ws = hz.workspace(n)
    st = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    words = torch.ones(L, dtype=torch.int32, device="cuda")
    sl, dl = hz.kvx_layout(src), hz.kvx_layout(dst)

    def call():
        kvx.stream(kvx.OP_TRANSFER, sl, s_dev, dl, d_dev, n, None, ws, st, layer_ready=words,
                   ready_value=1, buf_bytes=0)

    graph = _capture(call)
    for rep in range(3):
        dst.dev.copy_(torch.from_numpy(dst.host))
        exp = hz.make_mirror("slot_major", L, H, D, "bf16", num, 1, "sentinel", salt=3)
        s = inputs.distinct_slots(_rng(30 + rep), n, num)
        d = inputs.distinct_slots(_rng(40 + rep), n, num)
        s_dev.copy_(torch.from_numpy(s).cuda())
        d_dev.copy_(torch.from_numpy(d).cuda())
        graph.replay()
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [kvx.OK, 0, 0, 1]
        assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == oracle.OK
        hz.assert_same_bytes(dst.readback(), exp.host, f"stream replay {rep}")


@pytest.mark.parametrize("n", [700, 2500])  # one planner tile (status written by the planner) and two
def test_stream_graph_replay_is_a_new_call(n):
    """A replay must not inherit what an earlier replay of the same capture saw: after a replay
    with every layer ready, a replay with layer 2's ready word lowered stops there with
    KVX_ERR_TIMEOUT (layers 0 and 1 moved, layer 2 untouched, each row of the raised layer 3
    either moved or untouched, as kvx_stream allows for layers past the pending count); a third
    replay with the word raised again moves everything."""
    L, H, D, num = 4, 2, 64, 4096
    g = _rng(60 + n)
    src = hz.make_mirror("planes", L, H, D, "fp16", num, 1, "normal", g).to_device()
    dst = hz.make_mirror("planes", L, H, D, "fp16", num, 1, "sentinel", salt=4).to_device()
    s = inputs.distinct_slots(g, n, num)
    d = inputs.distinct_slots(g, n, num)
    s_dev, d_dev = hz.dev_i32(s), hz.dev_i32(d)
    ws = hz.workspace(n)
    st = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    words = torch.ones(L, dtype=torch.int32, device="cuda")
    sl, dl = hz.kvx_layout(src), hz.kvx_layout(dst)
    full = hz.make_mirror("planes", L, H, D, "fp16", num, 1, "sentinel", salt=4)
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(full), d)[0] == oracle.OK
    two = hz.make_mirror("planes", L, H, D, "fp16", num, 1, "sentinel", salt=4)
    assert oracle.transfer_layers(hz.oracle_pool(src), s, hz.oracle_pool(two), d, 2)[0] == oracle.OK

    def call():
        kvx.stream(kvx.OP_TRANSFER, sl, s_dev, dl, d_dev, n, None, ws, st, layer_ready=words,
                   ready_value=1, wait_ns=20_000_000, buf_bytes=0)

    graph = _capture(call)
    for rep, ready in enumerate([[1, 1, 1, 1], [1, 1, 0, 1], [1, 1, 1, 1]]):
        dst.dev.copy_(torch.from_numpy(dst.host))
        words.copy_(torch.tensor(ready, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        v = st.cpu().tolist()
        got = dst.readback()
        if 0 not in ready:
            assert v == [kvx.OK, 0, 0, 1], (rep, v)
            hz.assert_same_bytes(got, full.host, f"replay {rep}")
            continue
        assert v[0] == kvx.ERR_TIMEOUT and v[1] == L - 2 and v[3] == 1, (rep, v)
        body = got[hz.GUARD:hz.GUARD + two.body.nbytes].view(np.uint16).reshape(two.body.shape)
        late = body[6:8].reshape(2, num, -1)  # layer 3's K and V planes, rows by slot
        moved = (late == full.body[6:8].reshape(2, num, -1)).all(axis=2)
        kept = (late == two.body[6:8].reshape(2, num, -1)).all(axis=2)
        assert (moved | kept).all(), f"replay {rep}: a layer-3 row is neither moved nor untouched"
        merged = two.host.copy()
        merged_body = merged[hz.GUARD:hz.GUARD + two.body.nbytes].view(np.uint16) \
            .reshape(two.body.shape)
        merged_body[6:8] = body[6:8]
        hz.assert_same_bytes(got, merged, f"replay {rep} (layers 0-2 and guards)")
