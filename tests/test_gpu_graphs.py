"""libkvx calls captured into a CUDA graph and replayed (GPU).

A captured kvx_transfer / kvx_gather / kvx_scatter (and kvx_batch, the run-list forms, the
duplicate check with its table memset, the bulk engine) replays its planner and copy on every
launch of the graph, so new slot lists, requests and runs written in place into the captured
buffers move new rows.  Each replay is compared byte for byte with the oracle.
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


def test_batch_runs_and_checked_calls_replay():
    """One graph holding a kvx_batch, a kvx_transfer_runs and a duplicate-checked kvx_transfer
    on the bulk engine (its table memset and planner inside the graph): replays with new
    requests, runs and slot lists all match the oracle, and a replay with a repeated
    destination refuses only that call."""
    L, H, D, dt = 3, 2, 64, "fp16"
    num, n = 6000, 1500
    src = hz.make_mirror("planes", L, H, D, dt, num, 1, "normal", _rng(30)).to_device()
    dsts = [hz.make_mirror("planes", L, H, D, dt, num, 1, "sentinel", salt=40 + k).to_device()
            for k in range(3)]
    sl, dls = hz.kvx_layout(src), [hz.kvx_layout(m) for m in dsts]
    # batch: three transfer requests of 500 tokens over shared slot buffers
    lens = [500, 500, 500]
    reqs = [(kvx.OP_TRANSFER, ln, 500 * k, 500 * k, 0) for k, ln in enumerate(lens)]
    dreq = torch.from_numpy(np.frombuffer(b"".join(bytes(kvx.Request(*r)) for r in reqs),
                                          dtype=np.uint8).copy()).cuda()
    bs = torch.zeros(n, dtype=torch.int32, device="cuda")
    bd = torch.zeros(n, dtype=torch.int32, device="cuda")
    max_runs = 64
    runs = torch.zeros(3 * max_runs, dtype=torch.int32, device="cuda")
    ts = torch.zeros(n, dtype=torch.int32, device="cuda")
    td = torch.zeros(n, dtype=torch.int32, device="cuda")
    ws = [hz.workspace(n, max(len(reqs), max_runs)) for _ in range(3)]
    sts = [hz.status(len(reqs) + 1), hz.status(), hz.status()]

    def calls():
        kvx.batch(sl, dls[0], dreq, len(reqs), n, bs, n, bd, n, None, ws[0], sts[0], buf_bytes=0,
                  flags=0)
        kvx.transfer_runs(sl, dls[1], runs, max_runs, n, ws[1], sts[1], flags=kvx.CHECK_DUP)
        kvx.transfer(sl, ts, dls[2], td, n, ws[2], sts[2], flags=kvx.CHECK_DUP | kvx.USE_BULK)

    def load(rep, dup=False):
        g = _rng(100 + rep)
        s1, d1 = inputs.distinct_slots(g, n, num), inputs.distinct_slots(g, n, num)
        # runs: max_runs runs of varying lengths covering n tokens, distinct destinations
        cuts = np.sort(g.choice(np.arange(1, n), max_runs - 1, replace=False))
        lens_r = np.diff(np.concatenate([[0], cuts, [n]]))
        starts_s = g.choice(num - 64, max_runs, replace=False)
        base_d = np.cumsum(np.concatenate([[0], lens_r[:-1] + 1]))  # gaps keep them distinct
        rr = np.stack([starts_s[:max_runs] % (num - 64), base_d, lens_r], axis=1).astype(np.int32)
        rr[:, 0] = np.minimum(rr[:, 0], num - rr[:, 2])
        s3, d3 = inputs.distinct_slots(g, n, num), inputs.distinct_slots(g, n, num)
        if dup:
            d3[7] = d3[1000]
        bs.copy_(torch.from_numpy(s1).cuda())
        bd.copy_(torch.from_numpy(d1).cuda())
        runs.copy_(torch.from_numpy(rr.reshape(-1)).cuda())
        ts.copy_(torch.from_numpy(s3).cuda())
        td.copy_(torch.from_numpy(d3).cuda())
        rs = np.concatenate([np.arange(a, a + c) for a, _, c in rr]).astype(np.int32)
        rd = np.concatenate([np.arange(b, b + c) for _, b, c in rr]).astype(np.int32)
        return (s1, d1), (rs, rd), (s3, d3)

    side = torch.cuda.Stream()
    load(0)
    with torch.cuda.stream(side):  # warm up outside the capture
        calls()
    torch.cuda.synchronize()
    for m in dsts:  # back to the sentinel
        m.dev.copy_(torch.from_numpy(m.host).cuda())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()
    exps = [hz.make_mirror("planes", L, H, D, dt, num, 1, "sentinel", salt=40 + k)
            for k in range(3)]
    for rep in range(3):
        lists = load(rep + 1, dup=(rep == 2))
        graph.replay()
        torch.cuda.synchronize()
        want_batch = oracle.batch(hz.oracle_pool(src), hz.oracle_pool(exps[0]), reqs, lists[0][0],
                                  lists[0][1], np.zeros(16, np.uint8))
        assert sts[0].cpu().tolist() == list(want_batch)
        assert oracle.transfer(hz.oracle_pool(src), lists[1][0], hz.oracle_pool(exps[1]),
                               lists[1][1], check_dup=True)[0] == oracle.OK
        assert int(sts[1].item()) == kvx.OK
        rc = oracle.transfer(hz.oracle_pool(src), lists[2][0], hz.oracle_pool(exps[2]),
                             lists[2][1], check_dup=True)[0]
        assert int(sts[2].item()) == rc == (kvx.ERR_DUPLICATE_DST if rep == 2 else kvx.OK)
        for k in range(3):
            hz.assert_same_bytes(dsts[k].readback(), exps[k].host, f"replay {rep}, call {k}")
