"""Parity of libkvx (through its C ABI) with the CPU oracle, byte for byte.

Sizes are ones the oracle finishes in seconds while still spanning several planner tiles
(2048 tokens each) and a ragged tail.  Every comparison covers the whole destination -- the
touched rows, the untouched rows and the 64 KiB sentinel guard bands on both sides -- and the
source is checked unchanged.
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

# small shape: 3 layers (6 planes), 2 kv heads, head_dim 64, fp16 -> 256-byte rows
SH = dict(L=3, H=2, D=64, dtype="fp16")
KINDS = ["planes", "planes_separate", "slot_major", "hnd"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()  # fails loudly if libkvx.so was not built
    yield
    torch.cuda.synchronize()


PATHS = {
    # default routing: planner launch + row copy kernel (loads overlap the planner)
    "default": (0, kvx.ENGINE_AUTO),
    # one launch where it applies (rows under 2 KiB; every CTA validates and plans its slice)
    "fused": (kvx.FUSED_MAX_TOKENS, kvx.ENGINE_AUTO),
    # planner launch + TMA bulk copy (linear chunks)
    "planned_bulk": (0, kvx.ENGINE_BULK),
}


@pytest.fixture(params=sorted(PATHS))
def path(request):
    fused_max, engine = PATHS[request.param]
    kvx.set_fused_max_tokens(fused_max)
    kvx.set_copy_engine(engine)
    yield request.param
    kvx.set_fused_max_tokens(0)
    kvx.set_copy_engine(kvx.ENGINE_AUTO)


@pytest.fixture(params=["registers", "bulk"])
def engine(request):
    kvx.set_copy_engine(kvx.ENGINE_REGISTERS if request.param == "registers" else kvx.ENGINE_BULK)
    yield request.param
    kvx.set_copy_engine(kvx.ENGINE_AUTO)


def _rng(k):
    return np.random.Generator(np.random.PCG64(1000 + k))


def _pool(kind, fill, g=None, num_slots=8192, ps=16, salt=0, **sh):
    sh = {**SH, **sh}
    return hz.make_mirror(kind, sh["L"], sh["H"], sh["D"], sh["dtype"], num_slots,
                          ps if kind == "hnd" else 1, fill, g, salt=salt).to_device()


def _buffer(n, fill="sentinel", g=None, salt=7, **sh):
    sh = {**SH, **sh}
    return hz.make_mirror("buffer", sh["L"], sh["H"], sh["D"], sh["dtype"], n_tokens=n,
                          fill=fill, g=g, salt=salt).to_device()


def _sync_status(st):
    torch.cuda.synchronize()
    return st.cpu().numpy().tolist()


def _gather(src, slots, g_salt=0):
    n = len(slots)
    buf = _buffer(n)
    ws, st = hz.workspace(n), hz.status()
    lay = hz.kvx_layout(src)
    kvx.gather(lay, hz.dev_i32(slots), n, hz.GUARD + buf.dev.data_ptr(), ws, st,
               buf_bytes=n * src.P * src.R)
    return buf, st


def _slot_lists(k, n, num_slots):
    g = _rng(k)
    if n > num_slots // 2:
        return inputs.distinct_slots(g, n, num_slots)
    s, _ = inputs.fragmented_slots(g, n, num_slots, 1.6)
    return s


# ---------------------------------------------------------------------------------------
# gather / scatter / transfer
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [0, 1, 7, 2047, 2048, 2049, 4500])
def test_gather(kind, n, path):
    g = _rng(n)
    src = _pool(kind, "normal", g)
    slots = inputs.distinct_slots(g, n, src.num_slots) if n % 2 else _slot_lists(n, n, 8192)
    rc, want, _ = oracle.gather(hz.oracle_pool(src), slots)
    assert rc == oracle.OK
    buf, st = _gather(src, slots)
    assert _sync_status(st) == [kvx.OK]
    got = buf.readback()
    exp = buf.host.copy()
    exp[hz.GUARD:hz.GUARD + len(want)] = want
    hz.assert_same_bytes(got, exp, f"gather {kind} n={n}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [1, 2048, 3001])
def test_scatter(kind, n, path):
    g = _rng(100 + n)
    dst = _pool(kind, "sentinel", salt=3)
    slots = _slot_lists(100 + n, n, dst.num_slots)
    buf = _buffer(n, fill="normal", g=g)
    host_dst = dst.host.copy()
    exp_pool = hz.make_mirror(kind, SH["L"], SH["H"], SH["D"], SH["dtype"], dst.num_slots,
                              dst.page_size, "sentinel", salt=3)
    rc, _ = oracle.scatter(hz.oracle_pool(exp_pool), slots, hz.buffer_body_bytes(buf))
    assert rc == oracle.OK
    ws, st = hz.workspace(n), hz.status()
    kvx.scatter(hz.kvx_layout(dst), hz.dev_i32(slots), n, hz.GUARD + buf.dev.data_ptr(), ws, st,
                buf_bytes=n * dst.P * dst.R)
    assert _sync_status(st) == [kvx.OK]
    hz.assert_same_bytes(dst.readback(), exp_pool.host, f"scatter {kind} n={n}")
    hz.assert_same_bytes(buf.readback(), buf.host, "buffer")
    assert not np.array_equal(host_dst, exp_pool.host) or n == 0


@pytest.mark.parametrize("src_kind,dst_kind", [("planes", "planes"), ("slot_major", "hnd"),
                                               ("hnd", "planes_separate"), ("planes", "slot_major"),
                                               ("hnd", "hnd")])
@pytest.mark.parametrize("n", [5, 3000])
def test_transfer(src_kind, dst_kind, n, path):
    g = _rng(200 + n)
    src = _pool(src_kind, "normal", g)
    dst = _pool(dst_kind, "sentinel", salt=5)
    s = _slot_lists(300 + n, n, src.num_slots)
    d = _slot_lists(400 + n, n, dst.num_slots)
    exp = hz.make_mirror(dst_kind, SH["L"], SH["H"], SH["D"], SH["dtype"], dst.num_slots,
                         dst.page_size, "sentinel", salt=5)
    rc, _ = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)
    assert rc == oracle.OK
    ws, st = hz.workspace(n), hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n, ws, st)
    assert _sync_status(st) == [kvx.OK]
    hz.assert_same_bytes(dst.readback(), exp.host, f"transfer {src_kind}->{dst_kind}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


def test_small_gather_scatter_back_full_size(path):
    """Qwen2.5-1.5B shape (28 x 2 x 128 fp16), slot-major pool of 4096 slots, 128 random
    slots: gather, then scatter back into a sentinel copy and in place."""
    w = inputs.WORKLOADS["small_gather_scatter"]
    g = inputs.rng(w.seed_id, inputs.ROLE_VALUES)
    src = hz.make_mirror("slot_major", w.num_layers, w.kv_heads, w.head_dim, w.dtype,
                         w.num_slots, 1, "normal", g).to_device()
    slots = inputs.distinct_slots(inputs.rng(w.seed_id, inputs.ROLE_SRC_SLOTS), w.n_tokens, w.num_slots)
    rc, want, written = oracle.gather(hz.oracle_pool(src), slots)
    assert rc == oracle.OK and written == w.payload_bytes == 3670016
    buf = hz.make_mirror("buffer", w.num_layers, w.kv_heads, w.head_dim, w.dtype,
                         n_tokens=w.n_tokens, fill="sentinel").to_device()
    lay = hz.kvx_layout(src)
    ws, st = hz.workspace(w.n_tokens), hz.status()
    kvx.gather(lay, hz.dev_i32(slots), w.n_tokens, hz.GUARD + buf.dev.data_ptr(), ws, st,
               buf_bytes=w.payload_bytes)
    assert _sync_status(st) == [0]
    exp = buf.host.copy()
    exp[hz.GUARD:hz.GUARD + len(want)] = want
    got = buf.readback()
    hz.assert_same_bytes(got, exp, "small gather")
    # scatter back into a sentinel copy
    sent = hz.make_mirror("slot_major", w.num_layers, w.kv_heads, w.head_dim, w.dtype,
                          w.num_slots, 1, "sentinel", salt=9).to_device()
    exp_sent = hz.make_mirror("slot_major", w.num_layers, w.kv_heads, w.head_dim, w.dtype,
                              w.num_slots, 1, "sentinel", salt=9)
    assert oracle.scatter(hz.oracle_pool(exp_sent), slots, want)[0] == oracle.OK
    kvx.scatter(hz.kvx_layout(sent), hz.dev_i32(slots), w.n_tokens,
                hz.GUARD + buf.dev.data_ptr(), ws, st, buf_bytes=w.payload_bytes)
    assert _sync_status(st) == [0]
    hz.assert_same_bytes(sent.readback(), exp_sent.host, "small scatter into sentinel pool")
    # scatter back in place: the pool is unchanged
    kvx.scatter(lay, hz.dev_i32(slots), w.n_tokens, hz.GUARD + buf.dev.data_ptr(), ws, st,
                buf_bytes=w.payload_bytes)
    assert _sync_status(st) == [0]
    hz.assert_same_bytes(src.readback(), src.host, "small in-place scatter-back")


def test_hnd_page_table_gather_and_rebuild(path):
    """Fused [heads, seq, dim] -> [seq, heads, dim] gather through a page table, last page
    partial, then the inverse rebuild into a second pool under an independent page table."""
    g = _rng(77)
    L, H, D, ps, pages = 2, 4, 128, 16, 512
    src = hz.make_mirror("hnd", L, H, D, "bf16", pages * ps, ps, "normal", g).to_device()
    seq = ps * 150 + 5
    n_pages = (seq + ps - 1) // ps
    pt = inputs.random_pages(g, n_pages, pages)
    rc, want = oracle.hnd_gather(hz.oracle_pool(src), pt, seq)
    assert rc == oracle.OK
    slots = inputs.page_table_slots(pt, seq, ps)
    buf = hz.make_mirror("buffer", L, H, D, "bf16", n_tokens=seq, fill="sentinel").to_device()
    ws, st = hz.workspace(seq), hz.status()
    kvx.gather(hz.kvx_layout(src), hz.dev_i32(slots), seq, hz.GUARD + buf.dev.data_ptr(), ws, st,
               buf_bytes=len(want))
    assert _sync_status(st) == [0]
    exp = buf.host.copy()
    exp[hz.GUARD:hz.GUARD + len(want)] = want
    hz.assert_same_bytes(buf.readback(), exp, "hnd gather")
    # rebuild
    dst = hz.make_mirror("hnd", L, H, D, "bf16", pages * ps, ps, "sentinel", salt=4).to_device()
    exp_dst = hz.make_mirror("hnd", L, H, D, "bf16", pages * ps, ps, "sentinel", salt=4)
    pt2 = inputs.random_pages(_rng(78), n_pages, pages)
    assert oracle.hnd_rebuild(hz.oracle_pool(exp_dst), pt2, seq, want) == oracle.OK
    kvx.scatter(hz.kvx_layout(dst), hz.dev_i32(inputs.page_table_slots(pt2, seq, ps)), seq,
                hz.GUARD + buf.dev.data_ptr(), ws, st, buf_bytes=len(want))
    assert _sync_status(st) == [0]
    hz.assert_same_bytes(dst.readback(), exp_dst.host, "hnd rebuild")


# ---------------------------------------------------------------------------------------
# run lists
# ---------------------------------------------------------------------------------------

def _runs_from_slots(s, d):
    runs = []
    i = 0
    n = len(s)
    while i < n:
        j = i + 1
        while j < n and s[j] == s[j - 1] + 1 and d[j] == d[j - 1] + 1:
            j += 1
        runs.append((int(s[i]), int(d[i]), j - i))
        i = j
    return runs


def test_runs_gather_scatter_transfer(engine):
    g = _rng(500)
    n = 5000
    src = _pool("planes", "normal", g, num_slots=16384)
    s = np.concatenate([np.arange(100, 3100), inputs.distinct_slots(g, n - 3000, 3000) + 8000])
    d = np.concatenate([np.arange(4000, 7000), np.arange(9000, 9000 + n - 3000)])
    runs = _runs_from_slots(s, d) + [(0, 0, 0)]  # an empty run is allowed
    rt = hz.dev_i32(np.asarray(runs, np.int32).reshape(-1))
    ws, st = hz.workspace(n, len(runs)), hz.status()
    # gather by runs == gather by slots
    rc, want, _ = oracle.gather(hz.oracle_pool(src), s)
    buf = _buffer(n)
    kvx.gather_runs(hz.kvx_layout(src), rt, len(runs), n, hz.GUARD + buf.dev.data_ptr(), ws, st,
                    buf_bytes=len(want))
    assert _sync_status(st) == [0]
    exp = buf.host.copy()
    exp[hz.GUARD:hz.GUARD + len(want)] = want
    hz.assert_same_bytes(buf.readback(), exp, "gather_runs")
    # scatter by runs (dst_start field) into a sentinel pool
    dst = _pool("slot_major", "sentinel", num_slots=16384, salt=2)
    exp_dst = hz.make_mirror("slot_major", SH["L"], SH["H"], SH["D"], SH["dtype"], 16384, 1,
                             "sentinel", salt=2)
    assert oracle.scatter(hz.oracle_pool(exp_dst), d, want)[0] == oracle.OK
    druns = [(0, dd, ln) for (_, dd, ln) in runs]
    kvx.scatter_runs(hz.kvx_layout(dst), hz.dev_i32(np.asarray(druns, np.int32).reshape(-1)),
                     len(druns), n, hz.GUARD + buf.dev.data_ptr(), ws, st, buf_bytes=len(want))
    assert _sync_status(st) == [0]
    hz.assert_same_bytes(dst.readback(), exp_dst.host, "scatter_runs")
    # transfer by runs
    dst2 = _pool("hnd", "sentinel", num_slots=16384, salt=6)
    exp2 = hz.make_mirror("hnd", SH["L"], SH["H"], SH["D"], SH["dtype"], 16384, 16,
                          "sentinel", salt=6)
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp2), d)[0] == oracle.OK
    kvx.transfer_runs(hz.kvx_layout(src), hz.kvx_layout(dst2), rt, len(runs), n, ws, st)
    assert _sync_status(st) == [0]
    hz.assert_same_bytes(dst2.readback(), exp2.host, "transfer_runs")
    # a run total that disagrees with n_tokens is a device-side INVALID_ARG; nothing moves
    before = dst2.readback()
    kvx.transfer_runs(hz.kvx_layout(src), hz.kvx_layout(dst2), rt, len(runs), n - 1, ws, st)
    assert _sync_status(st) == [kvx.ERR_INVALID_ARG]
    hz.assert_same_bytes(dst2.readback(), before, "no move on bad run total")


# ---------------------------------------------------------------------------------------
# batch
# ---------------------------------------------------------------------------------------

def test_batch_mixed_ops_and_failing_request(engine):
    g = _rng(600)
    src = _pool("planes", "normal", g, num_slots=20000)
    dst = _pool("planes_separate", "sentinel", num_slots=20000, salt=8)
    exp_dst = hz.make_mirror("planes_separate", SH["L"], SH["H"], SH["D"], SH["dtype"], 20000,
                             1, "sentinel", salt=8)
    lens = [1500, 0, 2600, 700, 3000, 33]
    ops = [oracle.OP_TRANSFER, oracle.OP_TRANSFER, oracle.OP_GATHER, oracle.OP_SCATTER,
           oracle.OP_TRANSFER, oracle.OP_TRANSFER]
    n_src = sum(lens)
    ssl = inputs.distinct_slots(g, n_src, 20000)
    dsl = inputs.distinct_slots(g, n_src, 20000)
    ssl_bad = ssl.copy()
    bad_req = 4
    ssl_bad[sum(lens[:bad_req]) + 2999] = 20000  # last token of request 4 out of range
    P, R = 6, 256
    reqs, so, bo = [], 0, 0
    for op, ln in zip(ops, lens):
        reqs.append((op, ln, so, so, bo if op in (oracle.OP_GATHER, oracle.OP_SCATTER) else 0))
        if op in (oracle.OP_GATHER, oracle.OP_SCATTER):
            bo += P * ln * R
        so += ln
    buf_bytes = bo
    hbuf = np.zeros(buf_bytes, np.uint8)
    sc_off = reqs[3][4]
    hbuf[sc_off:sc_off + P * 700 * R] = g.integers(0, 256, P * 700 * R, dtype=np.uint8)
    exp_buf = hbuf.copy()
    want_status = oracle.batch(hz.oracle_pool(src), hz.oracle_pool(exp_dst), reqs, ssl_bad, dsl,
                               exp_buf)
    assert list(want_status) == [3, 0, 0, 0, 0, 3, 0]
    dbuf = torch.from_numpy(hbuf).to("cuda")
    dreq = torch.from_numpy(np.frombuffer(
        b"".join(bytes(kvx.Request(*r)) for r in reqs), dtype=np.uint8).copy()).to("cuda")
    ws, st = hz.workspace(n_src, len(reqs)), hz.status(len(reqs) + 1)
    kvx.batch(hz.kvx_layout(src), hz.kvx_layout(dst), dreq, len(reqs), n_src, hz.dev_i32(ssl_bad),
              n_src, hz.dev_i32(dsl), n_src, dbuf, ws, st)
    assert _sync_status(st) == list(want_status)
    hz.assert_same_bytes(dst.readback(), exp_dst.host, "batch destination pool")
    hz.assert_same_bytes(dbuf.cpu().numpy(), exp_buf, "batch buffer")
    # bad records: invalid op, negative length, offsets past the slot lists, unaligned buffer
    bad = [(7, 5, 0, 0, 0), (0, -1, 0, 0, 0), (2, 10, n_src - 5, 0, 0), (0, 4, 0, 0, 8)]
    dreq = torch.from_numpy(np.frombuffer(b"".join(bytes(kvx.Request(*r)) for r in bad),
                                          dtype=np.uint8).copy()).to("cuda")
    before = dst.readback()
    kvx.batch(hz.kvx_layout(src), hz.kvx_layout(dst), dreq, len(bad), 19, hz.dev_i32(ssl),
              n_src, hz.dev_i32(dsl), n_src, dbuf, ws, st)
    assert _sync_status(st)[0] == kvx.ERR_INVALID_ARG
    hz.assert_same_bytes(dst.readback(), before, "bad batch moves nothing")


# ---------------------------------------------------------------------------------------
# the plan (S1 / S2) against the oracle's run-length plan
# ---------------------------------------------------------------------------------------

def _export(ws, n):
    out = torch.zeros((n + 1, 4), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    kvx.plan_export(ws, n, out, n + 1, cnt)
    torch.cuda.synchronize()
    c = int(cnt.item())
    return out[:c].cpu().numpy()


def _assert_refines(chunks, runs, max_rows):
    """The kernel's plan refines the oracle's runs: every chunk lies inside one run, at the
    matching offset on both index lists and in the same request, and every run boundary is a
    chunk boundary, so the chunks, in order, concatenate to the runs.  How the kernel cuts a
    run (tiles, page starts, chunk size) is its own choice; only max_rows bounds a chunk."""
    assert len(chunks) >= len(runs)
    assert (chunks[:, 3] >= 1).all() and (chunks[:, 3] <= max_rows).all()
    ct = np.concatenate([[0], np.cumsum(chunks[:, 3].astype(np.int64))])
    rt = np.concatenate([[0], np.cumsum(runs[:, 3].astype(np.int64))])
    assert ct[-1] == rt[-1], "the chunks cover another number of tokens than the runs"
    r = np.searchsorted(rt, ct[:-1], side="right") - 1
    off = ct[:-1] - rt[r]
    assert (ct[1:] <= rt[r + 1]).all(), "a chunk crosses a run boundary"
    assert np.array_equal(chunks[:, 0], runs[r, 0]), "chunk request differs from its run's"
    assert np.array_equal(chunks[:, 1], runs[r, 1] + off), "chunk source offset"
    assert np.array_equal(chunks[:, 2], runs[r, 2] + off), "chunk destination offset"
    assert np.isin(rt, ct).all(), "a run boundary is not a chunk boundary"


@pytest.mark.parametrize("dst_kind", ["planes", "hnd"])
def test_plan_refines_oracle_runs(dst_kind):
    g = _rng(700)
    n = 6000
    src = _pool("planes", "normal", g, num_slots=40000)
    dst = _pool(dst_kind, "sentinel", num_slots=40000)
    s, _ = inputs.fragmented_slots(g, n, 40000, 3.0)
    d = np.concatenate([np.arange(1000, 1000 + 4100),
                        inputs.distinct_slots(g, n - 4100, 30000) + 6000])
    ws, st = hz.workspace(n), hz.status()
    kvx.plan(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst),
             hz.dev_i32(d), n, ws, st)
    assert _sync_status(st) == [0]
    got = _export(ws, n)
    want = oracle.runs(s, d, [0])
    _assert_refines(got, want, max(1, kvx.CHUNK_BYTES // src.R))
    if dst_kind == "hnd":  # a chunk is contiguous on an HND side only within one page
        assert not any((c[2] % 16) + c[3] > 16 for c in got)


def test_plan_batch_refines_oracle_runs():
    g = _rng(701)
    lens = [3000, 1, 0, 2500, 40]
    n = sum(lens)
    src = _pool("planes", "normal", g, num_slots=20000)
    dst = _pool("planes", "sentinel", num_slots=20000)
    s = np.arange(n) + 3  # one long run across requests and tiles
    d = np.arange(n) + 11
    reqs, off = [], 0
    for ln in lens:
        reqs.append((kvx.OP_TRANSFER, ln, off, off, 0))
        off += ln
    dreq = torch.from_numpy(np.frombuffer(b"".join(bytes(kvx.Request(*r)) for r in reqs),
                                          dtype=np.uint8).copy()).to("cuda")
    ws, st = hz.workspace(n, len(reqs)), hz.status(len(reqs) + 1)
    kvx.plan_batch(hz.kvx_layout(src), hz.kvx_layout(dst), dreq, len(reqs), n, hz.dev_i32(s), n,
                   hz.dev_i32(d), n, 0, ws, st)
    assert _sync_status(st) == [0] * (len(reqs) + 1)
    got = _export(ws, n)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    want = oracle.runs(s, d, starts)
    assert want[:, 3].tolist() == [3000, 1, 2500, 40]  # one run per non-empty request
    _assert_refines(got, want, max(1, kvx.CHUNK_BYTES // src.R))


# ---------------------------------------------------------------------------------------
# errors, two-phase use, host submission
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("bad", [8192, -1, 2 ** 31 - 1])
def test_out_of_range_moves_nothing(bad, path):
    g = _rng(800)
    n = 5000
    src = _pool("planes", "normal", g)
    dst = _pool("planes", "sentinel", salt=1)
    s = inputs.distinct_slots(g, n, 8192)
    d = inputs.distinct_slots(g, n, 8192)
    d[4321] = bad  # in the third planner tile; the first two tiles are clean
    ws, st = hz.workspace(n), hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n, ws, st)
    assert _sync_status(st) == [kvx.ERR_OUT_OF_RANGE]
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(dst), d)[0] == oracle.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(dst.readback(), dst.host, "destination untouched")


def test_host_side_errors():
    g = _rng(900)
    src = _pool("planes", "normal", g)
    lay = hz.kvx_layout(src)
    ws, st = hz.workspace(10), hz.status()
    slots = hz.dev_i32(np.arange(10))
    with pytest.raises(kvx.KvxError) as e:  # buffer inside the pool
        kvx.gather(lay, slots, 10, hz.GUARD + src.dev.data_ptr() + 4096, ws, st,
                   buf_bytes=10 * src.P * src.R)
    assert e.value.code == kvx.ERR_OVERLAP
    buf = _buffer(10)
    with pytest.raises(kvx.KvxError) as e:
        kvx.gather(lay, slots, 10, hz.GUARD + buf.dev.data_ptr() + 8, ws, st,
                   buf_bytes=10 * src.P * src.R)
    assert e.value.code == kvx.ERR_ALIGNMENT
    with pytest.raises(kvx.KvxError) as e:
        kvx.gather(lay, slots, 10, hz.GUARD + buf.dev.data_ptr(), ws, st,
                   buf_bytes=10 * src.P * src.R - 1)
    assert e.value.code == kvx.ERR_INVALID_ARG
    with pytest.raises(kvx.KvxError) as e:
        kvx.gather(lay, slots, 10, hz.GUARD + buf.dev.data_ptr(), ws[:256], st,
                   buf_bytes=10 * src.P * src.R)
    assert e.value.code == kvx.ERR_NO_WORKSPACE
    with pytest.raises(kvx.KvxError) as e:  # transfer within one pool
        kvx.transfer(lay, slots, lay, slots, 10, ws, st)
    assert e.value.code == kvx.ERR_OVERLAP
    other = _pool("planes", "sentinel", L=4)
    with pytest.raises(kvx.KvxError) as e:  # different number of layers
        kvx.transfer(lay, slots, hz.kvx_layout(other), slots, 10, ws, st)
    assert e.value.code == kvx.ERR_INVALID_ARG


def test_plan_once_execute_twice(engine):
    """A plan depends on indices and geometry only: one plan serves two destination pools."""
    g = _rng(1000)
    n = 3000
    src = _pool("planes", "normal", g)
    s = _slot_lists(1001, n, 8192)
    d = _slot_lists(1002, n, 8192)
    ws, st = hz.workspace(n), hz.status()
    a = _pool("hnd", "sentinel", salt=1)
    b = _pool("hnd", "sentinel", salt=2)
    kvx.plan(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(a), hz.dev_i32(d),
             n, ws, st)
    for m in (a, b):
        kvx.execute(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.kvx_layout(m), None, 0, n, None, ws,
                    st, buf_bytes=0)
        assert _sync_status(st) == [0]
        exp = hz.make_mirror("hnd", SH["L"], SH["H"], SH["D"], SH["dtype"], 8192, 16,
                             "sentinel", salt=1 if m is a else 2)
        assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == 0
        hz.assert_same_bytes(m.readback(), exp.host, "execute")
    # executing with another token count than the plan's is caught on the device
    c = _pool("hnd", "sentinel", salt=3)
    kvx.execute(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.kvx_layout(c), None, 0, n - 1, None, ws,
                st, buf_bytes=0)
    assert _sync_status(st) == [kvx.ERR_INVALID_ARG]
    hz.assert_same_bytes(c.readback(), c.host, "no move on plan mismatch")


def test_submit_with_host_slot_lists(path):
    g = _rng(1100)
    n = 2500
    src = _pool("planes", "normal", g)
    dst = _pool("planes", "sentinel", salt=1)
    s = torch.from_numpy(_slot_lists(1101, n, 8192).astype(np.int32)).pin_memory()
    d = torch.from_numpy(_slot_lists(1102, n, 8192).astype(np.int32)).pin_memory()
    hst = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    ws = hz.workspace(n)
    kvx.submit(kvx.OP_TRANSFER, hz.kvx_layout(src), s, hz.kvx_layout(dst), d, n, None, ws, hst,
               buf_bytes=0)
    torch.cuda.synchronize()
    assert int(hst[0]) == 0
    exp = hz.make_mirror("planes", SH["L"], SH["H"], SH["D"], SH["dtype"], 8192, 1, "sentinel",
                         salt=1)
    assert oracle.transfer(hz.oracle_pool(src), s.numpy(), hz.oracle_pool(exp), d.numpy())[0] == 0
    hz.assert_same_bytes(dst.readback(), exp.host, "submit")


# kvx_submit with the 2 KiB rows of the 144 KiB/token shape: the row kernel reads pinned slot
# lists in place and writes the status word itself; pageable lists / status are staged.
SUBMIT_MEM = ["pinned", "pageable", "pinned_lists_pageable_status"]


@pytest.mark.parametrize("mem", SUBMIT_MEM)
@pytest.mark.parametrize("op", ["gather", "scatter", "transfer"])
def test_submit_rows_2k(op, mem, path):
    sh = dict(L=4, H=8, D=128, dtype="bf16")
    n, num = 3000, 8192
    g = _rng(1200)
    src = _pool("planes", "normal", g, num_slots=num, **sh)
    s_np = _slot_lists(1201, n, num).astype(np.int32)
    d_np = _slot_lists(1202, n, num).astype(np.int32)
    pin_lists = mem != "pageable"
    s = torch.from_numpy(s_np).pin_memory() if pin_lists else s_np.copy()
    d = torch.from_numpy(d_np).pin_memory() if pin_lists else d_np.copy()
    hst = torch.full((1,), -1, dtype=torch.int32)
    hst = hst.pin_memory() if mem == "pinned" else hst
    ws = hz.workspace(n)
    if op == "gather":
        rc, want, _ = oracle.gather(hz.oracle_pool(src), s_np)
        buf = _buffer(n, **sh)
        kvx.submit(kvx.OP_GATHER, hz.kvx_layout(src), s, None, None, n,
                   hz.GUARD + buf.dev.data_ptr(), ws, hst, buf_bytes=n * buf.P * buf.R)
        torch.cuda.synchronize()
        got = buf.readback()
        exp = buf.host.copy()
        exp[hz.GUARD:hz.GUARD + want.size] = want
    else:
        dst = _pool("planes", "sentinel", num_slots=num, salt=2, **sh)
        exp_m = hz.make_mirror("planes", sh["L"], sh["H"], sh["D"], sh["dtype"], num, 1,
                               "sentinel", salt=2)
        if op == "scatter":
            buf = _buffer(n, "normal", g, **sh)
            rc = oracle.scatter(hz.oracle_pool(exp_m), d_np, hz.buffer_body_bytes(buf))[0]
            kvx.submit(kvx.OP_SCATTER, None, None, hz.kvx_layout(dst), d, n,
                       hz.GUARD + buf.dev.data_ptr(), ws, hst, buf_bytes=n * buf.P * buf.R)
        else:
            rc = oracle.transfer(hz.oracle_pool(src), s_np, hz.oracle_pool(exp_m), d_np)[0]
            kvx.submit(kvx.OP_TRANSFER, hz.kvx_layout(src), s, hz.kvx_layout(dst), d, n, None,
                       ws, hst, buf_bytes=0)
        torch.cuda.synchronize()
        got, exp = dst.readback(), exp_m.host
    assert rc == 0
    assert int(hst[0]) == kvx.OK
    hz.assert_same_bytes(got, exp, f"submit {op} {mem}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


@pytest.mark.parametrize("mem", SUBMIT_MEM)
def test_submit_rows_2k_out_of_range(mem, path):
    sh = dict(L=4, H=8, D=128, dtype="bf16")
    n, num = 3000, 8192
    g = _rng(1300)
    src = _pool("planes", "normal", g, num_slots=num, **sh)
    dst = _pool("planes", "sentinel", num_slots=num, salt=2, **sh)
    s_np = _slot_lists(1301, n, num).astype(np.int32)
    d_np = _slot_lists(1302, n, num).astype(np.int32)
    d_np[n - 5] = num  # one past the end: the whole request must move nothing
    pin = mem != "pageable"
    s = torch.from_numpy(s_np).pin_memory() if pin else s_np
    d = torch.from_numpy(d_np).pin_memory() if pin else d_np
    hst = torch.full((1,), -1, dtype=torch.int32)
    hst = hst.pin_memory() if mem == "pinned" else hst
    before = dst.readback()
    kvx.submit(kvx.OP_TRANSFER, hz.kvx_layout(src), s, hz.kvx_layout(dst), d, n, None,
               hz.workspace(n), hst, buf_bytes=0)
    torch.cuda.synchronize()
    assert int(hst[0]) == kvx.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(dst.readback(), before, "nothing moved")


# ---------------------------------------------------------------------------------------
# 2 KiB rows (the 144 KiB/token shape): one-row chunks, so the planned path runs the row
# kernel, which loads its rows before the planner's verdict and stores only after it
# ---------------------------------------------------------------------------------------

SH2K = dict(L=4, H=8, D=128, dtype="bf16")


@pytest.mark.parametrize("op", ["gather", "scatter", "transfer"])
@pytest.mark.parametrize("n", [1, 2048, 5000])
def test_rows_2k(op, n, path):
    g = _rng(3000 + n)
    num = 8192
    src = _pool("planes", "normal", g, num_slots=num, **SH2K)
    s = _slot_lists(3001 + n, n, num)
    d = _slot_lists(3002 + n, n, num)
    ws, st = hz.workspace(n), hz.status()
    P, R = 2 * SH2K["L"], SH2K["H"] * SH2K["D"] * 2
    if op == "gather":
        rc, want, _ = oracle.gather(hz.oracle_pool(src), s)
        buf = _buffer(n, **SH2K)
        kvx.gather(hz.kvx_layout(src), hz.dev_i32(s), n, hz.GUARD + buf.dev.data_ptr(), ws, st,
                   buf_bytes=n * P * R)
        exp = buf.host.copy()
        exp[hz.GUARD:hz.GUARD + len(want)] = want
        assert _sync_status(st) == [0]
        hz.assert_same_bytes(buf.readback(), exp, f"gather 2k {path}")
        return
    dst = _pool("planes_separate", "sentinel", num_slots=num, salt=4, **SH2K)
    exp = hz.make_mirror("planes_separate", SH2K["L"], SH2K["H"], SH2K["D"], SH2K["dtype"], num,
                         1, "sentinel", salt=4)
    if op == "scatter":
        buf = _buffer(n, fill="normal", g=g, **SH2K)
        assert oracle.scatter(hz.oracle_pool(exp), d, hz.buffer_body_bytes(buf))[0] == 0
        kvx.scatter(hz.kvx_layout(dst), hz.dev_i32(d), n, hz.GUARD + buf.dev.data_ptr(), ws, st,
                    buf_bytes=n * P * R)
    else:
        assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == 0
        kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n, ws, st)
    assert _sync_status(st) == [0]
    hz.assert_same_bytes(dst.readback(), exp.host, f"{op} 2k {path}")


@pytest.mark.parametrize("where", [0, 2047, 4999])
def test_rows_2k_out_of_range_moves_nothing(where, path):
    """The row kernel may load rows before the planner's verdict; it must store none of them
    when any index of the request (here in the first, a middle or the last tile) is bad."""
    g = _rng(4000 + where)
    n, num = 5000, 8192
    src = _pool("planes", "normal", g, num_slots=num, **SH2K)
    dst = _pool("planes", "sentinel", num_slots=num, salt=2, **SH2K)
    s = _slot_lists(4001, n, num)
    d = _slot_lists(4002, n, num)
    s[where] = num  # one source index out of range
    ws, st = hz.workspace(n), hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n, ws, st)
    assert _sync_status(st) == [kvx.ERR_OUT_OF_RANGE]
    hz.assert_same_bytes(dst.readback(), dst.host, "destination untouched")
