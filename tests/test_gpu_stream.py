"""kvx_stream -- layer-streamed, cancellable moves -- against the oracle, through the C ABI (GPU).

What is checked:
  * with every layer ready (no ready words, or ready words already raised) kvx_stream moves
    exactly the bytes the oracle's gather / scatter / transfer move, for every pool kind;
  * layers raised late by the host (pinned ready words written after the launch) are all moved,
    and the kernel cannot finish before the last one is raised;
  * a layer never raised ends the move with KVX_ERR_TIMEOUT after the bounded wait: every layer
    below it holds the oracle's rows, every layer from it on is untouched;
  * a request cancelled by the host (its pinned epoch word changed) while the kernel waits
    ends long before the wait bound with KVX_ERR_CANCELLED, layers below the waiting one moved
    and the rest untouched; a request cancelled before the launch moves nothing;
  * the "no further write" words (status[3] and the pinned host word) are set in every case.
Each case runs on the default grid and on a persistent grid of 40 CTAs in its three forms
(register and TMA bulk-copy warps mixed, registers only, TMA bulk copies only).

Every failure is made on the host: a ready word that nothing raises, an epoch word the host
changes.  Every device wait is bounded (wait_ns), so no case can hang the GPU.
"""
import time

import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SH = dict(L=6, H=2, D=64, dtype="fp16")      # 256-byte rows: 8 tokens per warp
SH2K = dict(L=6, H=8, D=128, dtype="bf16")   # 2 KiB rows: one token per warp
KINDS = ["planes", "slot_major", "hnd"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


# max_ctas: 0 = one warp per row group (default grid); 40 = a persistent grid of 40 CTAs, in
# its mixed form (the default: register warps and TMA bulk-copy warps), its register form and
# its bulk (TMA) form
GRIDS = {"rowgrid": (0, kvx.ENGINE_AUTO), "persistent40": (40, kvx.ENGINE_AUTO),
         "persistent40_registers": (40, kvx.ENGINE_REGISTERS),
         "persistent40_bulk": (40, kvx.ENGINE_BULK)}
ENGINES = dict(ids=["mixed", "registers", "bulk"])
ENGINE_LIST = [kvx.ENGINE_AUTO, kvx.ENGINE_REGISTERS, kvx.ENGINE_BULK]


@pytest.fixture(params=list(GRIDS))
def grid(request):
    max_ctas, engine = GRIDS[request.param]
    kvx.set_copy_engine(engine)
    yield max_ctas
    kvx.set_copy_engine(kvx.ENGINE_AUTO)


def _rng(k):
    return np.random.Generator(np.random.PCG64(5000 + k))


def _pool(kind, fill, g=None, num_slots=4096, salt=0, sh=SH):
    return hz.make_mirror(kind, sh["L"], sh["H"], sh["D"], sh["dtype"], num_slots,
                          16 if kind == "hnd" else 1, fill, g, salt=salt).to_device()


def _expected_pool(kind, num_slots, salt, sh=SH):
    return hz.make_mirror(kind, sh["L"], sh["H"], sh["D"], sh["dtype"], num_slots,
                          16 if kind == "hnd" else 1, "sentinel", salt=salt)


def _slots(k, n, num_slots):
    return inputs.distinct_slots(_rng(k), n, num_slots)


def _pinned_i32(values):
    return torch.tensor(values, dtype=torch.int32).pin_memory()


def _status():
    return torch.full((4,), -1, dtype=torch.int32, device="cuda")


def _transfer_case(kind, n, sh=SH, seed=0, stop=None):
    """Pools, slot lists and the oracle's expected destination: the whole transfer, or (stop)
    the transfer of the layers before `stop` only."""
    g = _rng(seed)
    src = _pool(kind, "normal", g, sh=sh)
    dst = _pool(kind, "sentinel", salt=5, sh=sh)
    s = _slots(seed + 1, n, src.num_slots)
    d = _slots(seed + 2, n, dst.num_slots)
    exp = _expected_pool(kind, dst.num_slots, 5, sh=sh)
    if stop is None:
        rc, _ = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)
    else:
        rc, _ = oracle.transfer_layers(hz.oracle_pool(src), s, hz.oracle_pool(exp), d, stop)
    assert rc == oracle.OK
    return src, dst, s, d, exp


def _run_transfer(src, dst, s, d, n, st, **kw):
    kvx.stream(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst),
               hz.dev_i32(d), n, None, hz.workspace(n), st, buf_bytes=0, **kw)


# ---- every layer ready: the same bytes as the oracle ---------------------------------------

@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [1, 777, 2500])
@pytest.mark.parametrize("ready", ["none", "device_words"])
def test_stream_transfer_all_ready(kind, n, ready, grid):
    src, dst, s, d, exp = _transfer_case(kind, n, seed=n)
    st = _status()
    rw = None
    if ready == "device_words":
        rw = torch.full((SH["L"],), 3, dtype=torch.int32, device="cuda")
    _run_transfer(src, dst, s, d, n, st, layer_ready=rw, ready_value=3, max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.OK and v[1] == 0 and v[3] == 1, v
    hz.assert_same_bytes(dst.readback(), exp.host, f"stream transfer {kind} n={n}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


@pytest.mark.parametrize("kind", KINDS)
def test_stream_gather_and_scatter(kind, grid):
    n = 1500
    g = _rng(77)
    src = _pool(kind, "normal", g)
    s = _slots(78, n, src.num_slots)
    rc, want, _ = oracle.gather(hz.oracle_pool(src), s)
    assert rc == oracle.OK
    buf = hz.make_mirror("buffer", SH["L"], SH["H"], SH["D"], SH["dtype"], n_tokens=n,
                         fill="sentinel").to_device()
    st = _status()
    kvx.stream(kvx.OP_GATHER, hz.kvx_layout(src), hz.dev_i32(s), None, None, n,
               hz.GUARD + buf.dev.data_ptr(), hz.workspace(n), st, buf_bytes=len(want),
               max_ctas=grid)
    torch.cuda.synchronize()
    assert st.cpu().tolist()[0:2] == [kvx.OK, 0]
    exp_buf = buf.host.copy()
    exp_buf[hz.GUARD:hz.GUARD + len(want)] = want
    hz.assert_same_bytes(buf.readback(), exp_buf, f"stream gather {kind}")

    # scatter the gathered rows into a fresh pool at other slots
    dst = _pool(kind, "sentinel", salt=9)
    d = _slots(79, n, dst.num_slots)
    exp = _expected_pool(kind, dst.num_slots, 9)
    assert oracle.scatter(hz.oracle_pool(exp), d, want)[0] == oracle.OK
    st2 = _status()
    kvx.stream(kvx.OP_SCATTER, None, None, hz.kvx_layout(dst), hz.dev_i32(d), n,
               hz.GUARD + buf.dev.data_ptr(), hz.workspace(n), st2, buf_bytes=len(want),
               max_ctas=grid)
    torch.cuda.synchronize()
    assert st2.cpu().tolist()[0:2] == [kvx.OK, 0]
    hz.assert_same_bytes(dst.readback(), exp.host, f"stream scatter {kind}")


@pytest.mark.parametrize("engine", ENGINE_LIST, **ENGINES)
def test_stream_2k_rows_few_ctas(engine):
    """2 KiB rows (one token per warp) on a grid capped at 3 CTAs: every warp (every thread of
    the bulk form) walks many layers' items."""
    n = 2048
    src, dst, s, d, exp = _transfer_case("planes", n, sh=SH2K, seed=90)
    st = _status()
    done = _pinned_i32([0])
    kvx.set_copy_engine(engine)
    try:
        _run_transfer(src, dst, s, d, n, st, max_ctas=3, host_done=done)
        torch.cuda.synchronize()
    finally:
        kvx.set_copy_engine(kvx.ENGINE_AUTO)
    assert st.cpu().tolist()[0:2] == [kvx.OK, 0] and st[3].item() == 1
    assert int(done[0]) == 1
    hz.assert_same_bytes(dst.readback(), exp.host, "stream 2k rows, 3 CTAs")


SH_LONG = dict(L=3, H=3, D=768, dtype="bf16")  # 4608-byte rows of three 1536-byte head vectors


@pytest.mark.parametrize("kinds", [("planes", "hnd"), ("hnd", "slot_major"), ("hnd", "hnd")])
@pytest.mark.parametrize("max_ctas", [1, 8])
@pytest.mark.parametrize("engine", [kvx.ENGINE_AUTO, kvx.ENGINE_BULK], ids=["registers", "bulk"])
def test_stream_bulk_rows_longer_than_a_stage(kinds, max_ctas, engine):
    # (rows longer than a stage take the register form under the default engine)
    """The bulk form's rows longer than its 2 KiB stage, in three pieces whose boundaries cut
    head vectors (1536 bytes, not a power of two) on HND sides: every piece reaches the right
    bytes of the right pages."""
    n = 300
    g = _rng(130 + max_ctas + len(kinds[0]) + 3 * len(kinds[1]))
    src = _pool(kinds[0], "normal", g, num_slots=1024, sh=SH_LONG)
    dst = _pool(kinds[1], "sentinel", salt=13, num_slots=1024, sh=SH_LONG)
    exp = _expected_pool(kinds[1], 1024, 13, sh=SH_LONG)
    s = _slots(131, n, 1024)
    d = _slots(132, n, 1024)
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == oracle.OK
    st = _status()
    ready = torch.ones(SH_LONG["L"], dtype=torch.int32, device="cuda")
    kvx.set_copy_engine(engine)
    try:
        _run_transfer(src, dst, s, d, n, st, layer_ready=ready, ready_value=1, max_ctas=max_ctas)
        torch.cuda.synchronize()
    finally:
        kvx.set_copy_engine(kvx.ENGINE_AUTO)
    v = st.cpu().tolist()
    assert v[0:2] == [kvx.OK, 0] and v[3] == 1, v
    hz.assert_same_bytes(dst.readback(), exp.host, f"long rows {kinds}, {max_ctas} CTAs")
    hz.assert_same_bytes(src.readback(), src.host, "source")


def test_stream_n0_and_out_of_range(grid):
    src, dst, s, d, exp = _transfer_case("planes", 300, seed=120)
    st = _status()
    _run_transfer(src, dst, s, d, 0, st, max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.OK and v[1] == 0 and v[3] == 1, v

    before = dst.readback()
    d_bad = d.copy()
    d_bad[-1] = dst.num_slots  # one past the end: nothing may move
    st = _status()
    _run_transfer(src, dst, s, d_bad, 300, st, max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_OUT_OF_RANGE and v[1] == SH["L"] and v[3] == 1, v
    hz.assert_same_bytes(dst.readback(), before, "out of range: nothing moved")


# ---- layers raised by the host after the launch --------------------------------------------

@pytest.mark.parametrize("sh", [SH, SH2K], ids=["256B", "2KiB"])
def test_stream_layers_raised_late(sh, grid):
    n = 1024
    src, dst, s, d, exp = _transfer_case("planes", n, sh=sh, seed=140)
    ready = _pinned_i32([0] * sh["L"])
    done = _pinned_i32([0])
    st = _status()
    ws, sd, dd = hz.workspace(n), hz.dev_i32(s), hz.dev_i32(d)
    torch.cuda.synchronize()
    kvx.stream(kvx.OP_TRANSFER, hz.kvx_layout(src), sd, hz.kvx_layout(dst), dd, n, None, ws, st,
               layer_ready=ready, ready_value=1, wait_ns=2_000_000_000, host_done=done,
               max_ctas=grid, buf_bytes=0)
    for layer in range(sh["L"]):
        time.sleep(0.01)
        assert int(done[0]) == 0, f"finished before layer {layer} was raised"
        ready[layer] = 1
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.OK and v[1] == 0 and v[3] == 1, v
    assert int(done[0]) == 1
    hz.assert_same_bytes(dst.readback(), exp.host, "layers raised late")


# ---- a layer never raised: bounded wait, KVX_ERR_TIMEOUT -----------------------------------

@pytest.mark.parametrize("kind", ["planes", "slot_major"])
@pytest.mark.parametrize("k", [0, 4])
def test_stream_timeout_at_layer(kind, k, grid):
    n = 900
    src, dst, s, d, exp = _transfer_case(kind, n, seed=160 + k, stop=k)
    ready = _pinned_i32([1 if layer < k else 0 for layer in range(SH["L"])])
    done = _pinned_i32([0])
    st = _status()
    t0 = time.perf_counter()
    _run_transfer(src, dst, s, d, n, st, layer_ready=ready, ready_value=1, wait_ns=30_000_000,
                  host_done=done, max_ctas=grid)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_TIMEOUT and v[1] == SH["L"] - k and v[3] == 1, v
    assert int(done[0]) == 1
    assert 0.02 < elapsed < 5.0, elapsed
    hz.assert_same_bytes(dst.readback(), exp.host, f"timeout at layer {k}")


# ---- cancellation through the epoch word ---------------------------------------------------

def test_stream_cancel_while_waiting(grid):
    n, k = 1200, 3
    src, dst, s, d, exp = _transfer_case("planes", n, seed=180, stop=k)
    ready = _pinned_i32([1 if layer < k else 0 for layer in range(SH["L"])])
    epoch = _pinned_i32([41])
    done = _pinned_i32([0])
    st = _status()
    ws, sd, dd = hz.workspace(n), hz.dev_i32(s), hz.dev_i32(d)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvx.stream(kvx.OP_TRANSFER, hz.kvx_layout(src), sd, hz.kvx_layout(dst), dd, n, None, ws, st,
               layer_ready=ready, ready_value=1, epoch_word=epoch, epoch=41,
               wait_ns=5_000_000_000, host_done=done, max_ctas=grid, buf_bytes=0)
    time.sleep(0.05)
    assert int(done[0]) == 0  # still waiting for layer k
    epoch[0] = 42             # the receiver gives up on the request
    deadline = time.perf_counter() + 4.0
    while int(done[0]) == 0 and time.perf_counter() < deadline:
        time.sleep(0.001)
    assert int(done[0]) == 1, "the kernel did not acknowledge the cancellation"
    elapsed = time.perf_counter() - t0
    torch.cuda.synchronize()
    assert elapsed < 4.0, elapsed  # well inside the 5 s wait bound
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_CANCELLED and v[1] == SH["L"] - k and v[3] == 1, v
    hz.assert_same_bytes(dst.readback(), exp.host, "cancelled while waiting")


def test_stream_cancelled_before_launch(grid):
    n = 500
    src, dst, s, d, _ = _transfer_case("hnd", n, seed=200)
    before = dst.readback()
    epoch = torch.tensor([7], dtype=torch.int32, device="cuda")  # device epoch word
    st = _status()
    _run_transfer(src, dst, s, d, n, st, epoch_word=epoch, epoch=6, max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_CANCELLED and v[1] == SH["L"] and v[3] == 1, v
    hz.assert_same_bytes(dst.readback(), before, "cancelled before launch: nothing moved")


def test_stream_pageable_control_word_refused():
    n = 10
    src, dst, s, d, _ = _transfer_case("planes", n, seed=220)
    ready = np.ones(SH["L"], dtype=np.int32)  # pageable host memory
    with pytest.raises(kvx.KvxError) as e:
        _run_transfer(src, dst, s, d, n, _status(), layer_ready=ready)
    assert e.value.code == kvx.ERR_INVALID_ARG


# ---- destination pages handed to another request (per-page owner epochs) -------------------

EP = 8  # slots per epoch page


def _owners(num_slots, taken, epoch=41, other=77):
    """Owner epoch per destination page: `epoch`, except the pages in `taken`."""
    e = np.full((num_slots + EP - 1) // EP, epoch, dtype=np.int32)
    e[list(taken)] = other
    return e


def test_stream_pages_reassigned_before_launch(grid):
    n = 1200
    src, dst, s, d, _ = _transfer_case("planes", n, seed=240)
    taken = sorted(set((d[[3, 500, 999, 1199]] // EP).tolist()))
    owners = _owners(dst.num_slots, taken)
    exp = _expected_pool("planes", dst.num_slots, 5)
    rc, w = oracle.transfer_owned(hz.oracle_pool(src), s, hz.oracle_pool(exp), d, SH["L"], owners,
                                  EP, 41)
    dropped = int(np.isin(d // EP, taken).sum())
    assert rc == oracle.OK and w == (n - dropped) * 2 * SH["L"] * src.R
    st = _status()
    _run_transfer(src, dst, s, d, n, st, dst_page_epochs=torch.from_numpy(owners).cuda(),
                  epoch_page=EP, epoch=41, max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_CANCELLED and v[1] == SH["L"] and v[3] == 1, v
    hz.assert_same_bytes(dst.readback(), exp.host, "rows of reassigned pages dropped")


def test_stream_pages_reassigned_while_waiting(grid):
    """Layers below k are raised; while the kernel waits for layer k the receiver hands some
    destination pages to another request (pinned host owner words), then the producer raises the
    rest: rows of layers < k are all written, rows of later layers only into owned pages."""
    n, k = 1000, 3
    src, dst, s, d, _ = _transfer_case("planes", n, seed=260)
    taken = sorted(set((d[[0, 17, 640, 999]] // EP).tolist()))
    owners = torch.from_numpy(_owners(dst.num_slots, [])).pin_memory()
    ready = _pinned_i32([1 if l < k else 0 for l in range(SH["L"])])
    done = _pinned_i32([0])
    st = _status()
    ws, sd, dd = hz.workspace(n), hz.dev_i32(s), hz.dev_i32(d)
    torch.cuda.synchronize()
    kvx.stream(kvx.OP_TRANSFER, hz.kvx_layout(src), sd, hz.kvx_layout(dst), dd, n, None, ws, st,
               layer_ready=ready, ready_value=1, epoch=41, dst_page_epochs=owners, epoch_page=EP,
               wait_ns=5_000_000_000, host_done=done, max_ctas=grid, buf_bytes=0)
    time.sleep(0.05)
    assert int(done[0]) == 0  # still waiting for layer k
    for pg in taken:
        owners[pg] = 77
    for layer in range(k, SH["L"]):
        ready[layer] = 1
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_CANCELLED and v[1] == SH["L"] - k and v[3] == 1, v
    exp = _expected_pool("planes", dst.num_slots, 5)
    assert oracle.transfer_owned(hz.oracle_pool(src), s, hz.oracle_pool(exp), d, SH["L"],
                                 owners.numpy(), EP, 41)[0] == oracle.OK
    assert oracle.transfer_layers(hz.oracle_pool(src), s, hz.oracle_pool(exp), d, k)[0] == oracle.OK
    hz.assert_same_bytes(dst.readback(), exp.host, "late rows of reassigned pages dropped")


def test_stream_all_pages_owned_moves_everything(grid):
    n = 700
    src, dst, s, d, exp = _transfer_case("hnd", n, seed=280)
    owners = torch.from_numpy(_owners(dst.num_slots, [])).cuda()
    st = _status()
    _run_transfer(src, dst, s, d, n, st, dst_page_epochs=owners, epoch_page=EP, epoch=41,
                  max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.OK and v[1] == 0 and v[3] == 1, v
    hz.assert_same_bytes(dst.readback(), exp.host, "every page owned")


@pytest.mark.parametrize("n", [2048, 8192])
def test_stream_cancelled_before_launch_while_validating(n, grid):
    """The epoch word changed before the call: every CTA stops at its first look, often while the
    one-CTA validation (which initialises all four status words) is still running.  Over 100
    calls each must report CANCELLED with every layer pending and the done word set, and leave
    the pool untouched."""
    g = _rng(210)
    src = _pool("planes", "normal", g, num_slots=16384)
    dst = _pool("planes", "sentinel", salt=5, num_slots=16384)
    s, d = _slots(211, n, 16384), _slots(212, n, 16384)
    before = dst.readback()
    epoch = torch.tensor([7], dtype=torch.int32, device="cuda")
    sd, dd, ws = hz.dev_i32(s), hz.dev_i32(d), hz.workspace(n)
    sts = [_status() for _ in range(100)]
    for st in sts:
        kvx.stream(kvx.OP_TRANSFER, hz.kvx_layout(src), sd, hz.kvx_layout(dst), dd, n, None, ws,
                   st, epoch_word=epoch, epoch=6, max_ctas=grid, buf_bytes=0)
    torch.cuda.synchronize()
    got = [st.cpu().tolist() for st in sts]
    bad = [v for v in got if not (v[0] == kvx.ERR_CANCELLED and v[1] == SH["L"] and v[3] == 1)]
    assert not bad, (len(bad), bad[:5])
    hz.assert_same_bytes(dst.readback(), before, "cancelled before launch: nothing moved")
