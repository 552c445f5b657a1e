"""kvx_stream_reshard -- a whole TP reshard, layer-streamed and cancellable -- against the
oracle, through the C ABI (GPU).

Expected pools come from the oracle's kvxo_reshard: of the whole pools when every layer moves,
of the pools restricted to their first k layers (the plane lists cut after layer k) when the
move stops at layer k, and of the token subset whose destination pages are still owned when
pages are reassigned.  Every failure is made on the host (ready words nothing raises, an epoch
word the host changes, owner words changed before or during the move), and every device wait
is bounded, so no case can hang the GPU.  Each case runs on the row grid and on a capped
persistent grid of 24 CTAs.
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

L, D, DT = 5, 64, "fp16"
HEADS = 8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


def _rng(k):
    return np.random.Generator(np.random.PCG64(15000 + k))


# max_ctas: 0 = the row grid (default); 24 = a capped persistent grid of 24 CTAs
@pytest.fixture(params=[0, 24], ids=["rowgrid", "persistent24"])
def grid(request):
    return request.param


def _pinned(values):
    return torch.tensor(values, dtype=torch.int32).pin_memory()


def _status():
    return torch.full((4,), -1, dtype=torch.int32, device="cuda")


def _cut(pool: oracle.Pool, k: int) -> oracle.Pool:
    """The same pool seen through its first k layers only."""
    return oracle.Pool(k, pool.kv_heads, pool.head_dim, pool.elem_bytes, pool.kind,
                       pool.num_slots, pool.planes[:pool.kv_planes * k], pool.slot_stride,
                       pool.page_size, pool.kv_planes)


class Case:
    def __init__(self, p_tp, d_tp, n, seed, src_kind="hnd", dst_kind="planes", num=4096):
        g = _rng(seed)
        sh = lambda t: HEADS // t if t <= HEADS else 1
        ps = lambda kind: 16 if kind == "hnd" else 1
        self.p = [hz.make_mirror(src_kind, L, sh(p_tp), D, DT, num, ps(src_kind), "normal", g)
                  .to_device() for _ in range(p_tp)]
        self.d = [hz.make_mirror(dst_kind, L, sh(d_tp), D, DT, num, ps(dst_kind), "sentinel",
                                 salt=r).to_device() for r in range(d_tp)]
        self.exp = [hz.make_mirror(dst_kind, L, sh(d_tp), D, DT, num, ps(dst_kind), "sentinel",
                                   salt=r) for r in range(d_tp)]
        self.parts = kvx.tp_plan(HEADS, p_tp, d_tp)
        self.n, self.num = n, num
        self.s = inputs.distinct_slots(g, n, num)
        self.dslots = inputs.distinct_slots(g, n, num)
        self.ws, self.sd, self.dd = hz.workspace(n), hz.dev_i32(self.s), hz.dev_i32(self.dslots)

    def expect(self, layers=L, keep=None):
        if layers == 0:
            return  # nothing moves
        s, d = self.s, self.dslots
        if keep is not None:
            s, d = s[keep], d[keep]
        rc, _ = oracle.reshard([_cut(hz.oracle_pool(m), layers) for m in self.p], s,
                               [_cut(hz.oracle_pool(m), layers) for m in self.exp], d,
                               self.parts, len(s))
        assert rc == oracle.OK

    def run(self, st, **kw):
        kvx.stream_reshard([hz.kvx_layout(m) for m in self.p], self.sd,
                           [hz.kvx_layout(m) for m in self.d], self.dd, self.parts, self.n,
                           self.ws, st, **kw)

    def check(self, what):
        for r, (m, e) in enumerate(zip(self.d, self.exp)):
            hz.assert_same_bytes(m.readback(), e.host, f"{what}: D rank {r}")
        for r, m in enumerate(self.p):
            hz.assert_same_bytes(m.readback(), m.host, f"{what}: P rank {r} (source)")


@pytest.mark.parametrize("p_tp,d_tp", [(8, 1), (4, 2), (1, 2), (2, 4)])
@pytest.mark.parametrize("n", [1, 700, 2600])
def test_all_layers_ready(p_tp, d_tp, n, grid):
    c = Case(p_tp, d_tp, n, seed=p_tp * 10 + d_tp + n)
    c.expect()
    st = _status()
    words = torch.ones(L, dtype=torch.int32, device="cuda")
    c.run(st, layer_ready=words, ready_value=1, max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0:2] == [kvx.OK, 0] and v[3] == 1, v
    c.check(f"P TP {p_tp} -> D TP {d_tp}, n={n}, {grid} CTAs")


def test_layers_raised_late(grid):
    c = Case(4, 2, 1500, seed=1)
    c.expect()
    ready, done = _pinned([0] * L), _pinned([0])
    st = _status()
    torch.cuda.synchronize()
    c.run(st, layer_ready=ready, ready_value=1, wait_ns=2_000_000_000, host_done=done,
          max_ctas=grid)
    for layer in range(L):
        time.sleep(0.01)
        assert int(done[0]) == 0, f"finished before layer {layer} was raised"
        ready[layer] = 1
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0:2] == [kvx.OK, 0] and v[3] == 1, v
    assert int(done[0]) == 1
    c.check("layers raised late")


@pytest.mark.parametrize("k", [0, 3])
def test_timeout_at_layer(k, grid):
    c = Case(8, 1, 900, seed=10 + k)
    c.expect(layers=k)
    ready, done = _pinned([1 if layer < k else 0 for layer in range(L)]), _pinned([0])
    st = _status()
    t0 = time.perf_counter()
    c.run(st, layer_ready=ready, ready_value=1, wait_ns=30_000_000, host_done=done, max_ctas=grid)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_TIMEOUT and v[1] == L - k and v[3] == 1, v
    assert int(done[0]) == 1
    assert 0.02 < elapsed < 5.0, elapsed
    c.check(f"timeout at layer {k}")


def test_cancel_while_waiting(grid):
    k = 2
    c = Case(2, 4, 1200, seed=20)
    c.expect(layers=k)
    ready = _pinned([1 if layer < k else 0 for layer in range(L)])
    epoch, done = _pinned([5]), _pinned([0])
    st = _status()
    torch.cuda.synchronize()
    c.run(st, layer_ready=ready, ready_value=1, epoch_word=epoch, epoch=5,
          wait_ns=5_000_000_000, host_done=done, max_ctas=grid)
    time.sleep(0.05)
    assert int(done[0]) == 0  # waiting for layer k
    epoch[0] = 6
    deadline = time.perf_counter() + 4.0
    while int(done[0]) == 0 and time.perf_counter() < deadline:
        time.sleep(0.001)
    assert int(done[0]) == 1, "the cancellation was not acknowledged"
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_CANCELLED and v[1] == L - k and v[3] == 1, v
    c.check("cancelled while waiting")


def test_cancelled_before_launch_moves_nothing(grid):
    c = Case(8, 1, 600, seed=30)
    epoch = _pinned([9])
    st = _status()
    c.run(st, epoch_word=epoch, epoch=8, max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_CANCELLED and v[1] == L and v[3] == 1, v
    c.check("cancelled before launch")


@pytest.mark.parametrize("when", ["before", "while_waiting"])
def test_destination_pages_reassigned(when, grid):
    """Owner epochs per 16-slot destination page: rows into pages given to another request are
    dropped (KVX_ERR_CANCELLED), every other row moves."""
    k = 2
    c = Case(4, 2, 1000, seed=40 + len(when))
    pages = c.num // 16
    # pinned host words: the host changes them while the kernel runs, without the stream
    owners = torch.full((pages,), 3, dtype=torch.int32).pin_memory()
    taken = np.arange(0, pages, 5)
    keep = ~np.isin(c.dslots // 16, taken)
    st = _status()
    if when == "before":
        owners[torch.from_numpy(taken)] = 4
        c.expect(keep=keep)
        c.run(st, dst_page_epochs=owners, epoch_page=16, epoch=3, max_ctas=grid)
        torch.cuda.synchronize()
        v = st.cpu().tolist()
        assert v[0] == kvx.ERR_CANCELLED and v[3] == 1, v
    else:
        # layers below k move with every page owned; then pages are reassigned and the rest
        # of the layers are raised: their rows into reassigned pages are dropped
        ready, done = _pinned([1 if layer < k else 0 for layer in range(L)]), _pinned([0])
        rc, _ = oracle.reshard([_cut(hz.oracle_pool(m), k) for m in c.p], c.s,
                               [_cut(hz.oracle_pool(m), k) for m in c.exp], c.dslots, c.parts,
                               c.n)
        assert rc == oracle.OK
        torch.cuda.synchronize()
        c.run(st, layer_ready=ready, ready_value=1, wait_ns=5_000_000_000, host_done=done,
              dst_page_epochs=owners, epoch_page=16, epoch=3, max_ctas=grid)
        time.sleep(0.05)
        owners[torch.from_numpy(taken)] = 4
        time.sleep(0.01)  # the owner words are visible before any later layer is raised
        for layer in range(k, L):
            ready[layer] = 1
        torch.cuda.synchronize()
        v = st.cpu().tolist()
        assert v[0] == kvx.ERR_CANCELLED and v[3] == 1, v
        # rows of layers >= k: only into owned pages
        full = [_cut(hz.oracle_pool(m), L) for m in c.exp]
        rc, _ = oracle.reshard([hz.oracle_pool(m) for m in c.p], c.s[keep], full, c.dslots[keep],
                               c.parts, int(keep.sum()))
        assert rc == oracle.OK
    c.check(f"pages reassigned {when}")


def test_n0_and_out_of_range(grid):
    c = Case(2, 1, 0, seed=50)
    st = _status()
    c.run(st, max_ctas=grid)
    torch.cuda.synchronize()
    assert st.cpu().tolist()[:2] == [kvx.OK, 0] and st.cpu().tolist()[3] == 1
    c = Case(2, 1, 800, seed=51)
    c.dslots[400] = c.num
    c.dd = hz.dev_i32(c.dslots)
    st = _status()
    c.run(st, max_ctas=grid)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_OUT_OF_RANGE and v[1] == L and v[3] == 1, v
    c.check("nothing moved")
