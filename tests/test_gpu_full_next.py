"""The layer-streamed, head-range and format moves at the sizes bench.py times (GPU), checked
byte for byte against the CPU oracle over the whole destination.

As in test_gpu_full.py: each source pool is read back into host memory before the move, the
oracle runs over that host copy with the real slot lists (kvxo_transfer_layers for the stopped
streamed move, kvxo_move_heads and kvxo_reshard for the TP moves, kvxo_transfer for the
formats), and every byte of every destination pool, between 64 KiB sentinel guard bands, is
compared with the oracle's.
"""
import numpy as np
import pytest

import oracle
from tests import fullsize, inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SENT = 0x7FC1  # bf16 quiet NaN
GUARD = fullsize.GUARD
L, H, D, N, S = 36, 8, 128, 2048, 65536  # the 288 MiB request and its pools
R, P = H * D * 2, 72


@pytest.fixture(scope="module")
def stager():
    return fullsize.Stager()


@pytest.fixture(autouse=True)
def _clean():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _rows(arr, layers, heads, dim, elem, num_slots, kv_planes=2):
    """Oracle view of per-plane token-row pools laid out plane after plane after a guard band."""
    rb = heads * dim * elem
    planes = kv_planes * layers
    return oracle.Pool(layers, heads, dim, elem, oracle.TOKEN_ROWS, num_slots,
                       [(arr, GUARD + p * num_slots * rb) for p in range(planes)], rb,
                       kv_planes=kv_planes)


def _hnd(arr, layers, heads, dim, num_slots, ps=16):
    pb = num_slots * heads * dim * 2
    return oracle.Pool(layers, heads, dim, 2, oracle.HND_PAGES, num_slots,
                       [(arr, GUARD + p * pb) for p in range(2 * layers)], 0, ps)


@pytest.mark.parametrize("max_ctas", [0, 76], ids=["rowgrid", "capped76"])
def test_stream_full_size_timeout_at_layer_20(stager, max_ctas):
    """The headline request through kvx_stream with ready words in pinned host memory, layers
    0..19 raised and 20.. never: KVX_ERR_TIMEOUT, and the whole destination pool equals the
    oracle's transfer of layers 0..19 (every later layer untouched); on the row grid and on a
    persistent grid capped at half the SMs."""
    k = 20
    fullsize.require_host_bytes(3 * (P * S * R + 2 * GUARD))
    src_all, src = fullsize.guarded((P, S, H, D), torch.bfloat16, "normal", SENT, inputs.seed(2, 0))
    dst_all, dst = fullsize.guarded((P, S, H, D), torch.bfloat16, "sentinel", SENT)
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N, S)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N, S)
    host_src = stager.to_host(src_all)
    sl = kvx.Layout(L, H, D, kvx.BF16, S, base=src, plane_stride=S * R)
    dl = kvx.Layout(L, H, D, kvx.BF16, S, base=dst, plane_stride=S * R)
    ready = torch.tensor([1 if l < k else 0 for l in range(L)], dtype=torch.int32).pin_memory()
    st = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvx.workspace_size(N), dtype=torch.uint8, device="cuda")
    kvx.stream(kvx.OP_TRANSFER, sl, _dev_i32(s), dl, _dev_i32(d), N, None, ws, st,
               layer_ready=ready, ready_value=1, wait_ns=50_000_000, buf_bytes=0,
               max_ctas=max_ctas)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_TIMEOUT and v[1] == L - k and v[3] == 1, v
    host_dst = fullsize.filled(P * S * R + 2 * GUARD, SENT)
    rc, w = oracle.transfer_layers(_rows(host_src, L, H, D, 2, S), s,
                                   _rows(host_dst, L, H, D, 2, S), d, k)
    assert rc == oracle.OK and w == N * 2 * k * R
    stager.assert_equal(dst_all, host_dst, "destination pool (layers < 20 moved)", R)
    stager.assert_equal(src_all, host_src, "source pool unchanged", R)


def test_tp_reshard_full_size(stager):
    """The headline request resharded from P TP 1 (one 8-head HND pool, page 16) to D TP 2 (two
    4-head token-row pools) with the plan kvx_tp_slice gives, one kvx_move_heads per pair."""
    NS = 32768
    src_all, p_pool = fullsize.guarded((P, NS // 16, H, 16, D), torch.bfloat16, "normal", SENT,
                                       inputs.seed(2, 0))
    d_pools = [fullsize.guarded((P, NS, H // 2, D), torch.bfloat16, "sentinel", SENT)
               for _ in range(2)]
    pl = kvx.Layout(L, H, D, kvx.BF16, NS, kind=kvx.HND_PAGED, page_size=16, base=p_pool,
                    plane_stride=NS * R)
    dls = [kvx.Layout(L, H // 2, D, kvx.BF16, NS, base=t, plane_stride=NS * R // 2)
           for _, t in d_pools]
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N, NS)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N, NS)
    host_src = stager.to_host(src_all)
    ws = torch.empty(kvx.workspace_size(N), dtype=torch.uint8, device="cuda")
    for dr in range(2):
        sh0, dh0, nh = kvx.tp_slice(H, 1, 0, 2, dr)
        assert (sh0, dh0, nh) == (4 * dr, 0, 4)
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        kvx.move_heads(kvx.OP_TRANSFER, pl, _dev_i32(s), sh0, dls[dr], _dev_i32(d), dh0, nh, N,
                       None, ws, st, buf_bytes=0)
        torch.cuda.synchronize()
        assert int(st.item()) == kvx.OK
        host_dst = fullsize.filled(P * NS * R // 2 + 2 * GUARD, SENT)
        rc, _, _ = oracle.move_heads(2, _hnd(host_src, L, H, D, NS), s, sh0,
                                     _rows(host_dst, L, H // 2, D, 2, NS), d, dh0, nh, N)
        assert rc == oracle.OK
        stager.assert_equal(d_pools[dr][0], host_dst, f"D rank {dr} pool", R // 2)


def test_reshard_one_call_full_size(stager):
    """The headline request resharded from P TP 8 (eight 1-head HND pools, page 16) to D TP 1
    (one 8-head token-row pool) in one kvx_reshard call with the kvx_tp_plan plan, as the
    bench's tp workload times it, against the oracle's kvxo_reshard of the same parts."""
    NS = 32768
    p_pools = [fullsize.guarded((P, NS // 16, 1, 16, D), torch.bfloat16, "normal", SENT,
                                inputs.seed(2, 0) + r) for r in range(8)]
    dst_all, d_pool = fullsize.guarded((P, NS, H, D), torch.bfloat16, "sentinel", SENT)
    pls = [kvx.Layout(L, 1, D, kvx.BF16, NS, kind=kvx.HND_PAGED, page_size=16, base=t,
                      plane_stride=NS * D * 2) for _, t in p_pools]
    dl = kvx.Layout(L, H, D, kvx.BF16, NS, base=d_pool, plane_stride=NS * R)
    parts = kvx.tp_plan(H, 8, 1)
    assert parts == [(r, 0, 0, r, 1) for r in range(8)]
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N, NS)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N, NS)
    host_srcs = [stager.to_host(whole) for whole, _ in p_pools]
    ws = torch.empty(kvx.workspace_size(N), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.reshard(pls, _dev_i32(s), [dl], _dev_i32(d), parts, N, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    host_dst = fullsize.filled(P * NS * R + 2 * GUARD, SENT)
    rc, _ = oracle.reshard([_hnd(x, L, 1, D, NS) for x in host_srcs], s,
                           [_rows(host_dst, L, H, D, 2, NS)], d, parts, N)
    assert rc == oracle.OK
    stager.assert_equal(dst_all, host_dst, "D pool", R)


@pytest.mark.parametrize("elem", [2, 1], ids=["bf16", "fp8"])
def test_mla_full_size(stager, elem):
    """DeepSeek-V2-Lite-shaped latent rows (27 planes x 576 elements), 16,384 tokens, the
    bench's formats case: the whole destination pool against the oracle."""
    Lm, Dm, n, NS = 27, 576, 16384, 65536
    Rm = Dm * elem
    src_all, src = fullsize.guarded((Lm, NS, Rm), torch.uint8, "bytes", 0x7F7F, 7)
    dst_all, dst = fullsize.guarded((Lm, NS, Rm), torch.uint8, "sentinel", 0x7F7F)
    dt = kvx.BF16 if elem == 2 else kvx.FP8
    sl = kvx.Layout(Lm, 1, Dm, dt, NS, base=src, plane_stride=NS * Rm, kv_planes=1)
    dl = kvx.Layout(Lm, 1, Dm, dt, NS, base=dst, plane_stride=NS * Rm, kv_planes=1)
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), n, NS)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), n, NS)
    host_src = stager.to_host(src_all)
    ws = torch.empty(kvx.workspace_size(n), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.transfer(sl, _dev_i32(s), dl, _dev_i32(d), n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    host_dst = fullsize.filled(Lm * NS * Rm + 2 * GUARD, 0x7F7F)
    rc, w = oracle.transfer(_rows(host_src, Lm, 1, Dm, elem, NS, kv_planes=1), s,
                            _rows(host_dst, Lm, 1, Dm, elem, NS, kv_planes=1), d)
    assert rc == oracle.OK and w == n * Lm * Rm
    stager.assert_equal(dst_all, host_dst, "latent destination pool", Rm)


def test_narrow_rows_full_size(stager):
    """200-byte rows (one head of head_dim 100 fp16), 16,384 tokens x 72 planes, through the
    narrow kernel with 8-byte accesses (the bench's formats case)."""
    Ln, Dn, n, NS = 36, 100, 16384, 65536
    Rn, Pn = Dn * 2, 72
    src_all, src = fullsize.guarded((Pn, NS, Rn), torch.uint8, "bytes", 0x7E7E, 8)
    dst_all, dst = fullsize.guarded((Pn, NS, Rn), torch.uint8, "sentinel", 0x7E7E)
    sl = kvx.Layout(Ln, 1, Dn, kvx.F16, NS, base=src, plane_stride=NS * Rn)
    dl = kvx.Layout(Ln, 1, Dn, kvx.F16, NS, base=dst, plane_stride=NS * Rn)
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), n, NS)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), n, NS)
    host_src = stager.to_host(src_all)
    ws = torch.empty(kvx.workspace_size(n), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.transfer(sl, _dev_i32(s), dl, _dev_i32(d), n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    host_dst = fullsize.filled(Pn * NS * Rn + 2 * GUARD, 0x7E7E)
    rc, _ = oracle.transfer(_rows(host_src, Ln, 1, Dn, 2, NS), s, _rows(host_dst, Ln, 1, Dn, 2, NS), d)
    assert rc == oracle.OK
    stager.assert_equal(dst_all, host_dst, "narrow-row destination pool", Rn)
