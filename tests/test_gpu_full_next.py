"""The layer-streamed, head-range and format moves at the sizes bench.py times (GPU).

As in test_gpu_full.py: pools filled on the device (seeded torch.randn; destinations with a
quiet-NaN sentinel); each test checks the status words, sampled outputs computed one by one by
the CPU oracle from the sampled source rows read back into small host pools, and properties
that hold at any size (exactly the named destination rows changed).
"""
import numpy as np
import pytest

import oracle
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SENT = 0x7FC1  # bf16 quiet NaN
L, H, D, N, S = 36, 8, 128, 2048, 65536  # the 288 MiB request and its pools
R, P = H * D * 2, 72


@pytest.fixture(autouse=True)
def _clean():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _pool(shape, fill, seed=0):
    t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    if fill == "normal":
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        torch.randn(t.shape, dtype=t.dtype, device="cuda", generator=g, out=t)
    else:
        t.view(torch.int16).fill_(SENT)
    return t


def _host(t):
    return np.ascontiguousarray(t.cpu().view(torch.int16).numpy()).view(np.uint16)


def _sample(n, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return np.unique(np.concatenate([[0, n - 1], g.choice(n, k, replace=False)]))


def _changed(pool, slots_per_plane):
    """Per plane p (first axis), which slots differ from the sentinel anywhere in the row."""
    return torch.stack([(pool[p].view(torch.int16).reshape(pool.shape[1], -1) != SENT).any(dim=1)
                        for p in range(pool.shape[0])])


@pytest.mark.parametrize("max_ctas", [0, 76], ids=["rowgrid", "capped76"])
def test_stream_full_size_timeout_at_layer_20(max_ctas):
    """The headline request through kvx_stream with ready words in pinned host memory, layers
    0..19 raised and 20.. never: KVX_ERR_TIMEOUT, layers below 20 moved (sampled rows equal the
    oracle's layer-range transfer), every row of the later layers untouched; on the row grid and
    on a persistent grid capped at half the SMs."""
    k = 20
    src = _pool((P, S, H, D), "normal", inputs.seed(2, 0))
    dst = _pool((P, S, H, D), "sentinel")
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N, S)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N, S)
    sl = kvx.Layout(L, H, D, kvx.BF16, S, base=src, plane_stride=S * R)
    dl = kvx.Layout(L, H, D, kvx.BF16, S, base=dst, plane_stride=S * R)
    ready = torch.tensor([1 if l < k else 0 for l in range(L)], dtype=torch.int32).pin_memory()
    st = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvx.workspace_size(N), dtype=torch.uint8, device="cuda")
    kvx.stream(kvx.OP_TRANSFER, sl, torch.from_numpy(s).cuda(), dl, torch.from_numpy(d).cuda(), N,
               None, ws, st, layer_ready=ready, ready_value=1, wait_ns=50_000_000, buf_bytes=0,
               max_ctas=max_ctas)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_TIMEOUT and v[1] == L - k and v[3] == 1, v
    samp = _sample(N, 254, 11)
    st_i = torch.from_numpy(s[samp]).long().cuda()
    dt_i = torch.from_numpy(d[samp]).long().cuda()
    m = len(samp)
    mini_src = _host(src[:, st_i])
    dst_host = np.full((P, m, H, D), SENT, dtype=np.uint16)
    planes_s = [(mini_src, p * m * R) for p in range(P)]
    planes_d = [(dst_host, p * m * R) for p in range(P)]
    rc, w = oracle.transfer_layers(oracle.Pool(L, H, D, 2, oracle.TOKEN_ROWS, m, planes_s, R),
                                   np.arange(m),
                                   oracle.Pool(L, H, D, 2, oracle.TOKEN_ROWS, m, planes_d, R),
                                   np.arange(m), k)
    assert rc == oracle.OK and w == m * 2 * k * R
    assert np.array_equal(_host(dst[:, dt_i]), dst_host), "sampled rows differ from the oracle"
    want = torch.zeros((P, S), dtype=torch.bool, device="cuda")
    want[: 2 * k, torch.from_numpy(d).long().cuda()] = True
    assert torch.equal(_changed(dst, S), want), "rows other than layers < 20 of the named slots changed"


def test_tp_reshard_full_size():
    """The headline request resharded from P TP 1 (one 8-head HND pool, page 16) to D TP 2 (two
    4-head token-row pools) with the plan kvx_tp_slice gives, one kvx_move_heads per pair."""
    NS = 32768
    p_pool = _pool((P, NS // 16, H, 16, D), "normal", inputs.seed(2, 0))
    d_pools = [_pool((P, NS, H // 2, D), "sentinel") for _ in range(2)]
    pl = kvx.Layout(L, H, D, kvx.BF16, NS, kind=kvx.HND_PAGED, page_size=16, base=p_pool,
                    plane_stride=NS * R)
    dls = [kvx.Layout(L, H // 2, D, kvx.BF16, NS, base=t, plane_stride=NS * R // 2) for t in d_pools]
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N, NS)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N, NS)
    s_d, d_d = torch.from_numpy(s).cuda(), torch.from_numpy(d).cuda()
    ws = torch.empty(kvx.workspace_size(N), dtype=torch.uint8, device="cuda")
    samp = _sample(N, 126, 12)
    m = len(samp)
    spage = torch.from_numpy(s[samp] // 16).long().cuda()
    soff = torch.from_numpy(s[samp] % 16).long().cuda()
    # the sampled tokens' source rows as a small HND-free host pool [P][m][H][D]
    rows = p_pool[:, spage, :, soff]  # advanced indexing: [m, P, H, D]
    mini_src = np.ascontiguousarray(_host(rows).transpose(1, 0, 2, 3))
    src_pool = oracle.Pool(L, H, D, 2, oracle.TOKEN_ROWS, m,
                           [(mini_src, p * m * R) for p in range(P)], R)
    for dr in range(2):
        sh0, dh0, nh = kvx.tp_slice(H, 1, 0, 2, dr)
        assert (sh0, dh0, nh) == (4 * dr, 0, 4)
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        kvx.move_heads(kvx.OP_TRANSFER, pl, s_d, sh0, dls[dr], d_d, dh0, nh, N, None, ws, st,
                       buf_bytes=0)
        torch.cuda.synchronize()
        assert int(st.item()) == kvx.OK
        dst_host = np.full((P, m, H // 2, D), SENT, dtype=np.uint16)
        dst_pool = oracle.Pool(L, H // 2, D, 2, oracle.TOKEN_ROWS, m,
                               [(dst_host, p * m * R // 2) for p in range(P)], R // 2)
        rc, _, _ = oracle.move_heads(2, src_pool, np.arange(m), sh0, dst_pool, np.arange(m), dh0,
                                     nh, m)
        assert rc == oracle.OK
        got = _host(d_pools[dr][:, torch.from_numpy(d[samp]).long().cuda()])
        assert np.array_equal(got, dst_host), f"D rank {dr}: sampled rows differ from the oracle"
        want = torch.zeros((P, NS), dtype=torch.bool, device="cuda")
        want[:, d_d.long()] = True
        assert torch.equal(_changed(d_pools[dr], NS), want), f"D rank {dr}: other rows changed"


def test_reshard_one_call_full_size():
    """The headline request resharded from P TP 8 (eight 1-head HND pools, page 16) to D TP 1
    (one 8-head token-row pool) in one kvx_reshard call with the kvx_tp_plan plan, as the
    bench's tp workload times it: sampled rows against the oracle's kvxo_reshard of the same
    parts on the sampled source rows, exact changed-row mask."""
    NS = 32768
    p_pools = [_pool((P, NS // 16, 1, 16, D), "normal", inputs.seed(2, 0) + r) for r in range(8)]
    d_pool = _pool((P, NS, H, D), "sentinel")
    pls = [kvx.Layout(L, 1, D, kvx.BF16, NS, kind=kvx.HND_PAGED, page_size=16, base=t,
                      plane_stride=NS * D * 2) for t in p_pools]
    dl = kvx.Layout(L, H, D, kvx.BF16, NS, base=d_pool, plane_stride=NS * R)
    parts = kvx.tp_plan(H, 8, 1)
    assert parts == [(r, 0, 0, r, 1) for r in range(8)]
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N, NS)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N, NS)
    s_d, d_d = torch.from_numpy(s).cuda(), torch.from_numpy(d).cuda()
    ws = torch.empty(kvx.workspace_size(N), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.reshard(pls, s_d, [dl], d_d, parts, N, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    samp = _sample(N, 126, 13)
    m = len(samp)
    spage = torch.from_numpy(s[samp] // 16).long().cuda()
    soff = torch.from_numpy(s[samp] % 16).long().cuda()
    minis = []
    for t in p_pools:  # the sampled tokens' source rows, [P][m][1][D] per P rank
        minis.append(np.ascontiguousarray(_host(t[:, spage, :, soff]).transpose(1, 0, 2, 3)))
    srcs = [oracle.Pool(L, 1, D, 2, oracle.TOKEN_ROWS, m, [(x, p * m * D * 2) for p in range(P)],
                        D * 2) for x in minis]
    dst_host = np.full((P, m, H, D), SENT, dtype=np.uint16)
    dst = oracle.Pool(L, H, D, 2, oracle.TOKEN_ROWS, m, [(dst_host, p * m * R) for p in range(P)],
                      R)
    rc, _ = oracle.reshard(srcs, np.arange(m), [dst], np.arange(m), parts, m)
    assert rc == oracle.OK
    got = _host(d_pool[:, torch.from_numpy(d[samp]).long().cuda()])
    assert np.array_equal(got, dst_host), "sampled rows differ from the oracle"
    want = torch.zeros((P, NS), dtype=torch.bool, device="cuda")
    want[:, d_d.long()] = True
    assert torch.equal(_changed(d_pool, NS), want), "other rows changed"


@pytest.mark.parametrize("elem", [2, 1], ids=["bf16", "fp8"])
def test_mla_full_size(elem):
    """DeepSeek-V2-Lite-shaped latent rows (27 planes x 576 elements), 16,384 tokens, the
    bench's formats case: sampled rows against the oracle, exact changed-row mask."""
    Lm, Dm, n, NS = 27, 576, 16384, 65536
    Rm = Dm * elem
    src = torch.randint(0, 255, (Lm, NS, Rm), dtype=torch.uint8, device="cuda",
                        generator=torch.Generator(device="cuda").manual_seed(7))
    dst = torch.full((Lm, NS, Rm), 0x7F, dtype=torch.uint8, device="cuda")
    dt = kvx.BF16 if elem == 2 else kvx.FP8
    sl = kvx.Layout(Lm, 1, Dm, dt, NS, base=src, plane_stride=NS * Rm, kv_planes=1)
    dl = kvx.Layout(Lm, 1, Dm, dt, NS, base=dst, plane_stride=NS * Rm, kv_planes=1)
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), n, NS)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), n, NS)
    ws = torch.empty(kvx.workspace_size(n), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.transfer(sl, torch.from_numpy(s).cuda(), dl, torch.from_numpy(d).cuda(), n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    samp = _sample(n, 510, 13)
    m = len(samp)
    mini_src = np.ascontiguousarray(src[:, torch.from_numpy(s[samp]).long().cuda()].cpu().numpy())
    dst_host = np.full((Lm, m, Rm), 0x7F, dtype=np.uint8)
    rc, w = oracle.transfer(
        oracle.Pool(Lm, 1, Dm, elem, oracle.TOKEN_ROWS, m, [(mini_src, p * m * Rm) for p in range(Lm)],
                    Rm, kv_planes=1), np.arange(m),
        oracle.Pool(Lm, 1, Dm, elem, oracle.TOKEN_ROWS, m, [(dst_host, p * m * Rm) for p in range(Lm)],
                    Rm, kv_planes=1), np.arange(m))
    assert rc == oracle.OK and w == m * Lm * Rm
    got = dst[:, torch.from_numpy(d[samp]).long().cuda()].cpu().numpy()
    assert np.array_equal(got, dst_host), "sampled latent rows differ from the oracle"
    changed = (dst != 0x7F).any(dim=2)
    want = torch.zeros((Lm, NS), dtype=torch.bool, device="cuda")
    want[:, torch.from_numpy(d).long().cuda()] = True
    # a random source row can hold 0x7F in every byte only with probability 256^-576
    assert torch.equal(changed, want), "rows other than the named ones changed"


def test_narrow_rows_full_size():
    """200-byte rows (one head of head_dim 100 fp16), 16,384 tokens x 72 planes, through the
    narrow kernel with 8-byte accesses (the bench's formats case)."""
    Ln, Dn, n, NS = 36, 100, 16384, 65536
    Rn, Pn = Dn * 2, 72
    src = torch.randint(0, 255, (Pn, NS, Rn), dtype=torch.uint8, device="cuda",
                        generator=torch.Generator(device="cuda").manual_seed(8))
    dst = torch.full((Pn, NS, Rn), 0x7E, dtype=torch.uint8, device="cuda")
    sl = kvx.Layout(Ln, 1, Dn, kvx.F16, NS, base=src, plane_stride=NS * Rn)
    dl = kvx.Layout(Ln, 1, Dn, kvx.F16, NS, base=dst, plane_stride=NS * Rn)
    s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), n, NS)
    d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), n, NS)
    ws = torch.empty(kvx.workspace_size(n), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.transfer(sl, torch.from_numpy(s).cuda(), dl, torch.from_numpy(d).cuda(), n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    samp = _sample(n, 510, 14)
    m = len(samp)
    mini_src = np.ascontiguousarray(src[:, torch.from_numpy(s[samp]).long().cuda()].cpu().numpy())
    dst_host = np.full((Pn, m, Rn), 0x7E, dtype=np.uint8)
    rc, _ = oracle.transfer(
        oracle.Pool(Ln, 1, Dn, 2, oracle.TOKEN_ROWS, m, [(mini_src, p * m * Rn) for p in range(Pn)], Rn),
        np.arange(m),
        oracle.Pool(Ln, 1, Dn, 2, oracle.TOKEN_ROWS, m, [(dst_host, p * m * Rn) for p in range(Pn)], Rn),
        np.arange(m))
    assert rc == oracle.OK
    got = dst[:, torch.from_numpy(d[samp]).long().cuda()].cpu().numpy()
    assert np.array_equal(got, dst_host), "sampled narrow rows differ from the oracle"
    changed = (dst != 0x7E).any(dim=2)
    want = torch.zeros((Pn, NS), dtype=torch.bool, device="cuda")
    want[:, torch.from_numpy(d).long().cuda()] = True
    assert torch.equal(changed, want), "rows other than the named ones changed"
