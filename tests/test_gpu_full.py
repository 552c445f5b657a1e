"""The five workloads at full size (GPU), with the default routing the benchmark uses.

Pools are filled on the device (torch.randn, bf16/fp16, seeded; destinations with a quiet-NaN
sentinel).  Each test checks:
  * the status word(s);
  * sampled outputs computed one by one by the CPU oracle: the sampled source rows (or pages)
    are read back into a small host pool, the oracle runs the same operation on it, and its
    result is compared byte for byte with the device's rows;
  * properties that hold at any size: exactly the named destination rows changed (every other
    row still holds the sentinel), and the source is unchanged where it was sampled.
"""
import numpy as np
import pytest

import oracle
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SENT = 0x7FC1  # bf16 quiet NaN; fp16 pools use 0x7E01
DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(autouse=True)
def _clean():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _planes_pool(P, S, H, D, dtype, fill, seed):
    t = torch.empty((P, S, H, D), dtype=DT[dtype], device="cuda")
    if fill == "normal":
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        torch.randn(t.shape, dtype=t.dtype, device="cuda", generator=g, out=t)
    else:
        t.view(torch.int16).fill_(SENT if dtype == "bf16" else 0x7E01)
    return t


def _host_rows_pool(rows):
    """A host oracle pool of per-plane token rows from a [P, k, H, D] tensor."""
    arr = np.ascontiguousarray(rows.cpu().view(torch.int16).numpy()).view(np.uint16)
    P, k, H, D = arr.shape
    planes = [(arr, p * k * H * D * 2) for p in range(P)]
    return oracle.Pool(P // 2, H, D, 2, oracle.TOKEN_ROWS, k, planes, H * D * 2), arr


def _changed_rows(pool, sentinel):
    """Per plane, which slots differ from the sentinel somewhere (device)."""
    P = pool.shape[0]
    out = []
    for p in range(P):
        out.append((pool[p].view(torch.int16).reshape(pool.shape[1], -1) != sentinel).any(dim=1))
    return torch.stack(out)


def _check_sampled_transfer(src, s, dst, d, sample):
    """Oracle on the sampled tokens: rows src[:, s[sample]] -> a fresh sentinel mini pool."""
    st = torch.as_tensor(s[sample], dtype=torch.long, device="cuda")
    dt = torch.as_tensor(d[sample], dtype=torch.long, device="cuda")
    mini_src, _ = _host_rows_pool(src[:, st])
    got = dst[:, dt].cpu().view(torch.int16).numpy().view(np.uint16)
    k = len(sample)
    P, H, D = src.shape[0], src.shape[2], src.shape[3]
    dst_host = np.full((P, k, H, D), SENT, dtype=np.uint16)
    mini_dst = oracle.Pool(P // 2, H, D, 2, oracle.TOKEN_ROWS, k,
                           [(dst_host, p * k * H * D * 2) for p in range(P)], H * D * 2)
    rc, _ = oracle.transfer(mini_src, np.arange(k), mini_dst, np.arange(k))
    assert rc == oracle.OK
    assert np.array_equal(got, dst_host), "sampled rows differ from the oracle"


def test_transfer_2048_tokens_full_size():
    w = inputs.WORKLOADS["transfer"]
    P, S = w.planes, w.num_slots
    src = _planes_pool(P, S, w.kv_heads, w.head_dim, w.dtype, "normal", inputs.seed(w.seed_id, 0))
    dst = _planes_pool(P, S, w.kv_heads, w.head_dim, w.dtype, "sentinel", 0)
    s = inputs.distinct_slots(inputs.rng(w.seed_id, inputs.ROLE_SRC_SLOTS), w.n_tokens, S)
    d = inputs.distinct_slots(inputs.rng(w.seed_id, inputs.ROLE_DST_SLOTS), w.n_tokens, S)
    R = w.row_bytes
    sl = kvx.Layout(w.num_layers, w.kv_heads, w.head_dim, kvx.BF16, S, base=src, plane_stride=S * R)
    dl = kvx.Layout(w.num_layers, w.kv_heads, w.head_dim, kvx.BF16, S, base=dst, plane_stride=S * R)
    ws = torch.empty(kvx.workspace_size(w.n_tokens), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.transfer(sl, torch.from_numpy(s).cuda(), dl, torch.from_numpy(d).cuda(), w.n_tokens, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    g = np.random.Generator(np.random.PCG64(5))
    sample = np.unique(np.concatenate([[0, w.n_tokens - 1], g.choice(w.n_tokens, 254, replace=False)]))
    _check_sampled_transfer(src, s, dst, d, sample)
    want = torch.zeros((P, S), dtype=torch.bool, device="cuda")
    want[:, torch.from_numpy(d).long().cuda()] = True
    assert torch.equal(_changed_rows(dst, SENT), want), "rows other than the named ones changed"


def test_fragmented_gather_scatter_full_size():
    w = inputs.WORKLOADS["fragmented"]
    P, S, H, D = w.planes, w.num_slots, w.kv_heads, w.head_dim
    R = w.row_bytes
    # per-layer separate K and V pools: one allocation per plane
    src_planes = [_planes_pool(1, S, H, D, w.dtype, "normal", inputs.seed(w.seed_id, 0) + p)[0] for p in range(P)]
    s, runs = inputs.fragmented_slots(inputs.rng(w.seed_id, inputs.ROLE_SRC_SLOTS), w.n_tokens, S, 1.6)
    assert 900 <= len(runs) <= 1050
    sl = kvx.Layout(w.num_layers, H, D, kvx.BF16, S, plane_ptrs=src_planes)
    ws = torch.empty(kvx.workspace_size(w.n_tokens), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    buf = torch.empty((P, w.n_tokens, H, D), dtype=torch.bfloat16, device="cuda")
    kvx.gather(sl, torch.from_numpy(s).cuda(), w.n_tokens, buf, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    # the whole 216 MiB buffer against the oracle, over a host pool holding the gathered rows
    st_idx = torch.from_numpy(s).long().cuda()
    rows = torch.stack([pl[st_idx] for pl in src_planes])
    mini, _ = _host_rows_pool(rows)
    rc, want, written = oracle.gather(mini, np.arange(w.n_tokens))
    assert rc == oracle.OK and written == w.payload_bytes == 226492416
    got = buf.cpu().view(torch.int16).numpy().view(np.uint8).reshape(-1)
    assert np.array_equal(got, want)
    # scatter into a fresh destination run layout
    dst_planes = [_planes_pool(1, S, H, D, w.dtype, "sentinel", 0)[0] for _ in range(P)]
    d, _ = inputs.fragmented_slots(inputs.rng(w.seed_id, inputs.ROLE_DST_SLOTS), w.n_tokens, S, 1.6)
    dl = kvx.Layout(w.num_layers, H, D, kvx.BF16, S, plane_ptrs=dst_planes)
    kvx.scatter(dl, torch.from_numpy(d).cuda(), w.n_tokens, buf, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    dd = torch.from_numpy(d).long().cuda()
    for p in range(P):
        assert torch.equal(dst_planes[p][dd].view(torch.int16), buf[p].view(torch.int16))
        changed = (dst_planes[p].view(torch.int16).reshape(S, -1) != SENT).any(dim=1)
        want = torch.zeros(S, dtype=torch.bool, device="cuda")
        want[dd] = True
        assert torch.equal(changed, want)


def test_batch_64_requests_full_size():
    w = inputs.WORKLOADS["batch"]
    P, S, H, D, ps = w.planes, w.num_slots, w.kv_heads, w.head_dim, w.page_size
    R = w.row_bytes
    lens = inputs.batch_lengths()
    assert len(lens) == 64 and 1000 <= min(lens) and max(lens) <= 2000
    s, offs = inputs.paged_request_slots(inputs.rng(w.seed_id, inputs.ROLE_SRC_SLOTS), lens, ps, S)
    d, _ = inputs.paged_request_slots(inputs.rng(w.seed_id, inputs.ROLE_DST_SLOTS), lens, ps, S)
    src = _planes_pool(P, S, H, D, w.dtype, "normal", inputs.seed(w.seed_id, 0))
    dst = _planes_pool(P, S, H, D, w.dtype, "sentinel", 0)
    sl = kvx.Layout(w.num_layers, H, D, kvx.BF16, S, base=src, plane_stride=S * R)
    dl = kvx.Layout(w.num_layers, H, D, kvx.BF16, S, base=dst, plane_stride=S * R)
    reqs = [kvx.Request(kvx.OP_TRANSFER, L, int(o), int(o), 0) for L, o in zip(lens, offs[:-1])]
    dreq = torch.from_numpy(np.frombuffer(b"".join(bytes(r) for r in reqs), dtype=np.uint8).copy()).cuda()
    total = int(sum(lens))
    ws = torch.empty(kvx.workspace_size(total, len(reqs)), dtype=torch.uint8, device="cuda")
    st = torch.full((len(reqs) + 1,), -1, dtype=torch.int32, device="cuda")
    ds = torch.from_numpy(s).cuda()
    dd = torch.from_numpy(d).cuda()
    kvx.batch(sl, dl, dreq, len(reqs), total, ds, total, dd, total, None, ws, st, buf_bytes=0)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0] * (len(reqs) + 1)
    # sampled tokens of every request, including each request's last (partial-page) token
    g = np.random.Generator(np.random.PCG64(6))
    sample = []
    for q, L in enumerate(lens):
        o = int(offs[q])
        sample += [o, o + L - 1] + list(o + g.choice(L, 6, replace=False))
    sample = np.unique(np.asarray(sample))
    _check_sampled_transfer(src, s, dst, d, sample)
    want = torch.zeros((P, S), dtype=torch.bool, device="cuda")
    want[:, dd.long()] = True  # the tails of partial destination pages stay sentinel
    assert torch.equal(_changed_rows(dst, SENT), want)


def test_hnd_permute_gather_and_rebuild_full_size():
    w = inputs.WORKLOADS["hnd_permute"]
    P, H, D, ps = w.planes, w.kv_heads, w.head_dim, w.page_size
    pages = w.num_slots // ps
    seq = w.n_tokens
    n_pages = seq // ps
    R = w.row_bytes
    g = torch.Generator(device="cuda")
    g.manual_seed(inputs.seed(w.seed_id, 0))
    src = torch.randn((P, pages, H, ps, D), dtype=torch.bfloat16, device="cuda", generator=g)
    pt = inputs.random_pages(inputs.rng(w.seed_id, inputs.ROLE_SRC_SLOTS), n_pages, pages)
    slots = inputs.page_table_slots(pt, seq, ps)
    sl = kvx.Layout(w.num_layers, H, D, kvx.BF16, pages * ps, kind=kvx.HND_PAGED, page_size=ps,
                    base=src, plane_stride=pages * ps * R)
    ws = torch.empty(kvx.workspace_size(seq), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    buf = torch.empty((P, seq, H, D), dtype=torch.bfloat16, device="cuda")
    kvx.gather(sl, torch.from_numpy(slots).cuda(), seq, buf, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    # oracle on 32 sampled logical pages (first, last and random): their physical pages are
    # read back into a small host HND pool, gathered by the oracle through [heads, seq, dim]
    rng = np.random.Generator(np.random.PCG64(7))
    lp = np.unique(np.concatenate([[0, n_pages - 1], rng.choice(n_pages, 30, replace=False)]))
    k = len(lp)
    mini_pages = src[:, torch.from_numpy(pt[lp]).long().cuda()].cpu().view(torch.int16).numpy().view(np.uint16)
    mini_pages = np.ascontiguousarray(mini_pages)  # [P, k, H, ps, D]
    mini = oracle.Pool(P // 2, H, D, 2, oracle.HND_PAGES, k * ps,
                       [(mini_pages, p * k * H * ps * D * 2) for p in range(P)], 0, ps)
    rc, want = oracle.hnd_gather(mini, np.arange(k), k * ps)
    assert rc == oracle.OK
    tok = (lp[:, None] * ps + np.arange(ps)[None, :]).reshape(-1)
    got = buf[:, torch.from_numpy(tok).long().cuda()].cpu().view(torch.int16).numpy().view(np.uint8).reshape(-1)
    assert np.array_equal(got, want)
    del src
    torch.cuda.empty_cache()
    # inverse rebuild into a second pool under an independent page table
    dst = torch.empty((P, pages, H, ps, D), dtype=torch.bfloat16, device="cuda")
    dst.view(torch.int16).fill_(SENT)
    pt2 = inputs.random_pages(inputs.rng(w.seed_id, inputs.ROLE_DST_SLOTS), n_pages, pages)
    dl = kvx.Layout(w.num_layers, H, D, kvx.BF16, pages * ps, kind=kvx.HND_PAGED, page_size=ps,
                    base=dst, plane_stride=pages * ps * R)
    kvx.scatter(dl, torch.from_numpy(inputs.page_table_slots(pt2, seq, ps)).cuda(), seq, buf, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    host = np.full((P, k, H, ps, D), SENT, dtype=np.uint16)
    mini_dst = oracle.Pool(P // 2, H, D, 2, oracle.HND_PAGES, k * ps,
                           [(host, p * k * H * ps * D * 2) for p in range(P)], 0, ps)
    assert oracle.hnd_rebuild(mini_dst, np.arange(k), k * ps, want) == oracle.OK
    got_pages = dst[:, torch.from_numpy(pt2[lp]).long().cuda()].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_pages, host)
    changed = torch.stack([(dst[p].view(torch.int16).reshape(pages, -1) != SENT).any(dim=1) for p in range(P)])
    want_mask = torch.zeros((P, pages), dtype=torch.bool, device="cuda")
    want_mask[:, torch.from_numpy(pt2).long().cuda()] = True
    assert torch.equal(changed, want_mask)
