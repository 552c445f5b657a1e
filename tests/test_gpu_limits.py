"""The documented limits of one call, at the limit, against the oracle (GPU).

- KVX_MAX_TOKENS (8,388,608) rows per plane in one transfer (16-byte rows, one latent plane,
  pools of exactly that many slots, both slot lists random permutations): sampled rows against
  the oracle, and the property that holds at any size -- every destination row equals its
  source row, on the device -- plus the gather of the same request.
- KVX_MAX_PLANES (256) planes, as 128 layers x K/V and as 256 latent planes: whole pools.
- A reshard whose layouts bring exactly KVX_RESHARD_MAX_PLANE_TABLE uneven plane addresses.
- The last slots of the largest pool a layout may describe (INT32_MAX slots of 16 bytes, token
  rows and HND pages), and the first slot past them.
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402


@pytest.fixture(autouse=True)
def _clean():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _rng(k):
    return np.random.Generator(np.random.PCG64(13000 + k))


def test_max_tokens_transfer_and_gather():
    n = kvx.MAX_TOKENS
    R = 16  # one head of 8 fp16
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    src = torch.randint(-2 ** 31, 2 ** 31 - 1, (n, R // 4), dtype=torch.int32, device="cuda",
                        generator=g)
    dst = torch.full((n, R // 4), -1, dtype=torch.int32, device="cuda")
    s = _rng(1).permutation(n).astype(np.int32)
    d = _rng(2).permutation(n).astype(np.int32)
    s_d, d_d = torch.from_numpy(s).cuda(), torch.from_numpy(d).cuda()
    sl = kvx.Layout(1, 1, 8, kvx.F16, n, base=src, plane_stride=n * R, kv_planes=1)
    dl = kvx.Layout(1, 1, 8, kvx.F16, n, base=dst, plane_stride=n * R, kv_planes=1)
    ws = torch.empty(kvx.workspace_size(n, 0), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.transfer(sl, s_d, dl, d_d, n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    # every row, on the device: dst[d[i]] == src[s[i]] (the slot lists are permutations, so
    # this covers the whole destination)
    assert torch.equal(dst[d_d.long()], src[s_d.long()])
    # sampled rows against the oracle
    samp = np.unique(np.concatenate([[0, n - 1], _rng(3).choice(n, 500, replace=False)]))
    m = len(samp)
    mini = src[torch.from_numpy(s[samp]).long().cuda()].cpu().numpy().view(np.uint8).reshape(-1)
    out = np.full(m * R, 0xFF, dtype=np.uint8)
    src_pool = oracle.Pool(1, 1, 8, 2, oracle.TOKEN_ROWS, m, [(mini, 0)], R, kv_planes=1)
    dst_pool = oracle.Pool(1, 1, 8, 2, oracle.TOKEN_ROWS, m, [(out, 0)], R, kv_planes=1)
    rc, _ = oracle.transfer(src_pool, np.arange(m), dst_pool, np.arange(m))
    assert rc == oracle.OK
    got = dst[torch.from_numpy(d[samp]).long().cuda()].cpu().numpy().view(np.uint8).reshape(-1)
    assert np.array_equal(got, out)
    # the gather of the same request: buffer row i is source row s[i]
    buf = torch.empty((n, R // 4), dtype=torch.int32, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.gather(sl, s_d, n, buf, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    assert torch.equal(buf, src[s_d.long()])


def test_max_tokens_plus_one_refused():
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    sl = kvx.Layout(1, 1, 8, kvx.F16, 4, base=t, plane_stride=64, kv_planes=1)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(kvx.KvxError):
        kvx.gather(sl, t, kvx.MAX_TOKENS + 1, t, t, st, buf_bytes=1 << 40, ws_bytes=1 << 40)
    assert int(st.item()) == -1  # nothing enqueued


@pytest.mark.parametrize("kvp", [2, 1], ids=["128_layers_kv", "256_latent"])
@pytest.mark.parametrize("kinds", [("planes", "hnd"), ("slot_major", "planes")])
def test_max_planes(kvp, kinds):
    layers = kvx.MAX_PLANES // kvp
    n, num = 3000, 4096
    g = _rng(kvp + len(kinds[0]))
    src = hz.make_mirror(kinds[0], layers, 1, 8, "fp16", num, 16 if kinds[0] == "hnd" else 1,
                         "normal", g, kvp=kvp).to_device()
    dst = hz.make_mirror(kinds[1], layers, 1, 8, "fp16", num, 16 if kinds[1] == "hnd" else 1,
                         "sentinel", salt=2, kvp=kvp).to_device()
    exp = hz.make_mirror(kinds[1], layers, 1, 8, "fp16", num, 16 if kinds[1] == "hnd" else 1,
                         "sentinel", salt=2, kvp=kvp)
    assert src.P == kvx.MAX_PLANES
    s = inputs.distinct_slots(g, n, num)
    d = inputs.distinct_slots(g, n, num)
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == oracle.OK
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"{kvx.MAX_PLANES} planes {kinds}")


def test_reshard_full_plane_table():
    """Eleven source pools and one destination pool whose planes are not evenly spaced, 256
    planes each: 12 x 256 = 3072 plane addresses, the whole table."""
    assert 12 * kvx.MAX_PLANES == kvx.RESHARD_MAX_PLANE_TABLE
    layers, n, num = 128, 700, 1024
    g = _rng(77)
    # an 11-head model from P TP 11 to D TP 1: source r gives its head to destination head r
    srcs = [hz.make_mirror("planes_rotated", layers, 1, 8, "fp16", num, 1, "normal", g)
            .to_device() for _ in range(11)]
    dst = hz.make_mirror("planes_rotated", layers, 11, 8, "fp16", num, 1, "sentinel",
                         salt=4).to_device()
    exp = hz.make_mirror("planes_rotated", layers, 11, 8, "fp16", num, 1, "sentinel", salt=4)
    parts = kvx.tp_plan(11, 11, 1)
    assert parts == [(r, 0, 0, r, 1) for r in range(11)]
    s = inputs.distinct_slots(g, n, num)
    d = inputs.distinct_slots(g, n, num)
    rc, _ = oracle.reshard([hz.oracle_pool(x) for x in srcs], s, [hz.oracle_pool(exp)], d,
                           parts, n)
    assert rc == oracle.OK
    st = hz.status()
    kvx.reshard([hz.kvx_layout(x) for x in srcs], hz.dev_i32(s), [hz.kvx_layout(dst)],
                hz.dev_i32(d), parts, n, hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, "3072 plane addresses")
    # one more uneven layout is one table entry too many: refused before anything is enqueued
    extra = hz.make_mirror("planes_rotated", layers, 1, 8, "fp16", num, 1, "normal", g).to_device()
    with pytest.raises(kvx.KvxError):
        kvx.reshard([hz.kvx_layout(x) for x in srcs + [extra]], hz.dev_i32(s),
                    [hz.kvx_layout(dst)], hz.dev_i32(d), parts, n, hz.workspace(n), hz.status())


def _sampled_oracle_rows(src, s, m_idx, R):
    """The oracle's transfer of the sampled tokens m_idx between mini pools built from the
    sampled source rows (the pools themselves are too large to mirror on the host)."""
    rows = src[torch.from_numpy(s[m_idx]).long().cuda()].cpu().numpy().view(np.uint8).reshape(-1)
    m = len(m_idx)
    out = np.full(m * R, 0xFF, dtype=np.uint8)
    sp = oracle.Pool(1, 1, R // 2, 2, oracle.TOKEN_ROWS, m, [(rows, 0)], R, kv_planes=1)
    dp = oracle.Pool(1, 1, R // 2, 2, oracle.TOKEN_ROWS, m, [(out, 0)], R, kv_planes=1)
    assert oracle.transfer(sp, np.arange(m), dp, np.arange(m))[0] == oracle.OK
    return out


@pytest.mark.parametrize("kind", ["planes", "hnd"])
def test_top_slot_of_the_largest_pool(kind):
    """A pool of the most slots a layout may have (num_slots = INT32_MAX, or the largest
    multiple of the page size below it for HND pages of 16): 16-byte rows, one plane of 32 GiB
    per side.  The request names the last slots of both pools (byte offsets past 2^35), slot 0
    and random slots; every destination row is checked on the device (the moved rows equal
    their source rows, every other row keeps its sentinel), sampled rows against the oracle,
    and the gather of the same slots.  Slot INT32_MAX itself is one past the end: refused,
    nothing moved."""
    ps = 16 if kind == "hnd" else 1
    num = (2 ** 31 - 1) // ps * ps
    R = 16
    n = 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    src = torch.randint(-2 ** 31, 2 ** 31 - 1, (num, R // 4), dtype=torch.int32, device="cuda",
                        generator=g)
    dst = torch.full((num, R // 4), -1, dtype=torch.int32, device="cuda")
    rng = _rng(40 + ps)
    top = np.arange(num - 8, num, dtype=np.int64)  # the last eight slots, and slot 0
    s = rng.permutation(np.concatenate([top, [0], rng.integers(0, num, n - 9)])).astype(np.int32)
    others = rng.permutation(np.unique(rng.integers(1, num - 8, 2 * n)))[:n - 9]
    d = rng.permutation(np.concatenate([top, [0], others])).astype(np.int32)
    assert len(d) == n and len(np.unique(d)) == n and d.max() == num - 1 and s.max() == num - 1

    def layout(t):
        if kind == "hnd":
            return kvx.Layout(1, 1, 8, kvx.F16, num, kind=kvx.HND_PAGED, page_size=ps, base=t,
                              plane_stride=num * R, kv_planes=1)
        return kvx.Layout(1, 1, 8, kvx.F16, num, base=t, plane_stride=num * R, kv_planes=1)

    sl, dl = layout(src), layout(dst)
    s_d, d_d = torch.from_numpy(s).cuda(), torch.from_numpy(d).cuda()
    ws = torch.empty(kvx.workspace_size(n, 0), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvx.transfer(sl, s_d, dl, d_d, n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    # with one head and one plane, a slot's row is contiguous in both kinds: HND page p holds
    # tokens p*16 .. p*16+15 one after another (one head), so row i of the tensor is slot i
    assert torch.equal(dst[d_d.long()], src[s_d.long()])
    moved = dst[d_d.long()].clone()
    dst[d_d.long()] = -1
    assert bool((dst == -1).all()), "a row outside the request changed"
    dst[d_d.long()] = moved
    samp = np.unique(np.concatenate([np.flatnonzero(s >= num - 8), np.flatnonzero(d >= num - 8),
                                     rng.choice(n, 300, replace=False)]))
    want = _sampled_oracle_rows(src, s, samp, R)
    got = dst[torch.from_numpy(d[samp]).long().cuda()].cpu().numpy().view(np.uint8).reshape(-1)
    assert np.array_equal(got, want)
    # the gather of the same slots: buffer row i is source row s[i]
    buf = torch.empty((n, R // 4), dtype=torch.int32, device="cuda")
    kvx.gather(sl, s_d, n, buf, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    assert torch.equal(buf, src[s_d.long()])
    # one past the end (INT32_MAX for token rows): refused, nothing moved
    bad = d.copy()
    bad[n // 2] = num
    before = dst[d_d.long()].clone()
    dst2_rows = torch.from_numpy(bad).cuda()
    kvx.transfer(sl, s_d, dl, dst2_rows, n, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_OUT_OF_RANGE
    assert torch.equal(dst[d_d.long()], before)
    del src, dst, buf
    torch.cuda.empty_cache()
