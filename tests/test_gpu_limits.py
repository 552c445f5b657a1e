"""The documented limits of one call, at the limit, against the oracle (GPU).

- KVX_MAX_TOKENS (8,388,608) rows per plane in one transfer (16-byte rows, one latent plane,
  pools of exactly that many slots, both slot lists random permutations): sampled rows against
  the oracle, and the property that holds at any size -- every destination row equals its
  source row, on the device -- plus the gather of the same request.
- KVX_MAX_PLANES (256) planes, as 128 layers x K/V and as 256 latent planes: whole pools.
- A reshard whose layouts bring exactly KVX_RESHARD_MAX_PLANE_TABLE uneven plane addresses.
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
