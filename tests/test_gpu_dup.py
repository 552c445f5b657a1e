"""The duplicate-destination check (kvx_set_check_duplicates) against the oracle's check_dup,
through the C ABI (GPU): repeated destination slots -- inside one planner tile, across tiles,
through every entry point that writes pools from slot lists -- give KVX_ERR_DUPLICATE_DST and
move nothing; distinct lists pass unchanged; with the switch off the same lists move.
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SH = dict(L=3, H=8, D=128, dtype="bf16")  # 2 KiB rows


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


@pytest.fixture
def check_on():
    kvx.set_check_duplicates(True)
    yield
    kvx.set_check_duplicates(False)


@pytest.fixture(params=["default", "planned_bulk", "small_rows"])
def variant(request):
    if request.param == "planned_bulk":
        kvx.set_copy_engine(kvx.ENGINE_BULK)
    yield request.param
    kvx.set_copy_engine(kvx.ENGINE_AUTO)


def _rng(k):
    return np.random.Generator(np.random.PCG64(13000 + k))


def _pools(variant, num=8192):
    sh = dict(SH)
    if variant == "small_rows":
        sh.update(H=2, D=64, dtype="fp16")  # 256-byte rows: multi-row chunks, fused-capable
    g = _rng(1)
    src = hz.make_mirror("planes", sh["L"], sh["H"], sh["D"], sh["dtype"], num, 1, "normal",
                         g).to_device()
    dst = hz.make_mirror("planes", sh["L"], sh["H"], sh["D"], sh["dtype"], num, 1, "sentinel",
                         salt=2).to_device()
    exp = hz.make_mirror("planes", sh["L"], sh["H"], sh["D"], sh["dtype"], num, 1, "sentinel",
                         salt=2)
    return src, dst, exp


@pytest.mark.parametrize("n,i,j", [(2, 0, 1), (2048, 5, 2000), (5000, 17, 4990), (5000, 2047, 2048)])
def test_transfer_duplicate_refused(n, i, j, variant, check_on):
    src, dst, exp = _pools(variant)
    s = inputs.distinct_slots(_rng(n), n, 8192)
    d = inputs.distinct_slots(_rng(n + 1), n, 8192)
    d[j] = d[i]  # slot named twice (same tile or another tile)
    rc, _ = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d, check_dup=True)
    assert rc == oracle.ERR_DUPLICATE_DST
    before = dst.readback()
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_DUPLICATE_DST
    hz.assert_same_bytes(dst.readback(), before, "nothing moved")


@pytest.mark.parametrize("n", [1, 777, 6000])
def test_distinct_lists_pass(n, variant, check_on):
    src, dst, exp = _pools(variant)
    s = inputs.distinct_slots(_rng(3 * n), n, 8192)
    d = inputs.distinct_slots(_rng(3 * n + 1), n, 8192)
    rc, _ = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d, check_dup=True)
    assert rc == oracle.OK
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, "distinct destinations")


def test_duplicates_move_when_unchecked(variant):
    src, dst, _ = _pools(variant)
    n = 300
    s = inputs.distinct_slots(_rng(7), n, 8192)
    d = inputs.distinct_slots(_rng(8), n, 8192)
    d[10] = d[250]
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK


def test_other_entry_points_refuse(check_on):
    src, dst, exp = _pools("default")
    n = 900
    s = inputs.distinct_slots(_rng(20), n, 8192)
    d = inputs.distinct_slots(_rng(21), n, 8192)
    d[899] = d[0]
    before = dst.readback()
    P, R = 2 * SH["L"], SH["H"] * SH["D"] * 2
    # scatter from a buffer
    buf = hz.make_mirror("buffer", SH["L"], SH["H"], SH["D"], SH["dtype"], n_tokens=n, fill="normal",
                         g=_rng(22)).to_device()
    st = hz.status()
    kvx.scatter(hz.kvx_layout(dst), hz.dev_i32(d), n, hz.GUARD + buf.dev.data_ptr(), hz.workspace(n),
                st, buf_bytes=n * P * R)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_DUPLICATE_DST
    # plan + execute
    ws, st = hz.workspace(n), hz.status()
    kvx.plan(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d),
             n, ws, st)
    kvx.execute(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.kvx_layout(dst), None, 0, n, None, ws, st,
                buf_bytes=0)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_DUPLICATE_DST
    # submit with pinned lists
    hs = torch.from_numpy(s).pin_memory()
    hd = torch.from_numpy(d).pin_memory()
    hst = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    kvx.submit(kvx.OP_TRANSFER, hz.kvx_layout(src), hs, hz.kvx_layout(dst), hd, n, None,
               hz.workspace(n), hst, buf_bytes=0)
    torch.cuda.synchronize()
    assert int(hst[0]) == kvx.ERR_DUPLICATE_DST
    # streamed move
    st4 = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    kvx.stream(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst),
               hz.dev_i32(d), n, None, hz.workspace(n), st4, buf_bytes=0)
    torch.cuda.synchronize()
    v = st4.cpu().tolist()
    assert v[0] == kvx.ERR_DUPLICATE_DST and v[1] == SH["L"] and v[3] == 1, v
    # head-range move
    st = hz.status()
    kvx.move_heads(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), 0, hz.kvx_layout(dst),
                   hz.dev_i32(d), 4, 4, n, None, hz.workspace(n), st, buf_bytes=0)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_DUPLICATE_DST
    hz.assert_same_bytes(dst.readback(), before, "nothing moved by any entry point")
    # the fixed scratch of kvx_transfer_noalloc holds the table for requests this small ...
    st = hz.status()
    kvx.transfer_noalloc(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                         st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_DUPLICATE_DST
    hz.assert_same_bytes(dst.readback(), before, "nothing moved by kvx_transfer_noalloc")
    # ... but not at its token limit
    big = kvx.NOALLOC_MAX_TOKENS
    sb = hz.dev_i32(np.arange(big) % 8192)
    with pytest.raises(kvx.KvxError) as e:
        kvx.transfer_noalloc(hz.kvx_layout(src), sb, hz.kvx_layout(dst), sb, big, hz.status())
    assert e.value.code == kvx.ERR_NO_WORKSPACE
