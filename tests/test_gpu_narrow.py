"""Rows that do not allow 16-byte accesses, against the oracle, through the C ABI (GPU).

Row sizes and head vectors that are not multiples of 16 bytes -- 200-byte rows (head_dim 100
fp16), 36-byte fp8 rows, 7-byte rows, 8-byte head vectors in HND pages -- move through the
narrow row kernel with the widest access the call allows.  Every case compares the whole
destination (guard bands included) byte for byte with the oracle; the fused and bulk settings
must fall back to the narrow kernel and give the same bytes.
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

KINDS = ["planes", "slot_major", "hnd"]
SHAPES = {  # (layers, heads, head_dim, dtype)
    "r200_fp16": (3, 1, 100, "fp16"),   # 8-byte accesses
    "r36_fp8": (2, 3, 12, "fp8"),       # 4-byte accesses
    "r7_fp8": (2, 1, 7, "fp8"),         # byte accesses
    "h8_fp16": (2, 2, 4, "fp16"),       # 16-byte rows of 8-byte head vectors
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


@pytest.fixture(params=["default", "fused", "planned_bulk"])
def path(request):
    fused, engine = {"default": (0, kvx.ENGINE_AUTO), "fused": (8192, kvx.ENGINE_AUTO),
                     "planned_bulk": (0, kvx.ENGINE_BULK)}[request.param]
    kvx.set_fused_max_tokens(fused)
    kvx.set_copy_engine(engine)
    yield request.param
    kvx.set_fused_max_tokens(0)
    kvx.set_copy_engine(kvx.ENGINE_AUTO)


def _rng(k):
    return np.random.Generator(np.random.PCG64(11000 + k))


def _mirror(kind, shape, fill, g=None, num=2048, salt=0):
    L, H, D, dt = SHAPES[shape]
    return hz.make_mirror(kind, L, H, D, dt, num, 16 if kind == "hnd" else 1, fill, g, salt=salt)


def _slots(k, n, num):
    return inputs.distinct_slots(_rng(k), n, num)


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("src_kind", KINDS)
@pytest.mark.parametrize("dst_kind", KINDS)
def test_transfer_narrow(shape, src_kind, dst_kind, path):
    n = 1500
    src = _mirror(src_kind, shape, "normal", _rng(1)).to_device()
    dst = _mirror(dst_kind, shape, "sentinel", salt=2).to_device()
    exp = _mirror(dst_kind, shape, "sentinel", salt=2)
    s, d = _slots(2, n, src.num_slots), _slots(3, n, dst.num_slots)
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == oracle.OK
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"{shape} {src_kind}->{dst_kind}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("kind", KINDS)
def test_gather_scatter_plan_execute_narrow(shape, kind, path):
    """Gather by kvx_gather, then scatter through a separate kvx_plan + kvx_execute."""
    L, H, D, dt = SHAPES[shape]
    n = 2500
    src = _mirror(kind, shape, "normal", _rng(5), num=4096).to_device()
    s = _slots(6, n, src.num_slots)
    rc, want, w = oracle.gather(hz.oracle_pool(src), s)
    assert rc == oracle.OK
    buf = hz.make_mirror("buffer", L, H, D, dt, n_tokens=n, fill="sentinel").to_device()
    st = hz.status()
    kvx.gather(hz.kvx_layout(src), hz.dev_i32(s), n, hz.GUARD + buf.dev.data_ptr(),
               hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    exp_buf = buf.host.copy()
    exp_buf[hz.GUARD:hz.GUARD + w] = want
    hz.assert_same_bytes(buf.readback(), exp_buf, f"gather {shape} {kind}")

    dst = _mirror(kind, shape, "sentinel", num=4096, salt=7).to_device()
    exp = _mirror(kind, shape, "sentinel", num=4096, salt=7)
    d = _slots(8, n, dst.num_slots)
    assert oracle.scatter(hz.oracle_pool(exp), d, want)[0] == oracle.OK
    ws, st = hz.workspace(n), hz.status()
    lay = hz.kvx_layout(dst)
    kvx.plan(kvx.OP_SCATTER, None, None, lay, hz.dev_i32(d), n, ws, st)
    kvx.execute(kvx.OP_SCATTER, None, lay, None, 0, n, hz.GUARD + buf.dev.data_ptr(), ws, st,
                buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"plan+execute scatter {shape} {kind}")


@pytest.mark.parametrize("shape", ["r200_fp16", "r7_fp8"])
def test_batch_and_out_of_range_narrow(shape, path):
    src = _mirror("planes", shape, "normal", _rng(20), num=4096).to_device()
    dst = _mirror("hnd", shape, "sentinel", num=4096, salt=9).to_device()
    exp = _mirror("hnd", shape, "sentinel", num=4096, salt=9)
    lens = [100, 1, 2049, 33]
    total = sum(lens)
    s, d = _slots(21, total, 4096), _slots(22, total, 4096)
    d_bad = d.copy()
    d_bad[100] = 4096  # request 1 (one token) is out of range; the others still move
    offs = np.concatenate([[0], np.cumsum(lens)])
    reqs = [kvx.Request(kvx.OP_TRANSFER, ln, int(o), int(o), 0) for ln, o in zip(lens, offs)]
    oreqs = [(kvx.OP_TRANSFER, ln, int(o), int(o), 0) for ln, o in zip(lens, offs)]
    want_st = oracle.batch(hz.oracle_pool(src), hz.oracle_pool(exp), oreqs, s, d_bad,
                           np.zeros(16, np.uint8))
    assert list(want_st) == [kvx.ERR_OUT_OF_RANGE, 0, kvx.ERR_OUT_OF_RANGE, 0, 0]
    dreq = torch.from_numpy(np.frombuffer(b"".join(bytes(r) for r in reqs), dtype=np.uint8).copy()).cuda()
    st = hz.status(len(lens) + 1)
    kvx.batch(hz.kvx_layout(src), hz.kvx_layout(dst), dreq, len(lens), total, hz.dev_i32(s), total,
              hz.dev_i32(d_bad), total, None, hz.workspace(total, len(lens)), st, buf_bytes=0)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == list(want_st)
    hz.assert_same_bytes(dst.readback(), exp.host, f"batch {shape}")


@pytest.mark.parametrize("mem", ["pinned", "pageable"])
def test_submit_narrow(mem, path):
    shape = "r36_fp8"
    n = 1200
    src = _mirror("slot_major", shape, "normal", _rng(30)).to_device()
    dst = _mirror("planes", shape, "sentinel", salt=3).to_device()
    exp = _mirror("planes", shape, "sentinel", salt=3)
    s_np, d_np = _slots(31, n, 2048), _slots(32, n, 2048)
    assert oracle.transfer(hz.oracle_pool(src), s_np, hz.oracle_pool(exp), d_np)[0] == oracle.OK
    s = torch.from_numpy(s_np).pin_memory() if mem == "pinned" else s_np
    d = torch.from_numpy(d_np).pin_memory() if mem == "pinned" else d_np
    hst = torch.full((1,), -1, dtype=torch.int32)
    hst = hst.pin_memory() if mem == "pinned" else hst
    kvx.submit(kvx.OP_TRANSFER, hz.kvx_layout(src), s, hz.kvx_layout(dst), d, n, None,
               hz.workspace(n), hst, buf_bytes=0)
    torch.cuda.synchronize()
    assert int(hst[0]) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"submit narrow {mem}")


def test_move_heads_narrow(path):
    """Heads of 8 bytes (head_dim 4 fp16): head ranges start on 8-byte boundaries."""
    n = 900
    src = hz.make_mirror("planes", 2, 4, 4, "fp16", 2048, 1, "normal", _rng(40)).to_device()
    dst = hz.make_mirror("hnd", 2, 3, 4, "fp16", 2048, 16, "sentinel", salt=4).to_device()
    exp = hz.make_mirror("hnd", 2, 3, 4, "fp16", 2048, 16, "sentinel", salt=4)
    s, d = _slots(41, n, 2048), _slots(42, n, 2048)
    rc, _, _ = oracle.move_heads(2, hz.oracle_pool(src), s, 1, hz.oracle_pool(exp), d, 0, 3, n)
    assert rc == oracle.OK
    st = hz.status()
    kvx.move_heads(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), 1, hz.kvx_layout(dst),
                   hz.dev_i32(d), 0, 3, n, None, hz.workspace(n), st, buf_bytes=0)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, "narrow head move")
