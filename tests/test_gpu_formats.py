"""Layout and dtype generality against the oracle, through the C ABI (GPU): MLA pools with one
latent plane per layer, fp8 KV, and moves between pool layouts of different kinds
(slot-major <-> per-plane <-> HND pages).

Every case compares the whole destination (pool or buffer, guard bands included) byte for
byte with the oracle on the same seeded inputs, on the three copy paths (planner + row
kernel, one-launch fused, planner + bulk engine) where the entry point has them.
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
# (layers, heads, head_dim, dtype, planes per layer): DeepSeek-V2-Lite-shaped MLA latent rows
# (512 latent + 64 rope) in bf16 (1152 B) and fp8 (576 B); GQA rows in fp8 (1 KiB)
SHAPES = {
    "mla_bf16": (27, 1, 576, "bf16", 1),
    "mla_fp8": (27, 1, 576, "fp8", 1),
    "gqa_fp8": (4, 8, 128, "fp8", 2),
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
    return np.random.Generator(np.random.PCG64(9000 + k))


def _mirror(kind, shape, fill, g=None, num=1024, salt=0):
    L, H, D, dt, kvp = SHAPES[shape]
    return hz.make_mirror(kind, L, H, D, dt, num, 16 if kind == "hnd" else 1, fill, g, salt=salt,
                          kvp=kvp)


def _slots(k, n, num):
    return inputs.distinct_slots(_rng(k), n, num)


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("src_kind", KINDS)
@pytest.mark.parametrize("dst_kind", KINDS)
def test_transfer_formats(shape, src_kind, dst_kind, path):
    n = 500
    src = _mirror(src_kind, shape, "normal", _rng(1)).to_device()
    dst = _mirror(dst_kind, shape, "sentinel", salt=2).to_device()
    exp = _mirror(dst_kind, shape, "sentinel", salt=2)
    s, d = _slots(2, n, src.num_slots), _slots(3, n, dst.num_slots)
    rc, w = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)
    assert rc == oracle.OK and w == n * src.P * src.R
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"{shape} {src_kind}->{dst_kind}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [1, 128, 1000])
def test_gather_scatter_formats(shape, kind, n, path):
    L, H, D, dt, kvp = SHAPES[shape]
    src = _mirror(kind, shape, "normal", _rng(n)).to_device()
    s = _slots(10 + n, n, src.num_slots)
    rc, want, w = oracle.gather(hz.oracle_pool(src), s)
    assert rc == oracle.OK and w == n * src.P * src.R
    buf = hz.make_mirror("buffer", L, H, D, dt, n_tokens=n, fill="sentinel", kvp=kvp).to_device()
    st = hz.status()
    kvx.gather(hz.kvx_layout(src), hz.dev_i32(s), n, hz.GUARD + buf.dev.data_ptr(),
               hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    exp_buf = buf.host.copy()
    exp_buf[hz.GUARD:hz.GUARD + w] = want
    hz.assert_same_bytes(buf.readback(), exp_buf, f"gather {shape} {kind} n={n}")

    dst = _mirror(kind, shape, "sentinel", salt=5).to_device()
    exp = _mirror(kind, shape, "sentinel", salt=5)
    d = _slots(20 + n, n, dst.num_slots)
    assert oracle.scatter(hz.oracle_pool(exp), d, want)[0] == oracle.OK
    st = hz.status()
    kvx.scatter(hz.kvx_layout(dst), hz.dev_i32(d), n, hz.GUARD + buf.dev.data_ptr(),
                hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"scatter {shape} {kind} n={n}")


@pytest.mark.parametrize("shape", ["mla_bf16", "mla_fp8"])
@pytest.mark.parametrize("max_ctas", [0, 40])
def test_stream_latent_layers(shape, max_ctas):
    """kvx_stream over one latent plane per layer: layers below a never-raised layer k move,
    the rest stay untouched (the oracle's layer-range transfer)."""
    L, H, D, dt, kvp = SHAPES[shape]
    n, k = 700, 11
    src = _mirror("planes", shape, "normal", _rng(30)).to_device()
    dst = _mirror("hnd", shape, "sentinel", salt=6).to_device()
    exp = _mirror("hnd", shape, "sentinel", salt=6)
    s, d = _slots(31, n, src.num_slots), _slots(32, n, dst.num_slots)
    rc, w = oracle.transfer_layers(hz.oracle_pool(src), s, hz.oracle_pool(exp), d, k)
    assert rc == oracle.OK and w == n * k * src.R
    ready = torch.tensor([1 if l < k else 0 for l in range(L)], dtype=torch.int32).pin_memory()
    st = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    kvx.stream(kvx.OP_TRANSFER, hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst),
               hz.dev_i32(d), n, None, hz.workspace(n), st, layer_ready=ready, ready_value=1,
               wait_ns=20_000_000, max_ctas=max_ctas, buf_bytes=0)
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    assert v[0] == kvx.ERR_TIMEOUT and v[1] == L - k and v[3] == 1, v
    hz.assert_same_bytes(dst.readback(), exp.host, f"stream {shape} stop {k}")


def test_batch_latent(path):
    """kvx_batch over MLA latent pools: 5 requests of mixed ops and lengths."""
    shape = "mla_bf16"
    L, H, D, dt, kvp = SHAPES[shape]
    g = _rng(40)
    src = _mirror("planes", shape, "normal", g, num=4096).to_device()
    dst = _mirror("slot_major", shape, "sentinel", num=4096, salt=7).to_device()
    exp = _mirror("slot_major", shape, "sentinel", num=4096, salt=7)
    lens = [300, 1, 777, 64, 2049]
    total = sum(lens)
    s = _slots(41, total, 4096)
    d = _slots(42, total, 4096)
    reqs = []
    off = 0
    for i, ln in enumerate(lens):
        reqs.append(kvx.Request(kvx.OP_TRANSFER, ln, off, off, 0))
        off += ln
    oreqs = [(kvx.OP_TRANSFER, ln, r.src_off, r.dst_off, 0) for ln, r in zip(lens, reqs)]
    status = oracle.batch(hz.oracle_pool(src), hz.oracle_pool(exp), oreqs, s, d,
                          np.zeros(16, np.uint8))
    assert list(status) == [0] * (len(lens) + 1)
    dreq = torch.from_numpy(np.frombuffer(b"".join(bytes(r) for r in reqs), dtype=np.uint8).copy()).cuda()
    st = hz.status(len(lens) + 1)
    kvx.batch(hz.kvx_layout(src), hz.kvx_layout(dst), dreq, len(lens), total, hz.dev_i32(s), total,
              hz.dev_i32(d), total, None, hz.workspace(total, len(lens)), st, buf_bytes=0)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0] * (len(lens) + 1)
    hz.assert_same_bytes(dst.readback(), exp.host, "batch of latent rows")
