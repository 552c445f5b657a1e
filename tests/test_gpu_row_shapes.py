"""Row lengths against the row kernel's lane shapes, byte for byte with the oracle (GPU).

The one-shot row kernel gives each token m lanes and each warp G = 32 / m tokens, in one or two
passes over the row, m chosen per row length (any m from 1 to 32, not only powers of two).
These cases pick row lengths that land on every kind of shape -- one lane per token, m not a
power of two, idle lanes past m * G, two passes, rows over 2 KiB -- and move them with gather,
scatter and transfer between token-row and HND layouts, with token counts that end in a
partial warp, comparing whole destinations (guard bands included) with the oracle.
"""
import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


# row bytes (fp16: two heads of R / 4 elements where those are whole 16-byte vectors, else one)
ROWS = [16, 32, 64, 80, 112, 192, 400, 576, 800, 1152, 1280, 1600, 2048, 2304, 4112]
L = 2


def _rng(k):
    return np.random.Generator(np.random.PCG64(5300 + k))


def _mirror(kind, R, fill, g=None, num_slots=2048, salt=0, n_tokens=0):
    H = 2 if R % 32 == 0 else 1
    D = R // (2 * H)
    return hz.make_mirror(kind, L, H, D, "fp16", num_slots, 16 if kind == "hnd" else 1, fill, g,
                          salt=salt, n_tokens=n_tokens)


@pytest.mark.parametrize("R", ROWS)
@pytest.mark.parametrize("n", [1, 333, 1000])
def test_gather_scatter(R, n):
    g = _rng(R + n)
    src = _mirror("hnd", R, "normal", g).to_device()
    s = inputs.distinct_slots(g, n, src.num_slots)
    rc, want, _ = oracle.gather(hz.oracle_pool(src), s)
    assert rc == oracle.OK
    buf = _mirror("buffer", R, "sentinel", n_tokens=n).to_device()
    st = hz.status()
    w = n * src.P * src.R
    kvx.gather(hz.kvx_layout(src), hz.dev_i32(s), n, hz.GUARD + buf.dev.data_ptr(),
               hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    exp = buf.host.copy()
    exp[hz.GUARD:hz.GUARD + w] = want[:w]
    hz.assert_same_bytes(buf.readback(), exp, f"gather R={R} n={n}")

    dst = _mirror("slot_major", R, "sentinel", salt=3).to_device()
    d = inputs.distinct_slots(g, n, dst.num_slots)
    exp_dst = _mirror("slot_major", R, "sentinel", salt=3)
    rc, _ = oracle.scatter(hz.oracle_pool(exp_dst), d, want[:w])
    assert rc == oracle.OK
    st = hz.status()
    kvx.scatter(hz.kvx_layout(dst), hz.dev_i32(d), n, hz.GUARD + buf.dev.data_ptr(),
                hz.workspace(n), st, buf_bytes=w)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp_dst.host, f"scatter R={R} n={n}")


@pytest.mark.parametrize("R", ROWS)
@pytest.mark.parametrize("kinds", [("planes", "hnd"), ("hnd", "planes"), ("slot_major", "planes")])
def test_transfer(R, kinds):
    n = 777
    g = _rng(10 * R + len(kinds[0]))
    src = _mirror(kinds[0], R, "normal", g).to_device()
    dst = _mirror(kinds[1], R, "sentinel", salt=5).to_device()
    s = inputs.distinct_slots(g, n, src.num_slots)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    exp = _mirror(kinds[1], R, "sentinel", salt=5)
    rc, _ = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)
    assert rc == oracle.OK
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    hz.assert_same_bytes(dst.readback(), exp.host, f"transfer R={R} {kinds}")
    hz.assert_same_bytes(src.readback(), src.host, "source")


@pytest.mark.parametrize("R", [576, 1152])
def test_out_of_range_moves_nothing(R):
    """A bad slot in a request whose rows take several lanes-per-token groups: nothing moves."""
    n = 500
    g = _rng(R)
    src = _mirror("planes", R, "normal", g).to_device()
    dst = _mirror("planes", R, "sentinel", salt=9).to_device()
    s = inputs.distinct_slots(g, n, src.num_slots)
    d = inputs.distinct_slots(g, n, dst.num_slots)
    d[n - 2] = dst.num_slots
    st = hz.status()
    kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d), n,
                 hz.workspace(n), st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_OUT_OF_RANGE
    hz.assert_same_bytes(dst.readback(), dst.host, "nothing moved")
