"""kvx_transfer_noalloc against kvx_transfer, through the C ABI (GPU).

kvx_transfer_noalloc serves callers that cannot allocate device memory when KV has to move --
an engine that reserved nearly all HBM for its KV pool at start-up has nothing left for a
workspace, and cudaMalloc would synchronise the device between decode steps.  It plans in a
fixed scratch array inside libkvx instead of a caller-given workspace.  This test checks that
it moves exactly the bytes the workspace-taking kvx_transfer moves, on two calls in a row (the
second call runs over the plan the first one left in the shared scratch), and that a request
larger than the scratch is refused with nothing moved.

It builds all its own inputs, so it runs the same alone in a fresh process or after the rest
of the suite; it lives in its own file so that pytest collects it last.
"""
import numpy as np
import pytest

from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

L, H, D, DT, SLOTS = 4, 8, 128, "bf16", 20000


def _pools(seed):
    g = np.random.Generator(np.random.PCG64(seed))
    src = hz.make_mirror("planes", L, H, D, DT, SLOTS, 1, "normal", g).to_device()
    a = hz.make_mirror("planes", L, H, D, DT, SLOTS, 1, "sentinel", salt=3).to_device()
    b = hz.make_mirror("planes", L, H, D, DT, SLOTS, 1, "sentinel", salt=3).to_device()
    return g, src, a, b


def test_noalloc_matches_kvx_transfer_on_two_calls():
    assert torch.cuda.is_available()
    g, src, a, b = _pools(4242)
    src_l, a_l, b_l = hz.kvx_layout(src), hz.kvx_layout(a), hz.kvx_layout(b)
    st_a, st_b = hz.status(), hz.status()
    # two calls in a row: 5000 tokens (three planner tiles), then 700 other tokens
    for n in (5000, 700):
        s = hz.dev_i32(inputs.distinct_slots(g, n, SLOTS))
        d = hz.dev_i32(inputs.distinct_slots(g, n, SLOTS))
        ws = hz.workspace(n)
        kvx.transfer_noalloc(src_l, s, a_l, d, n, st_a)           # fixed scratch
        kvx.transfer(src_l, s, b_l, d, n, ws, st_b)               # caller workspace
        torch.cuda.synchronize()
        assert int(st_a.item()) == kvx.OK and int(st_b.item()) == kvx.OK
        got, want = a.readback(), b.readback()
        hz.assert_same_bytes(got, want, f"noalloc vs transfer, n={n}")
        assert not np.array_equal(want, a.host)  # rows really moved
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


def test_noalloc_refuses_more_than_its_scratch():
    g, src, a, _ = _pools(4343)
    n = kvx.NOALLOC_MAX_TOKENS + 1
    s = hz.dev_i32(np.arange(n) % SLOTS)
    st = hz.status()
    before = a.readback()
    with pytest.raises(kvx.KvxError) as e:
        kvx.transfer_noalloc(hz.kvx_layout(src), s, hz.kvx_layout(a), s, n, st)
    assert e.value.code == kvx.ERR_NO_WORKSPACE
    torch.cuda.synchronize()
    assert int(st.item()) == -1  # nothing was enqueued
    hz.assert_same_bytes(a.readback(), before, "nothing moved")
