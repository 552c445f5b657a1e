"""kvx_transfer_noalloc through the C ABI (GPU), against the oracle and against kvx_transfer.

kvx_transfer_noalloc serves callers that cannot allocate device memory when KV has to move --
an engine that reserved nearly all HBM for its KV pool at start-up has nothing left for a
workspace, and cudaMalloc would synchronise the device between decode steps.  It plans in a
fixed scratch array inside libkvx instead of a caller-given workspace.  These tests check:

* that it moves exactly the bytes the oracle's transfer writes, and the same bytes as the
  workspace-taking kvx_transfer, on two calls in a row, with the register engine and with the
  TMA bulk engine (whose copy walks the plan's chunk table in the shared scratch, so the second
  call runs over whatever the first one left there);
* the exact limits: KVX_NOALLOC_MAX_TOKENS, and KVX_NOALLOC_MAX_DUP_TOKENS with the duplicate
  check (a repeat inside the limit is refused with nothing moved);
* in a fresh process: after one call with n = 0, later calls of every kind do not change the
  device's free memory (the first call loaded the scratch and every kernel).

It builds all its own inputs, so it runs the same alone in a fresh process or after the rest
of the suite; it lives in its own file so that pytest collects it last.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

L, H, D, DT, SLOTS = 4, 8, 128, "bf16", 20000
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pools(seed):
    g = np.random.Generator(np.random.PCG64(seed))
    src = hz.make_mirror("planes", L, H, D, DT, SLOTS, 1, "normal", g).to_device()
    a = hz.make_mirror("planes", L, H, D, DT, SLOTS, 1, "sentinel", salt=3).to_device()
    b = hz.make_mirror("planes", L, H, D, DT, SLOTS, 1, "sentinel", salt=3).to_device()
    exp = hz.make_mirror("planes", L, H, D, DT, SLOTS, 1, "sentinel", salt=3)
    return g, src, a, b, exp


@pytest.mark.parametrize("flags", [0, kvx.USE_BULK], ids=["registers", "bulk"])
def test_noalloc_matches_oracle_and_kvx_transfer_on_two_calls(flags):
    assert torch.cuda.is_available()
    g, src, a, b, exp = _pools(4242)
    src_l, a_l, b_l = hz.kvx_layout(src), hz.kvx_layout(a), hz.kvx_layout(b)
    st_a, st_b = hz.status(), hz.status()
    # two calls in a row: 5000 tokens (three planner tiles), then 700 other tokens
    for n in (5000, 700):
        s_np = inputs.distinct_slots(g, n, SLOTS)
        d_np = inputs.distinct_slots(g, n, SLOTS)
        s, d = hz.dev_i32(s_np), hz.dev_i32(d_np)
        kvx.transfer_noalloc(src_l, s, a_l, d, n, st_a, flags=flags)      # fixed scratch
        kvx.transfer(src_l, s, b_l, d, n, hz.workspace(n), st_b, flags=flags)  # caller workspace
        torch.cuda.synchronize()
        assert int(st_a.item()) == kvx.OK and int(st_b.item()) == kvx.OK
        assert oracle.transfer(hz.oracle_pool(src), s_np, hz.oracle_pool(exp), d_np)[0] == 0
        got = a.readback()
        hz.assert_same_bytes(got, exp.host, f"noalloc vs oracle, n={n}")
        hz.assert_same_bytes(got, b.readback(), f"noalloc vs kvx_transfer, n={n}")
    hz.assert_same_bytes(src.readback(), src.host, "source pool")


def test_noalloc_duplicate_check_at_its_limit():
    g, src, a, _, exp = _pools(4343)
    n = kvx.NOALLOC_MAX_DUP_TOKENS
    s_np = inputs.distinct_slots(g, n, SLOTS)
    d_np = inputs.distinct_slots(g, n, SLOTS)
    st = hz.status()
    # a repeat inside the limit: refused, nothing moved
    rep = d_np.copy()
    rep[n - 1] = rep[0]
    before = a.readback()
    kvx.transfer_noalloc(hz.kvx_layout(src), hz.dev_i32(s_np), hz.kvx_layout(a), hz.dev_i32(rep),
                         n, st, flags=kvx.CHECK_DUP)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.ERR_DUPLICATE_DST
    hz.assert_same_bytes(a.readback(), before, "nothing moved")
    # distinct lists at the limit move, exactly as the oracle
    kvx.transfer_noalloc(hz.kvx_layout(src), hz.dev_i32(s_np), hz.kvx_layout(a), hz.dev_i32(d_np),
                         n, st, flags=kvx.CHECK_DUP)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    assert oracle.transfer(hz.oracle_pool(src), s_np, hz.oracle_pool(exp), d_np, check_dup=True)[0] == 0
    hz.assert_same_bytes(a.readback(), exp.host, "at the duplicate-check limit")
    # one more token does not fit the scratch with the table: refused before anything runs
    s1 = hz.dev_i32(inputs.distinct_slots(g, n + 1, SLOTS))
    st.fill_(-1)
    with pytest.raises(kvx.KvxError) as e:
        kvx.transfer_noalloc(hz.kvx_layout(src), s1, hz.kvx_layout(a), s1, n + 1, st,
                             flags=kvx.CHECK_DUP)
    assert e.value.code == kvx.ERR_NO_WORKSPACE
    torch.cuda.synchronize()
    assert int(st.item()) == -1  # nothing was enqueued


def test_noalloc_refuses_more_than_its_scratch():
    g, src, a, _, _ = _pools(4444)
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


_FRESH = r"""
import sys
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
from disaggregated_paged_kv_gb300 import kvx
torch.cuda.set_device(0)
dev = torch.device("cuda", 0)
def pools(H, D, dt, num):
    s = torch.randn((8, num, H, D), dtype=dt, device=dev)
    d = torch.zeros_like(s)
    R = H * D * s.element_size()
    return (kvx.Layout(4, H, D, kvx.BF16 if dt == torch.bfloat16 else kvx.F16, num, base=s,
                       plane_stride=num * R),
            kvx.Layout(4, H, D, kvx.BF16 if dt == torch.bfloat16 else kvx.F16, num, base=d,
                       plane_stride=num * R), s, d)
big = pools(8, 128, torch.bfloat16, 8192)      # 2 KiB rows
small = pools(2, 64, torch.float16, 8192)      # 256-byte rows
narrow = pools(1, 100, torch.float16, 8192)    # 200-byte rows (narrow kernel)
g = np.random.Generator(np.random.PCG64(5))
lists = {n: torch.from_numpy(g.choice(8192, n, replace=False).astype(np.int32)).to(dev)
         for n in (100, 3000, 8000)}
st = torch.zeros(1, dtype=torch.int32, device=dev)
torch.cuda.synchronize()
kvx.transfer_noalloc(big[0], lists[100], big[1], lists[100], 0, st)   # the set-up call
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
calls = [(big, 100, 0), (big, 3000, 0), (big, 3000, kvx.USE_BULK), (big, 8000, kvx.CHECK_DUP),
         (small, 100, 0), (small, 3000, kvx.ONE_LAUNCH), (small, 3000, 0), (narrow, 3000, 0)]
for (sl, dl, _, _), n, flags in calls:
    kvx.transfer_noalloc(sl, lists[n], dl, lists[n], n, st, flags=flags)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, (n, flags, int(st.item()))
free1 = torch.cuda.mem_get_info()[0]
print("free", free0, free1)
assert free1 == free0, (free0, free1)
"""


def test_noalloc_first_call_sets_the_device_up():
    """A fresh process: one call with n = 0, then calls through every path this entry point
    can take (small requests, the planner with the register and bulk engines, the duplicate
    check, the one-launch path, narrow rows); the device's free memory must not change after
    the first call."""
    res = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
