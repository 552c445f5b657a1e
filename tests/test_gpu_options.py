"""Per-call options (the flags word) against the oracle, through the C ABI (GPU).

* Two host threads on two streams move KV at the same time with different flags while the
  process-wide defaults say something else: each call must follow its own flags only (the
  thread asking for the duplicate check gets KVX_ERR_DUPLICATE_DST on a repeated destination,
  the other thread's repeated destination moves), and every byte must match the oracle.
* The duplicate check on run lists (kvx_transfer_runs / kvx_scatter_runs): the runs expanded
  to slot lists and given to the oracle's check decide the status.
* The duplicate check on batches: statuses, destination pool and buffer against the oracle's
  batch with check_dup, on a fixed case and on random batches over a small pool.
"""
import threading

import numpy as np
import pytest

import oracle
from tests import harness as hz
from tests import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from disaggregated_paged_kv_gb300 import kvx  # noqa: E402

SH = dict(L=3, H=8, D=128, dtype="bf16")  # 2 KiB rows
SMALL = dict(L=2, H=2, D=64, dtype="fp16")  # 256-byte rows (multi-row chunks)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kvx.lib()
    yield


@pytest.fixture
def contrary_defaults():
    """Process-wide defaults that no call below asks for."""
    kvx.set_check_duplicates(True)
    kvx.set_copy_engine(kvx.ENGINE_BULK)
    kvx.set_fused_max_tokens(kvx.FUSED_MAX_TOKENS)
    yield
    kvx.set_check_duplicates(False)
    kvx.set_copy_engine(kvx.ENGINE_AUTO)
    kvx.set_fused_max_tokens(0)


def _rng(k):
    return np.random.Generator(np.random.PCG64(16000 + k))


def _mirrors(sh, num, salt):
    g = _rng(salt)
    src = hz.make_mirror("planes", sh["L"], sh["H"], sh["D"], sh["dtype"], num, 1, "normal", g)
    dst = hz.make_mirror("planes", sh["L"], sh["H"], sh["D"], sh["dtype"], num, 1, "sentinel",
                         salt=salt)
    return src.to_device(), dst.to_device()


def _worker(flags, sh, salt, rounds, out):
    """Runs `rounds` transfers on its own stream with `flags`; records what went wrong."""
    try:
        torch.cuda.set_device(0)
        stream = torch.cuda.Stream()
        num, n = 6144, 3000
        src, dst = _mirrors(sh, num, salt)
        exp = hz.make_mirror("planes", sh["L"], sh["H"], sh["D"], sh["dtype"], num, 1, "sentinel",
                             salt=salt)
        g = _rng(salt + 1)
        ws = hz.workspace(n)
        st = hz.status()
        for r in range(rounds):
            s = inputs.distinct_slots(g, n, num)
            d = inputs.distinct_slots(g, n, num)
            repeat = r % 2 == 1
            if repeat:
                d[n - 1] = d[7]  # one destination named twice
            with torch.cuda.stream(stream):
                kvx.transfer(hz.kvx_layout(src), hz.dev_i32(s), hz.kvx_layout(dst), hz.dev_i32(d),
                             n, ws, st, flags=flags, stream=stream)
            stream.synchronize()
            code = int(st.item())
            checked = bool(flags & kvx.CHECK_DUP)
            if repeat and checked:
                want, _ = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d,
                                          check_dup=True)
                assert want == oracle.ERR_DUPLICATE_DST
                assert code == kvx.ERR_DUPLICATE_DST, (flags, r, code)
                hz.assert_same_bytes(dst.readback(), exp.host, f"flags {flags:#x}: nothing moved")
                continue
            assert code == kvx.OK, (flags, r, code)
            got = dst.readback()
            if repeat:
                # unchecked repeat: the slot holds one of its two source rows, the rest as the
                # oracle writes them
                keep = exp.host.copy()
                assert oracle.transfer(hz.oracle_pool(src), s[:-1], hz.oracle_pool(exp), d[:-1])[0] == 0
                first = exp.host.copy()
                exp.host[:] = keep
                assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == 0
                last = exp.host.copy()
                assert hz.first_mismatch(got, first) is None or hz.first_mismatch(got, last) is None, \
                    f"flags {flags:#x}: repeated slot holds neither source row"
                exp.host[:] = got  # carry on from the device's state
            else:
                assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d)[0] == 0
                hz.assert_same_bytes(got, exp.host, f"flags {flags:#x} round {r}")
    except BaseException as e:  # reported by the test thread
        out.append(e)


@pytest.mark.parametrize("sh", [SH, SMALL], ids=["2KiB_rows", "256B_rows"])
def test_two_threads_two_streams_own_options(sh, contrary_defaults):
    errors = []
    a = threading.Thread(target=_worker, args=(kvx.CHECK_DUP | kvx.USE_REGISTERS, sh, 100, 6, errors))
    b = threading.Thread(target=_worker, args=(kvx.USE_BULK if sh is SH else kvx.ONE_LAUNCH, sh, 200,
                                               6, errors))
    a.start()
    b.start()
    a.join()
    b.join()
    assert not errors, errors[0]


@pytest.mark.parametrize("op", ["transfer", "scatter"])
def test_runs_duplicate_check(op):
    num = 8192
    src, dst = _mirrors(SH, num, 300)
    exp = hz.make_mirror("planes", SH["L"], SH["H"], SH["D"], SH["dtype"], num, 1, "sentinel",
                         salt=300)
    runs = np.array([[10, 100, 5], [40, 3000, 7], [70, 103, 4]], dtype=np.int32)  # dst 103 twice
    n = int(runs[:, 2].sum())
    s = np.concatenate([np.arange(a, a + k) for a, _, k in runs])
    d = np.concatenate([np.arange(b, b + k) for _, b, k in runs])
    if op == "transfer":
        want, _ = oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp), d, check_dup=True)
    else:
        buf_np = _rng(301).integers(0, 0x7C00, 2 * SH["L"] * n * SH["H"] * SH["D"]).astype(np.uint16)
        want, _ = oracle.scatter(hz.oracle_pool(exp), d, buf_np, check_dup=True)
    assert want == oracle.ERR_DUPLICATE_DST
    ws, st = hz.workspace(n, len(runs)), hz.status()
    druns = hz.dev_i32(runs.reshape(-1))
    for flags, code in ((kvx.CHECK_DUP, kvx.ERR_DUPLICATE_DST), (0, kvx.OK)):
        before = dst.readback()
        if op == "transfer":
            kvx.transfer_runs(hz.kvx_layout(src), hz.kvx_layout(dst), druns, len(runs), n, ws, st,
                              flags=flags)
        else:
            buf = torch.from_numpy(buf_np.view(np.int16)).cuda()
            kvx.scatter_runs(hz.kvx_layout(dst), druns, len(runs), n, buf, ws, st, flags=flags)
        torch.cuda.synchronize()
        assert int(st.item()) == code, (op, flags)
        if code != kvx.OK:
            hz.assert_same_bytes(dst.readback(), before, "nothing moved")
    # distinct runs pass the check and match the oracle
    runs[2, 1] = 5000
    d = np.concatenate([np.arange(b, b + k) for _, b, k in runs])
    dst2, exp2 = _mirrors(SH, num, 302)[1], hz.make_mirror("planes", SH["L"], SH["H"], SH["D"],
                                                            SH["dtype"], num, 1, "sentinel", salt=302)
    kvx.transfer_runs(hz.kvx_layout(src), hz.kvx_layout(dst2), hz.dev_i32(runs.reshape(-1)),
                      len(runs), n, ws, st, flags=kvx.CHECK_DUP)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    assert oracle.transfer(hz.oracle_pool(src), s, hz.oracle_pool(exp2), d, check_dup=True)[0] == 0
    hz.assert_same_bytes(dst2.readback(), exp2.host, "distinct runs")


def _run_batch(src, dst, reqs, ss, ds, buf, flags):
    total = int(sum(r[1] for r in reqs))
    dreq = torch.from_numpy(np.frombuffer(b"".join(bytes(kvx.Request(*r)) for r in reqs),
                                          dtype=np.uint8).copy()).cuda()
    ws, st = hz.workspace(max(total, 1), len(reqs)), hz.status(len(reqs) + 1)
    kvx.batch(hz.kvx_layout(src), hz.kvx_layout(dst), dreq, len(reqs), total, hz.dev_i32(ss),
              len(ss), hz.dev_i32(ds), len(ds), hz.GUARD + buf.dev.data_ptr(), ws, st,
              buf_bytes=buf.body.nbytes, flags=flags)
    torch.cuda.synchronize()
    return st.cpu().tolist()


def _check_batch(reqs, ss, ds, salt, flags=kvx.CHECK_DUP, num=64, unspecified=()):
    """Runs the batch and compares statuses, destination pool and buffer with the oracle's.
    Rows of the slots in `unspecified` (named by two requests with the check off, so which
    row lands there is not defined) are left out of the pool comparison."""
    src, dst = _mirrors(SH, num, salt)
    exp = hz.make_mirror("planes", SH["L"], SH["H"], SH["D"], SH["dtype"], num, 1, "sentinel",
                         salt=salt)
    nbuf = max(1, sum(r[1] for r in reqs if r[0] != kvx.OP_TRANSFER))
    buf = hz.make_mirror("buffer", SH["L"], SH["H"], SH["D"], SH["dtype"], n_tokens=nbuf,
                         fill="normal", g=_rng(salt + 5)).to_device()
    ebuf = buf.host[hz.GUARD: hz.GUARD + buf.body.nbytes].copy()
    want = oracle.batch(hz.oracle_pool(src), hz.oracle_pool(exp), reqs, ss, ds, ebuf,
                        check_dup=bool(flags & kvx.CHECK_DUP))
    got = _run_batch(src, dst, reqs, ss, ds, buf, flags)
    assert got == list(want), (got, list(want))
    pool, want_pool = dst.readback(), exp.host.copy()
    R = SH["H"] * SH["D"] * 2
    for slot in unspecified:
        for p in range(2 * SH["L"]):
            a = hz.GUARD + (p * num + slot) * R
            pool[a: a + R] = want_pool[a: a + R]
    hz.assert_same_bytes(pool, want_pool, "batch destination pool")
    got_buf = buf.readback()[hz.GUARD: hz.GUARD + buf.body.nbytes]
    assert np.array_equal(got_buf, ebuf), "batch buffer"
    return got


def test_batch_duplicate_check_fixed_case():
    T, G, S = kvx.OP_TRANSFER, kvx.OP_GATHER, kvx.OP_SCATTER
    R = 2 * SH["L"] * SH["H"] * SH["D"] * 2  # bytes of one token across the planes
    ss = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 99, 1, 2, 3], dtype=np.int32)
    ds = np.array([0, 1, 2, 2, 3, 4, 5, 6, 6, 7, 8, 9, 10, 11, 9], dtype=np.int32)
    reqs = [(T, 3, 0, 0, 0),      # dst 0 1 2: shares 2 with the next request
            (T, 3, 3, 3, 0),      # dst 2 3 4
            (T, 3, 6, 6, 0),      # dst 5 6 6: a repeat of its own
            (T, 3, 9, 9, 0),      # a source slot out of range; dst 7 8 9
            (S, 2, 0, 12, 0),     # dst 10 11
            (T, 1, 12, 14, 0),    # dst 9: shared only with the refused request, so it moves
            (G, 2, 13, 0, 2 * R)]
    got = _check_batch(reqs, ss, ds, 400)
    D_, O_ = kvx.ERR_DUPLICATE_DST, kvx.ERR_OUT_OF_RANGE
    assert got == [D_, D_, D_, D_, O_, 0, 0, 0]
    # the same batch without the check (flags, not defaults): every accepted request moves;
    # slots 2 and 6 are each written twice, so their rows are not compared
    assert _check_batch(reqs, ss, ds, 401, flags=0, unspecified=(2, 6)) == [O_, 0, 0, 0, O_, 0, 0, 0]


@pytest.mark.parametrize("trial", range(12))
def test_batch_duplicate_check_random(trial):
    g = _rng(500 + trial)
    T, G, S = kvx.OP_TRANSFER, kvx.OP_GATHER, kvx.OP_SCATTER
    R = 2 * SH["L"] * SH["H"] * SH["D"] * 2
    reqs, ss, ds, bo = [], [], [], 0
    for _ in range(int(g.integers(2, 9))):
        op = int(g.choice([T, T, S, G]))
        n = int(g.integers(1, 40))
        reqs.append((op, n, len(ss), len(ds), bo if op != T else 0))
        ss += list(g.integers(0, 400 if g.random() < 0.1 else 300, n))
        ds += list(g.choice(300, n, replace=False) if g.random() < 0.7 else g.integers(0, 300, n))
        if op != T:
            bo += n * R
    _check_batch(reqs, np.array(ss, np.int32), np.array(ds, np.int32), 600 + trial, num=300)


@pytest.mark.parametrize("trial", range(8))
def test_batch_duplicate_check_many_overlapping_requests(trial):
    """Many requests whose destination slots overlap in chains (a request sharing one slot with
    one request and another slot with a third), so that the check's inserts race with the
    statuses it raises; statuses, pool and buffer against the oracle.  With requests of up to 200
    tokens on 3000 slots nearly every request meets another; with up to 50 tokens on 20000
    slots about a third of them move."""
    g = _rng(700 + trial)
    T, G, S = kvx.OP_TRANSFER, kvx.OP_GATHER, kvx.OP_SCATTER
    R = 2 * SH["L"] * SH["H"] * SH["D"] * 2
    num, longest = (3000, 200) if trial % 2 == 0 else (20000, 50)
    reqs, ss, ds, bo = [], [], [], 0
    for _ in range(40):
        op = int(g.choice([T, T, T, S, G]))
        n = int(g.integers(1, longest))
        reqs.append((op, n, len(ss), len(ds), bo if op != T else 0))
        ss += list(g.integers(0, num + (20 if g.random() < 0.05 else 0), n))
        ds += list(g.choice(num, n, replace=False))
        if op != T:
            bo += n * R
    _check_batch(reqs, np.array(ss, np.int32), np.array(ds, np.int32), 800 + trial, num=num)
