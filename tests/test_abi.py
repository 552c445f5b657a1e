"""The C ABI on the CPU: the library loads, exports every entry point include/kvx.h declares,
and rejects bad host-visible arguments before touching CUDA (no GPU is needed for any of
these: each call returns before its first CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

from disaggregated_paged_kv_gb300 import build as kbuild
from disaggregated_paged_kv_gb300 import kvx
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvx.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(kvx.LIB_PATH):
        kbuild.build()
    return kvx.lib()


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^KVX_API\s+[\w\s\*]+?\*?(kvx_\w+)\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", kvx.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    # the binding covers the same set
    assert sorted(kvx.exported_names()) == names


def test_misc(lib):
    assert kvx.version() == 300
    assert kvx.status_str(kvx.OK) == "ok"
    assert "range" in kvx.status_str(kvx.ERR_OUT_OF_RANGE)
    ws = kvx.workspace_size(2048, 0)
    assert ws > 2048 * 16 and ws % 256 == 0
    assert kvx.workspace_size(kvx.MAX_TOKENS + 1, 0) == 0
    assert kvx.workspace_size(-1, 0) == 0
    assert kvx.workspace_size(10, -1) == 0


FAKE = 1 << 40  # a 16-byte-aligned address that is never dereferenced on the host


def test_layout_validation(lib):
    L = kvx.Layout(36, 8, 128, kvx.BF16, 65536, base=FAKE, plane_stride=65536 * 2048)
    assert L.row_bytes == 2048 and L.num_planes == 72
    L.close()
    bad = [
        dict(num_layers=0),
        dict(num_layers=129),
        dict(kv_heads=0),
        dict(dtype=9),
        dict(num_slots=0),
        dict(num_slots=2 ** 31),
        dict(kind=5),
        dict(base=None),
        dict(slot_stride=128),  # smaller than a row
    ]
    for kw in bad:
        args = dict(num_layers=2, kv_heads=2, head_dim=64, dtype=kvx.F16, num_slots=100,
                    base=FAKE, plane_stride=100 * 256)
        args.update(kw)
        with pytest.raises(kvx.KvxError) as e:
            kvx.Layout(**args)
        assert e.value.code == kvx.ERR_INVALID_ARG, kw
    # rows, strides and planes that are not 16-byte multiples are accepted (they move with
    # narrower accesses); a plane that splits an element is not
    for kw in [dict(head_dim=3), dict(base=FAKE + 8), dict(slot_stride=264)]:
        args = dict(num_layers=2, kv_heads=2, head_dim=64, dtype=kvx.F16, num_slots=100,
                    base=FAKE, plane_stride=100 * 256)
        args.update(kw)
        kvx.Layout(**args).close()
    with pytest.raises(kvx.KvxError) as e:
        kvx.Layout(2, 2, 64, kvx.F16, 100, base=FAKE + 1, plane_stride=100 * 256)
    assert e.value.code == kvx.ERR_ALIGNMENT
    with pytest.raises(kvx.KvxError):  # HND: slots must fill whole pages
        kvx.Layout(2, 2, 64, kvx.F16, 100, kind=kvx.HND_PAGED, page_size=16, base=FAKE,
                   plane_stride=1 << 20)
    kvx.Layout(2, 4, 4, kvx.F16, 32, kind=kvx.HND_PAGED, page_size=16, base=FAKE,
               plane_stride=1 << 20).close()  # 8-byte head vectors
    # explicit plane pointers
    ptrs = [FAKE + (1 << 30) * p for p in range(4)]
    L = kvx.Layout(2, 2, 64, kvx.F16, 100, plane_ptrs=ptrs)
    assert L.num_planes == 4
    with pytest.raises(kvx.KvxError):
        kvx.Layout(2, 2, 64, kvx.F16, 100, plane_ptrs=ptrs[:3] + [0])


def test_call_validation_before_cuda(lib):
    src = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE, plane_stride=1000 * 256)
    dst = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE * 2, plane_stride=1000 * 256)
    other = kvx.Layout(3, 2, 64, kvx.F16, 1000, base=FAKE * 3, plane_stride=1000 * 256)
    WS, ST, SL, BUF = FAKE * 4, FAKE * 5, FAKE * 6, FAKE * 7
    big = 1 << 30
    l = kvx.lib()
    # transfer: mismatched shapes, overlap, null status, negative n
    assert l.kvx_transfer(src.handle, SL, other.handle, SL, 10, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_transfer(src.handle, SL, src.handle, SL, 10, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_OVERLAP
    assert l.kvx_transfer(src.handle, SL, dst.handle, SL, 10, WS, big, None, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_transfer(src.handle, SL, dst.handle, SL, -1, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_transfer(src.handle, None, dst.handle, SL, 10, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_transfer(src.handle, SL, dst.handle, SL, 10, WS + 16, big, ST, kvx.DEFAULTS, None) == kvx.ERR_NO_WORKSPACE
    assert l.kvx_transfer(src.handle, SL, dst.handle, SL, 10, WS, 512, ST, kvx.DEFAULTS, None) == kvx.ERR_NO_WORKSPACE
    assert l.kvx_transfer(None, SL, dst.handle, SL, 10, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    # gather: buffer checks
    need = 4 * 10 * 256
    assert l.kvx_gather(src.handle, SL, 10, None, need, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_gather(src.handle, SL, 10, BUF + 4, need, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_ALIGNMENT
    assert l.kvx_gather(src.handle, SL, 10, BUF, need - 16, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_gather(src.handle, SL, 10, FAKE + 256, need, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_OVERLAP
    # execute / plan argument checks
    assert l.kvx_execute(9, src.handle, dst.handle, None, 0, 10, None, 0, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_plan(kvx.OP_BATCH, src.handle, SL, dst.handle, SL, 10, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_plan_runs(kvx.OP_TRANSFER, src.handle, dst.handle, None, 3, 10, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_plan_batch(src.handle, dst.handle, None, 2, 10, SL, 10, SL, 10, 0, WS, big, ST, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG
    assert l.kvx_submit(kvx.OP_TRANSFER, src.handle, None, dst.handle, None, 10, None, 0, WS, big, ctypes.c_void_p(0), kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG


def test_call_flags_checked_before_cuda(lib):
    """A call's flags word: unknown bits or both engines are refused on the host; the
    duplicate check needs its table in the workspace (kvx_workspace_size covers it)."""
    src = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE, plane_stride=1000 * 256)
    dst = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE * 2, plane_stride=1000 * 256)
    WS, ST, SL = FAKE * 4, FAKE * 5, FAKE * 6
    l = kvx.lib()
    big = 1 << 30

    def tr(flags, ws_bytes=big):
        return l.kvx_transfer(src.handle, SL, dst.handle, SL, 3000, WS, ws_bytes, ST, flags, None)

    for bad in (0x10, 0x80000000, kvx.USE_REGISTERS | kvx.USE_BULK, 0xFFFFFFFE):
        assert tr(bad) == kvx.ERR_INVALID_ARG, hex(bad)
        assert l.kvx_batch(src.handle, dst.handle, FAKE * 8, 1, 10, SL, 10, SL, 10, None, 0, WS,
                           big, ST, bad, None) == kvx.ERR_INVALID_ARG
        assert l.kvx_stream(kvx.OP_TRANSFER, src.handle, SL, dst.handle, SL, 10, None, 0, None, WS,
                            big, ST, bad, None) == kvx.ERR_INVALID_ARG
    # 100,000 bytes hold the plan of 3000 tokens (two tiles of 32 KiB chunk tables) but not
    # the duplicate table after it (8 bytes x 8192 slots); kvx_workspace_size covers both
    assert kvx.workspace_size(3000) > 100_000
    assert tr(kvx.CHECK_DUP, 100_000) == kvx.ERR_NO_WORKSPACE
    assert tr(kvx.CHECK_DUP | kvx.USE_BULK, 100_000) == kvx.ERR_NO_WORKSPACE


def test_stream_validation_before_cuda(lib):
    """kvx_stream's control block and arguments are checked on the host, nothing enqueued."""
    src = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE, plane_stride=1000 * 256)
    dst = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE * 2, plane_stride=1000 * 256)
    WS, ST, SL = FAKE * 4, FAKE * 5, FAKE * 6
    big = 1 << 30
    l = kvx.lib()

    def call(ctl, status=ST, op=kvx.OP_TRANSFER, n=10, s=src, d=dst):
        return l.kvx_stream(op, s.handle, SL, d.handle, SL, n, None, 0,
                            None if ctl is None else ctypes.byref(ctl), WS, big, status, kvx.DEFAULTS, None)

    def ctl(**kw):
        c = kvx.StreamCtl()
        c.wait_ns = 1000
        for k, v in kw.items():
            setattr(c, k, v)
        return c

    assert call(None) == kvx.ERR_INVALID_ARG                             # no control block
    assert call(ctl(wait_ns=0)) == kvx.ERR_INVALID_ARG                   # unbounded wait
    assert call(ctl(wait_ns=kvx.MAX_WAIT_NS + 1)) == kvx.ERR_INVALID_ARG
    assert call(ctl(max_ctas=-1)) == kvx.ERR_INVALID_ARG
    assert call(ctl(reserved=1)) == kvx.ERR_INVALID_ARG
    assert call(ctl(), status=ST + 4) == kvx.ERR_INVALID_ARG             # status not 16-aligned
    assert call(ctl(), status=None) == kvx.ERR_INVALID_ARG
    assert call(ctl(), op=kvx.OP_BATCH) == kvx.ERR_INVALID_ARG
    assert call(ctl(), n=-1) == kvx.ERR_INVALID_ARG
    assert call(ctl(), d=src) == kvx.ERR_OVERLAP


def test_tp_slice_matches_oracle(lib):
    """kvx_tp_slice (host arithmetic in libkvx) against the oracle's plan, exhaustively for
    small sizes, including the refusals."""
    sizes = (1, 2, 3, 4, 6, 8, 16)
    for heads in (1, 2, 4, 6, 8):
        for st in sizes:
            for dt in sizes:
                for sr in range(-1, st + 1):
                    for dr in (0, dt - 1, dt):
                        want = oracle.tp_slice(heads, st, sr, dt, dr)
                        a, b, c = ctypes.c_int32(-7), ctypes.c_int32(-7), ctypes.c_int32(-7)
                        rc = kvx.lib().kvx_tp_slice(heads, st, sr, dt, dr, ctypes.byref(a),
                                                    ctypes.byref(b), ctypes.byref(c))
                        assert rc == want[0], (heads, st, sr, dt, dr)
                        if rc == kvx.OK:
                            assert (a.value, b.value, c.value) == want[1:], (heads, st, sr, dt, dr)


def test_move_heads_validation_before_cuda(lib):
    src = kvx.Layout(2, 4, 64, kvx.F16, 1000, base=FAKE, plane_stride=1000 * 512)
    dst = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE * 2, plane_stride=1000 * 256)
    odd = kvx.Layout(2, 2, 4, kvx.F16, 1000, base=FAKE * 3, plane_stride=1000 * 16)
    other = kvx.Layout(3, 2, 64, kvx.F16, 1000, base=FAKE * 3, plane_stride=1000 * 256)
    WS, ST, SL = FAKE * 4, FAKE * 5, FAKE * 6
    big = 1 << 30
    l = kvx.lib()

    def mv(op, s, h0, d, g0, nh, n=10, buf=None, bb=0):
        return l.kvx_move_heads(op, s and s.handle, SL, h0, d and d.handle, SL, g0, nh, n, buf, bb,
                                WS, big, ST, kvx.DEFAULTS, None)

    T, G, S = kvx.OP_TRANSFER, kvx.OP_GATHER, kvx.OP_SCATTER
    assert mv(T, src, 3, dst, 0, 2) == kvx.ERR_INVALID_ARG      # source range past kv_heads
    assert mv(T, src, 0, dst, 1, 2) == kvx.ERR_INVALID_ARG      # destination range past kv_heads
    assert mv(T, src, 0, dst, 0, 0) == kvx.ERR_INVALID_ARG      # no heads
    assert mv(T, src, -1, dst, 0, 1) == kvx.ERR_INVALID_ARG
    assert mv(T, src, 0, other, 0, 2) == kvx.ERR_INVALID_ARG    # layer counts differ
    assert mv(T, src, 0, src, 0, 2) == kvx.ERR_OVERLAP
    assert mv(T, None, 0, dst, 0, 1) == kvx.ERR_INVALID_ARG
    assert mv(G, src, 0, None, 0, 2, buf=None, bb=0) == kvx.ERR_INVALID_ARG   # gather needs a buffer
    assert mv(G, src, 0, None, 0, 2, buf=FAKE * 7, bb=4 * 10 * 256 - 16) == kvx.ERR_INVALID_ARG


def test_tp_plan_matches_oracle(lib):
    """kvx_tp_plan is kvx_tp_slice over every rank pair (the oracle's), pairs with nothing to
    send left out, destination rank major; too small an output array is refused but reports
    the count; sizes the slice refuses are refused."""
    for heads in (1, 2, 8):
        for p_tp in (1, 2, 4, 8, 16):
            for d_tp in (1, 2, 4, 8, 16):
                ok = oracle.tp_slice(heads, p_tp, 0, d_tp, 0)[0] == oracle.OK
                if not ok:
                    with pytest.raises(kvx.KvxError):
                        kvx.tp_plan(heads, p_tp, d_tp)
                    continue
                want = []
                for dr in range(d_tp):
                    for pr in range(p_tp):
                        rc, h0, g0, nh = oracle.tp_slice(heads, p_tp, pr, d_tp, dr)
                        if nh:
                            want.append((pr, dr, h0, g0, nh))
                assert kvx.tp_plan(heads, p_tp, d_tp) == want
    n = ctypes.c_int32(-1)
    arr = (kvx.HeadPart * 3)()
    assert kvx.lib().kvx_tp_plan(8, 8, 1, arr, 3, ctypes.byref(n)) == kvx.ERR_INVALID_ARG
    assert n.value == 8
    assert kvx.lib().kvx_tp_plan(8, 8, 1, None, 0, None) == kvx.ERR_INVALID_ARG
    assert kvx.lib().kvx_tp_plan(8, 2048, 1, None, 0, ctypes.byref(n)) == kvx.ERR_INVALID_ARG


def test_reshard_validation_before_cuda(lib):
    """kvx_reshard refuses, before any CUDA call, every malformed reshard: counts and limits,
    sources (or destinations) that are not the same pool shape, geometry differing between the
    sides, parts with bad indices, head ranges or unequal sizes, two parts writing one
    destination head, overlapping memory, pieces not 16-byte aligned, missing workspace."""
    mk = lambda k, h, ns=1000, **kw: kvx.Layout(2, h, 64, kvx.F16, ns, base=FAKE * k,
                                               plane_stride=ns * h * 128, **kw)
    p = [mk(1, 2), mk(2, 2)]            # P TP 2 of a 4-head model
    d = [mk(3, 4)]                      # D TP 1
    WS, ST, SL = FAKE * 6, FAKE * 7, FAKE * 8
    big = 1 << 30
    l = kvx.lib()
    good = [(0, 0, 0, 0, 2), (1, 0, 0, 2, 2)]

    def rs(srcs, dsts, parts, n=10, ws=WS, wsb=big, st=ST, sl=SL):
        sa = (ctypes.c_void_p * max(1, len(srcs)))(*[x.handle for x in srcs])
        da = (ctypes.c_void_p * max(1, len(dsts)))(*[x.handle for x in dsts])
        pa = (kvx.HeadPart * max(1, len(parts)))(*[kvx.HeadPart(*q) for q in parts])
        return l.kvx_reshard(sa, len(srcs), sl, da, len(dsts), sl, pa, len(parts), n, ws, wsb, st, kvx.DEFAULTS,
                             None)

    E, O, A = kvx.ERR_INVALID_ARG, kvx.ERR_OVERLAP, kvx.ERR_ALIGNMENT
    assert rs(p, d, []) == E                                         # no parts
    assert rs([], d, good) == E and rs(p, [], good) == E
    assert rs(p, d, [(0, 0, 0, 0, 2)] * 129) == E                    # over KVX_RESHARD_MAX_PARTS
    many = [mk(10 + k, 2) for k in range(64)]
    assert rs(many, d, good) == E                                    # over KVX_RESHARD_MAX_LAYOUTS
    assert rs([p[0], mk(4, 2, ns=999)], d, good) == E                # sources of different shape
    assert rs([p[0], mk(4, 4)], d, good) == E
    assert rs(p, [d[0], mk(4, 2)], good) == E                        # destinations of different shape
    three = kvx.Layout(3, 4, 64, kvx.F16, 1000, base=FAKE * 5, plane_stride=1000 * 512)
    assert rs(p, [three], good) == E                                 # layer counts differ
    assert rs(p, d, [(0, 0, 0, 0, 2), (1, 0, 0, 2, 1)]) == E         # unequal n_heads
    assert rs(p, d, [(2, 0, 0, 0, 2)]) == E                          # no source 2
    assert rs(p, d, [(0, 1, 0, 0, 2)]) == E                          # no destination 1
    assert rs(p, d, [(0, 0, 1, 0, 2)]) == E                          # past the source's heads
    assert rs(p, d, [(0, 0, 0, 3, 2)]) == E                          # past the destination's heads
    assert rs(p, d, [(0, 0, 0, 0, 2), (1, 0, 0, 1, 2)]) == E         # head 1 written twice
    assert rs(p, d, [(0, 0, 0, 0, 2, 1)]) == E                       # reserved not 0
    assert rs(p, d, [(0, 0, 0, 0, 0)]) == E                          # no heads
    assert rs(p, d, good, st=None) == E
    assert rs(p, d, good, n=-1) == E
    assert rs(p, [p[0]], [(0, 0, 0, 0, 2)]) == O                     # a source is a destination
    assert rs(p, [d[0], d[0]], [(0, 0, 0, 0, 2), (1, 1, 0, 0, 2)]) == O   # one pool twice
    narrow = [kvx.Layout(2, 2, 4, kvx.F16, 1000, base=FAKE * (20 + k), plane_stride=1000 * 16)
              for k in range(2)]
    nd = kvx.Layout(2, 4, 4, kvx.F16, 1000, base=FAKE * 30, plane_stride=1000 * 32)
    assert rs(narrow, [nd], [(0, 0, 0, 0, 1), (1, 0, 0, 1, 1)]) == A  # 8-byte pieces
    assert rs(p, d, good, ws=None) == kvx.ERR_NO_WORKSPACE
    assert rs(p, d, good, wsb=16) == kvx.ERR_NO_WORKSPACE
    assert rs(p, d, good, sl=None) == E


def test_stream_reshard_validation_before_cuda(lib):
    """kvx_stream_reshard refuses a negative CTA cap, a missing or malformed control block, a
    status array that is not 16-byte aligned, and every malformed reshard kvx_reshard refuses."""
    mk = lambda k, h: kvx.Layout(2, h, 64, kvx.F16, 1000, base=FAKE * k, plane_stride=1000 * h * 128)
    p = [mk(1, 2), mk(2, 2)]
    d = [mk(3, 4)]
    WS, ST, SL = FAKE * 6, FAKE * 7, FAKE * 8
    l = kvx.lib()

    def rs(parts, ctl, st=ST, srcs=p):
        sa = (ctypes.c_void_p * len(srcs))(*[x.handle for x in srcs])
        da = (ctypes.c_void_p * 1)(d[0].handle)
        pa = (kvx.HeadPart * max(1, len(parts)))(*[kvx.HeadPart(*q) for q in parts])
        return l.kvx_stream_reshard(sa, len(srcs), SL, da, 1, SL, pa, len(parts), 10,
                                    ctypes.byref(ctl) if ctl is not None else None, WS, 1 << 30,
                                    st, kvx.DEFAULTS, None)

    good = [(0, 0, 0, 0, 2), (1, 0, 0, 2, 2)]
    ok = kvx._stream_ctl(None, 1, None, 0, 1000, 0, None, None, 1)
    assert rs(good, None) == kvx.ERR_INVALID_ARG
    assert rs(good, kvx._stream_ctl(None, 1, None, 0, 1000, -1, None, None, 1)) == kvx.ERR_INVALID_ARG
    assert rs(good, kvx._stream_ctl(None, 1, None, 0, 0, 0, None, None, 1)) == kvx.ERR_INVALID_ARG
    assert rs(good, ok, st=ST + 4) == kvx.ERR_INVALID_ARG
    assert rs([(0, 0, 0, 0, 2), (1, 0, 0, 1, 2)], ok) == kvx.ERR_INVALID_ARG  # one head twice
    assert rs(good, ok, srcs=[p[0], d[0]]) == kvx.ERR_INVALID_ARG            # sources differ


def test_latent_plane_layouts(lib):
    """kv_planes: 1 (MLA latent, P = L) or 2 (default, P = 2L); anything else refused; latent
    and K/V layouts do not mix in one move."""
    mla = kvx.Layout(27, 1, 576, kvx.BF16, 1000, base=FAKE, plane_stride=1000 * 1152, kv_planes=1)
    assert mla.num_planes == 27 and mla.row_bytes == 1152
    kv = kvx.Layout(27, 1, 576, kvx.BF16, 1000, base=FAKE * 2, plane_stride=1000 * 1152)
    assert kv.num_planes == 54
    with pytest.raises(kvx.KvxError):
        kvx.Layout(2, 1, 64, kvx.BF16, 10, base=FAKE, plane_stride=4096, kv_planes=3)
    with pytest.raises(kvx.KvxError):
        kvx.Layout(200, 1, 64, kvx.BF16, 10, base=FAKE, plane_stride=4096)  # 400 planes
    kvx.Layout(200, 1, 64, kvx.BF16, 10, base=FAKE, plane_stride=4096, kv_planes=1).close()
    l = kvx.lib()
    assert l.kvx_transfer(mla.handle, FAKE * 6, kv.handle, FAKE * 6, 10, FAKE * 4, 1 << 30,
                          FAKE * 5, kvx.DEFAULTS, None) == kvx.ERR_INVALID_ARG


def test_stream_refuses_narrow_rows(lib):
    """kvx_stream moves 16-byte vectors only: a layout with 200-byte rows is refused before
    anything is enqueued."""
    src = kvx.Layout(2, 1, 100, kvx.F16, 1000, base=FAKE, plane_stride=1000 * 200)
    dst = kvx.Layout(2, 1, 100, kvx.F16, 1000, base=FAKE * 2, plane_stride=1000 * 200)
    c = kvx.StreamCtl()
    c.wait_ns = 1000
    rc = kvx.lib().kvx_stream(kvx.OP_TRANSFER, src.handle, FAKE * 6, dst.handle, FAKE * 6, 10,
                              None, 0, ctypes.byref(c), FAKE * 4, 1 << 30, FAKE * 5, kvx.DEFAULTS, None)
    assert rc == kvx.ERR_ALIGNMENT


def test_check_duplicates_switch(lib):
    assert kvx.get_check_duplicates() is False
    kvx.set_check_duplicates(True)
    assert kvx.get_check_duplicates() is True
    kvx.set_check_duplicates(False)
    assert kvx.lib().kvx_set_check_duplicates(2) == kvx.ERR_INVALID_ARG
    assert kvx.get_check_duplicates() is False


def test_stream_page_epochs_validation(lib):
    src = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE, plane_stride=1000 * 256)
    dst = kvx.Layout(2, 2, 64, kvx.F16, 1000, base=FAKE * 2, plane_stride=1000 * 256)
    c = kvx.StreamCtl()
    c.wait_ns = 1000
    c.dst_page_epochs = FAKE * 8
    c.epoch_page = 0  # page size missing
    l = kvx.lib()
    args = lambda op, s, d: (op, s and s.handle, FAKE * 6, d and d.handle, FAKE * 6, 10, FAKE * 7,
                             10 * 4 * 256, ctypes.byref(c), FAKE * 4, 1 << 30, FAKE * 5,
                             kvx.DEFAULTS, None)
    assert l.kvx_stream(*args(kvx.OP_TRANSFER, src, dst)) == kvx.ERR_INVALID_ARG
    c.epoch_page = 16
    assert l.kvx_stream(*args(kvx.OP_GATHER, src, None)) == kvx.ERR_INVALID_ARG  # no destination pool
    c.reserved2 = 1
    assert l.kvx_stream(*args(kvx.OP_TRANSFER, src, dst)) == kvx.ERR_INVALID_ARG


def test_header_compiles_as_strict_c99_and_cpp17(tmp_path):
    """kvx.h alone, as C99 and as C++17, with every warning an error."""
    c = tmp_path / "h.c"
    c.write_text('#include "kvx.h"\nint main(void) { return kvx_version() > 0 ? 0 : 1; }\n')
    for cmd in (["gcc", "-std=c99"], ["g++", "-std=c++17", "-x", "c++"]):
        subprocess.run(cmd + ["-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                              "-I", os.path.dirname(HEADER), str(c)], check=True)


def test_c_program_builds_against_the_library(lib, tmp_path):
    """The plain-C transfer program (run on the GPU by tests/test_gpu_c_abi.py) compiles as
    strict C99 and links against libkvx.so."""
    from tests.cprog import build_c_program
    exe = build_c_program(str(tmp_path / "transfer_from_c"))
    assert os.path.exists(exe)
