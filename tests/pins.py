"""Pins that tie the oracle to something other than itself.

Every function here takes the oracle's ctypes library and raises AssertionError when the
oracle disagrees with: a size the pages print (tests/golden/kv_sizes.json), the
element-by-element brute-force model (tests/bruteforce.py) on every small injective slot map
and page table, an invariant the pages state, or a numpy routine that the method reduces to
in a special case.  test_oracle_pins.py runs them against the real oracle;
test_oracle_mutants.py runs them against oracle builds with a planted mistake and expects a
failure for each one.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np

import oracle
from tests import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kv_sizes.json")
UNITS = {"KiB": 2 ** 10, "MiB": 2 ** 20, "GiB": 2 ** 30}

# tiny shapes: 2 layers (4 planes), 2 heads, head_dim 4 -> 16-byte rows
L, H, D = 2, 2, 4


def _arange_fill(start):
    return lambda n: (np.arange(n, dtype=np.int64) + start).astype(np.uint16)


def _sentinel_fill(n):
    return (0x7E00 | (np.arange(n) % 509)).astype(np.uint16)


def _bytes_of(buf5d):
    return np.ascontiguousarray(buf5d).view(np.uint8).reshape(-1)


def pin_sizes(lib):
    """[DistServe] B_KV and the pages' printed sizes (golden fixture)."""
    table = json.load(open(GOLDEN))
    for e in table["entries"]:
        per_tok = oracle.bytes_per_token(e["layers"], e["kv_heads"], e["head_dim"],
                                         e["elem_bytes"], lib=lib)
        total = per_tok * e["tokens"]
        assert total == e["bytes"], (e["name"], total, e["bytes"])
        assert abs(total / UNITS[e["unit"]] - e["stated"]) <= e["tol"], e["name"]
        if "per_token_bytes" in e:
            assert per_tok == e["per_token_bytes"]
            assert per_tok / UNITS[e["per_token_unit"]] == e["per_token_stated"]


def pin_bytes_written(lib):
    """The oracle reports n * P * R bytes moved, and R = kv_heads * head_dim * elem_bytes."""
    pool = bf.make_pool("planes", L, H, D, 8, _arange_fill(0))
    op = bf.to_oracle(pool)
    rc, buf, written = oracle.gather(op, [3, 1, 6], lib=lib)
    assert rc == oracle.OK
    assert written == 3 * 2 * L * H * D * 2 == buf.nbytes
    assert written == 3 * oracle.bytes_per_token(L, H, D, 2, lib=lib)


def _maps(num_slots, nmax):
    for n in range(nmax + 1):
        yield from itertools.permutations(range(num_slots), n)


def pin_bruteforce_gather(lib):
    """All injective slot maps of n <= 3 tokens from 4-slot pools, every layout."""
    for layout, ps in (("planes", 1), ("slot_major", 1), ("hnd", 2)):
        pool = bf.make_pool(layout, L, H, D, 4, _arange_fill(1), page_size=ps)
        op = bf.to_oracle(pool)
        before = pool.data.copy()
        for slots in _maps(4, 3):
            want = _bytes_of(bf.gather(pool, slots))
            rc, buf, _ = oracle.gather(op, list(slots), lib=lib)
            assert rc == oracle.OK
            assert np.array_equal(buf, want), (layout, slots)
        assert np.array_equal(pool.data, before), "source modified"


def pin_bruteforce_scatter(lib):
    for layout, ps in (("planes", 1), ("slot_major", 1), ("hnd", 2)):
        base = bf.make_pool(layout, L, H, D, 4, _sentinel_fill, page_size=ps)
        for slots in _maps(4, 3):
            n = len(slots)
            buf = (np.arange(L * 2 * n * H * D) + 100).astype(np.uint16).reshape(L, 2, n, H, D)
            want = bf.scatter(base, slots, buf)
            buf_before = buf.copy()
            pool = base.copy()
            rc, _ = oracle.scatter(bf.to_oracle(pool), list(slots), buf, lib=lib)
            assert rc == oracle.OK
            assert np.array_equal(pool.data, want.data), (layout, slots)
            assert np.array_equal(buf, buf_before), "buffer modified"


def pin_bruteforce_transfer(lib):
    """Every pair of injective maps with n <= 2 between every pair of layouts."""
    layouts = (("planes", 1), ("slot_major", 1), ("hnd", 2))
    for (la, pa), (lb, pb) in itertools.product(layouts, layouts):
        src = bf.make_pool(la, L, H, D, 4, _arange_fill(1), page_size=pa)
        base = bf.make_pool(lb, L, H, D, 4, _sentinel_fill, page_size=pb)
        for n in range(3):
            for s in itertools.permutations(range(4), n):
                for d in itertools.permutations(range(4), n):
                    want = bf.transfer(src, s, base, d)
                    src_before = src.data.copy()
                    dst = base.copy()
                    rc, _ = oracle.transfer(bf.to_oracle(src), list(s), bf.to_oracle(dst),
                                            list(d), lib=lib)
                    assert rc == oracle.OK
                    assert np.array_equal(dst.data, want.data), (la, lb, s, d)
                    assert np.array_equal(src.data, src_before), "source modified"


def pin_bruteforce_transfer_layers(lib):
    """Every stop layer (0 .. L) of a layer-streamed transfer, for every pair of layouts and
    every injective map with n <= 2; bytes written = n * 2 * stop * R; stop outside [0, L]
    refused with nothing written."""
    layouts = (("planes", 1), ("slot_major", 1), ("hnd", 2))
    R = H * D * 2
    for (la, pa), (lb, pb) in itertools.product(layouts, layouts):
        src = bf.make_pool(la, L, H, D, 4, _arange_fill(3), page_size=pa)
        base = bf.make_pool(lb, L, H, D, 4, _sentinel_fill, page_size=pb)
        for n in range(3):
            for s in itertools.permutations(range(4), n):
                d = tuple(reversed(range(4)))[:n]
                for stop in range(L + 1):
                    want = bf.transfer_layers(src, s, base, d, stop)
                    dst = base.copy()
                    rc, written = oracle.transfer_layers(bf.to_oracle(src), list(s),
                                                         bf.to_oracle(dst), list(d), stop, lib=lib)
                    assert rc == oracle.OK and written == n * 2 * stop * R
                    assert np.array_equal(dst.data, want.data), (la, lb, s, stop)
        for bad in (-1, L + 1):
            dst = base.copy()
            rc, _ = oracle.transfer_layers(bf.to_oracle(src), [0], bf.to_oracle(dst), [1], bad,
                                           lib=lib)
            assert rc == oracle.ERR_INVALID_ARG and np.array_equal(dst.data, base.data)


def pin_bruteforce_transfer_owned(lib):
    """Rows whose destination page changed owner are never written: every owner pattern of a
    4-slot pool in pages of 1 and 2 slots, every stop layer, every layout pair, n <= 2 maps;
    every page owned gives the layer-range transfer, no page owned leaves the pool alone."""
    layouts = (("planes", 1), ("slot_major", 1), ("hnd", 2))
    R = H * D * 2
    for (la, pa), (lb, pb) in itertools.product(layouts, layouts):
        src = bf.make_pool(la, L, H, D, 4, _arange_fill(9), page_size=pa)
        base = bf.make_pool(lb, L, H, D, 4, _sentinel_fill, page_size=pb)
        for ep in (1, 2):
            for owners in itertools.product((5, 6), repeat=4 // ep):
                for n in (1, 2):
                    s_, d_ = [2, 0][:n], [3, 1][:n]
                    for stop in range(L + 1):
                        want = bf.transfer_owned(src, s_, base, d_, stop, owners, ep, 5)
                        dst = base.copy()
                        rc, w = oracle.transfer_owned(bf.to_oracle(src), s_, bf.to_oracle(dst),
                                                      d_, stop, list(owners), ep, 5, lib=lib)
                        moved = sum(owners[x // ep] == 5 for x in d_)
                        assert rc == oracle.OK and w == moved * 2 * stop * R
                        assert np.array_equal(dst.data, want.data), (la, lb, ep, owners, stop)
        full = base.copy()
        oracle.transfer_layers(bf.to_oracle(src), [2, 0], bf.to_oracle(full), [3, 1], L, lib=lib)
        dst = base.copy()
        oracle.transfer_owned(bf.to_oracle(src), [2, 0], bf.to_oracle(dst), [3, 1], L, [5] * 4, 1, 5,
                              lib=lib)
        assert np.array_equal(dst.data, full.data)
        dst = base.copy()
        oracle.transfer_owned(bf.to_oracle(src), [2, 0], bf.to_oracle(dst), [3, 1], L, [6] * 4, 1, 5,
                              lib=lib)
        assert np.array_equal(dst.data, base.data)


def pin_bruteforce_move_heads(lib):
    """Head-range gather / scatter / transfer between pools with different kv_heads, for every
    pair of layouts, every valid (src_head0, dst_head0, n_heads) and n <= 2; bad head ranges
    refused with nothing written."""
    layouts = (("planes", 1), ("slot_major", 1), ("hnd", 2))
    for (la, pa), (lb, pb) in itertools.product(layouts, layouts):
        for hs, hd in ((3, 2), (2, 3), (1, 2)):
            src = bf.make_pool(la, L, hs, D, 4, _arange_fill(5), page_size=pa)
            base = bf.make_pool(lb, L, hd, D, 4, _sentinel_fill, page_size=pb)
            for nh in range(1, min(hs, hd) + 1):
                for h0 in range(hs - nh + 1):
                    for g0 in range(hd - nh + 1):
                        for n in (1, 2):
                            s_, d_ = [3, 0][:n], [1, 2][:n]
                            want = bf.move_heads(2, src, s_, h0, base, d_, g0, nh)
                            dst = base.copy()
                            rc, _, w = oracle.move_heads(2, bf.to_oracle(src), s_, h0,
                                                         bf.to_oracle(dst), d_, g0, nh, n, lib=lib)
                            assert rc == oracle.OK and w == n * 2 * L * nh * D * 2
                            assert np.array_equal(dst.data, want.data), (la, lb, hs, hd, h0, g0, nh)
                            rc, got, _ = oracle.move_heads(0, bf.to_oracle(src), s_, h0, None, None,
                                                           0, nh, n, lib=lib)
                            gb = bf.move_heads(0, src, s_, h0, None, None, 0, nh)
                            assert rc == oracle.OK
                            assert np.array_equal(got[: gb.size * 2].view(np.uint16), gb.ravel())
                            dst = base.copy()
                            rc, _, _ = oracle.move_heads(1, None, None, 0, bf.to_oracle(dst), d_,
                                                         g0, nh, n, buf=gb.view(np.uint8), lib=lib)
                            want = bf.move_heads(1, None, None, 0, base, d_, g0, nh, buf=gb)
                            assert rc == oracle.OK and np.array_equal(dst.data, want.data)
            for h0, g0, nh in ((hs, 0, 1), (0, hd, 1), (0, 0, 0), (-1, 0, 1)):
                dst = base.copy()
                rc, _, _ = oracle.move_heads(2, bf.to_oracle(src), [0], h0, bf.to_oracle(dst), [1],
                                             g0, nh, 1, lib=lib)
                assert rc == oracle.ERR_INVALID_ARG and np.array_equal(dst.data, base.data)


def pin_move_heads_full_range_is_transfer(lib):
    """Moving every head (same kv_heads on both sides) is the plain transfer."""
    src = bf.make_pool("planes", L, H, D, 4, _arange_fill(7))
    a = bf.make_pool("hnd", L, H, D, 4, _sentinel_fill, page_size=2)
    b = a.copy()
    rc1, _, _ = oracle.move_heads(2, bf.to_oracle(src), [2, 1], 0, bf.to_oracle(a), [0, 3], 0, H, 2,
                                  lib=lib)
    rc2, _ = oracle.transfer(bf.to_oracle(src), [2, 1], bf.to_oracle(b), [0, 3], lib=lib)
    assert rc1 == rc2 == oracle.OK and np.array_equal(a.data, b.data)


def pin_tp_slice(lib):
    """The heterogeneous-TP transfer plan.  Worked cases of the passage (8 kv heads): P TP 4 ->
    D TP 2 merges two P shards into each D shard; P TP 2 -> D TP 4 splits each P shard over two
    D ranks.  Exhaustively for small sizes: every D rank receives each of its heads exactly
    once, from a P rank that holds it, at the matching offsets."""
    # P TP 4 (2 heads each) -> D TP 2 (4 heads each): D rank 0 <- P ranks 0, 1
    assert oracle.tp_slice(8, 4, 0, 2, 0, lib=lib) == (oracle.OK, 0, 0, 2)
    assert oracle.tp_slice(8, 4, 1, 2, 0, lib=lib) == (oracle.OK, 0, 2, 2)
    assert oracle.tp_slice(8, 4, 2, 2, 0, lib=lib)[3] == 0
    assert oracle.tp_slice(8, 4, 3, 2, 1, lib=lib) == (oracle.OK, 0, 2, 2)
    # P TP 2 (4 heads each) -> D TP 4 (2 heads each): P rank 1 -> D ranks 2, 3
    assert oracle.tp_slice(8, 2, 1, 4, 2, lib=lib) == (oracle.OK, 0, 0, 2)
    assert oracle.tp_slice(8, 2, 1, 4, 3, lib=lib) == (oracle.OK, 2, 0, 2)
    assert oracle.tp_slice(8, 2, 1, 4, 0, lib=lib)[3] == 0
    # replicated producer (2 kv heads, P TP 4): ranks 0 and 2 send, 1 and 3 are replicas
    assert oracle.tp_slice(2, 4, 0, 1, 0, lib=lib) == (oracle.OK, 0, 0, 1)
    assert oracle.tp_slice(2, 4, 1, 1, 0, lib=lib)[3] == 0
    assert oracle.tp_slice(2, 4, 2, 1, 0, lib=lib) == (oracle.OK, 0, 1, 1)

    def held(heads, t, r):
        if t <= heads:
            return list(range(r * heads // t, (r + 1) * heads // t))
        return [r // (t // heads)]

    sizes = (1, 2, 4, 8, 16)
    for heads in (1, 2, 4, 8):
        for p_tp in sizes:
            for d_tp in sizes:
                ok = lambda t: (heads % t == 0) if t <= heads else (t % heads == 0)
                if not (ok(p_tp) and ok(d_tp)):
                    assert oracle.tp_slice(heads, p_tp, 0, d_tp, 0, lib=lib)[0] == oracle.ERR_INVALID_ARG
                    continue
                for dr in range(d_tp):
                    got = []
                    for pr in range(p_tp):
                        rc, sh0, dh0, nh = oracle.tp_slice(heads, p_tp, pr, d_tp, dr, lib=lib)
                        assert rc == oracle.OK
                        for j in range(nh):
                            g_src = held(heads, p_tp, pr)[sh0 + j]
                            g_dst = held(heads, d_tp, dr)[dh0 + j]
                            assert g_src == g_dst
                            got.append(g_dst)
                    assert sorted(got) == held(heads, d_tp, dr), (heads, p_tp, d_tp, dr)
    for bad in ((0, 1, 0, 1, 0), (8, 3, 0, 1, 0), (8, 2, 2, 1, 0), (8, 1, 0, 2, -1), (2, 3, 0, 1, 0)):
        assert oracle.tp_slice(*bad, lib=lib)[0] == oracle.ERR_INVALID_ARG


def _tp_parts(heads, p_tp, d_tp, lib):
    """(pr, dr, h0, g0, nh) for every pair the oracle's tp_slice plan connects."""
    parts = []
    for dr in range(d_tp):
        for pr in range(p_tp):
            rc, h0, g0, nh = oracle.tp_slice(heads, p_tp, pr, d_tp, dr, lib=lib)
            assert rc == oracle.OK
            if nh:
                parts.append((pr, dr, h0, g0, nh))
    return parts


def pin_bruteforce_reshard(lib):
    """A whole TP reshard in one call against the element-by-element model of its parts, for
    merges (4 -> 2, 2 -> 1), splits (1 -> 2, 2 -> 4), replicated heads (2 -> 4 with 2 heads)
    and layout pairs; then the refusals: two parts writing one destination head, a part
    naming no pool, a head range past a pool, and a slot valid in one pool of a side but not
    in another -- each with nothing written."""
    heads = 4
    layouts = (("planes", 1), ("hnd", 2), ("slot_major", 1))
    for (la, pa), (lb, pb) in itertools.product(layouts, layouts):
        for p_tp, d_tp, hh in ((4, 2, 4), (2, 1, 4), (1, 2, 4), (2, 4, 4), (2, 4, 2)):
            parts = _tp_parts(hh, p_tp, d_tp, lib)
            srcs = [bf.make_pool(la, L, max(1, hh // p_tp), D, 4, _arange_fill(11 + r),
                                 page_size=pa) for r in range(p_tp)]
            base = [bf.make_pool(lb, L, max(1, hh // d_tp), D, 4, _sentinel_fill, page_size=pb)
                    for _ in range(d_tp)]
            for s_, d_ in (([3], [1]), ([3, 0], [1, 2]), ([], [])):
                want = bf.reshard(srcs, s_, base, d_, parts)
                got = [b.copy() for b in base]
                rc, w = oracle.reshard([bf.to_oracle(x) for x in srcs], s_,
                                       [bf.to_oracle(x) for x in got], d_, parts, len(s_), lib=lib)
                assert rc == oracle.OK, (la, lb, p_tp, d_tp)
                assert w == sum(len(s_) * 2 * L * q[4] * D * 2 for q in parts)
                for g, e in zip(got, want):
                    assert np.array_equal(g.data, e.data), (la, lb, p_tp, d_tp, hh, s_)
    srcs = [bf.make_pool("planes", L, 2, D, 4, _arange_fill(3 + r)) for r in range(2)]
    small = bf.make_pool("planes", L, 2, D, 3, _sentinel_fill)
    base = [bf.make_pool("hnd", L, 4, D, 4, _sentinel_fill, page_size=2) for _ in range(2)]
    bad = {
        "one head written twice": ([(0, 0, 0, 0, 2), (1, 0, 1, 1, 1)], base),
        "no such source": ([(2, 0, 0, 0, 1)], base),
        "no such destination": ([(0, 2, 0, 0, 1)], base),
        "head past the source": ([(0, 0, 1, 0, 2)], base),
        "head past the destination": ([(0, 1, 0, 3, 2)], base),
        "no heads": ([(0, 0, 0, 0, 0)], base),
        "no parts": ([], base),
    }
    for name, (parts, dsts) in bad.items():
        got = [b.copy() for b in dsts]
        rc, _ = oracle.reshard([bf.to_oracle(x) for x in srcs], [1], [bf.to_oracle(x) for x in got],
                               [0], parts, 1, lib=lib)
        assert rc == oracle.ERR_INVALID_ARG, name
        assert all(np.array_equal(g.data, b.data) for g, b in zip(got, dsts)), name
    # slot 3 is valid in the first destination pool, not in the second (3 slots): refused,
    # although only the first pool is written by the part
    got = [base[0].copy(), small.copy()]
    rc, _ = oracle.reshard([bf.to_oracle(x) for x in srcs], [0, 1],
                           [bf.to_oracle(x) for x in got], [0, 3], [(0, 0, 0, 0, 2)], 2, lib=lib)
    assert rc == oracle.ERR_OUT_OF_RANGE
    assert np.array_equal(got[0].data, base[0].data) and np.array_equal(got[1].data, small.data)
    got = [b.copy() for b in base]
    rc, _ = oracle.reshard([bf.to_oracle(srcs[0]), bf.to_oracle(small)], [3, 0],
                           [bf.to_oracle(x) for x in got], [0, 1], [(0, 0, 0, 0, 2)], 2, lib=lib)
    assert rc == oracle.ERR_OUT_OF_RANGE
    assert all(np.array_equal(g.data, b.data) for g, b in zip(got, base))


def pin_reshard_reassembles_model(lib):
    """What a reshard must achieve, stated without parts: a model's KV (8 kv heads) split by
    heads over the pools of a P TP group and resharded with the tp_slice plan leaves in every
    D rank's pool, at each destination slot, exactly that rank's heads of the model's rows at
    the matching source slot (numpy slicing of the whole-model pool, replicated heads
    included); every other slot keeps its bytes."""
    heads, L2, D2, ns = 8, 2, 4, 6
    full = np.arange(2 * L2 * ns * heads * D2, dtype=np.uint16).reshape(2 * L2, ns, heads, D2)
    full = (full * 7 + 3).astype(np.uint16)
    s_, d_ = [5, 0, 2], [1, 4, 3]

    def shard(t, r):  # heads of rank r in a group of size t
        if t <= heads:
            return list(range(r * heads // t, (r + 1) * heads // t))
        return [r // (t // heads)]

    for p_tp, d_tp in ((1, 8), (8, 1), (2, 4), (4, 2), (16, 2), (2, 16), (8, 8), (1, 1)):
        srcs = [bf.BFPool("planes", L2, len(shard(p_tp, r)), D2, ns,
                          np.ascontiguousarray(full[:, :, shard(p_tp, r)])) for r in range(p_tp)]
        dsts = [bf.make_pool("planes", L2, len(shard(d_tp, r)), D2, ns, _sentinel_fill)
                for r in range(d_tp)]
        before = [x.data.copy() for x in dsts]
        parts = _tp_parts(heads, p_tp, d_tp, lib)
        rc, _ = oracle.reshard([bf.to_oracle(x) for x in srcs], s_, [bf.to_oracle(x) for x in dsts],
                               d_, parts, len(s_), lib=lib)
        assert rc == oracle.OK
        for r, x in enumerate(dsts):
            want = before[r].copy()
            want[:, d_] = full[:, s_][:, :, shard(d_tp, r)]
            assert np.array_equal(x.data, want), (p_tp, d_tp, r)


def pin_mla(lib):
    """One latent plane per layer (MLA).  Sizes from the pages' table ([mini-infer] KV 传输大小):
    DeepSeek-V2-Lite (27 layers, latent 512 + rope 64, 2-byte elements) 3.80 MB at 128 tokens
    and 30.38 MB at 1024, about 54 % of Qwen2.5-7B's 7.00 MB.  Brute force: gather, scatter,
    transfer and the layer-range transfer of kv_planes = 1 pools for every pair of layouts."""
    gold = json.load(open(os.path.join(os.path.dirname(GOLDEN), "mla_sizes.json")))
    for e in gold["entries"]:
        got = oracle.mla_bytes_per_token(e["layers"], e["latent_dim"], e["rope_dim"],
                                         e["elem_bytes"], lib=lib) * e["tokens"]
        assert got == e["bytes"], e["name"]
        assert abs(got / 2**20 - e["stated"]) <= e["tol"], e["name"]
    mla = oracle.mla_bytes_per_token(27, 512, 64, 2, lib=lib)
    gqa7b = oracle.bytes_per_token(28, 4, 128, 2, lib=lib)
    r = gold["ratio_to_qwen25_7b"]
    assert abs(mla / gqa7b - r["stated"]) <= r["tol"]
    layouts = (("planes", 1), ("slot_major", 1), ("hnd", 2))
    R = H * D * 2
    for (la, pa), (lb, pb) in itertools.product(layouts, layouts):
        src = bf.make_pool(la, L, H, D, 4, _arange_fill(11), page_size=pa, kvp=1)
        base = bf.make_pool(lb, L, H, D, 4, _sentinel_fill, page_size=pb, kvp=1)
        s_, d_ = [2, 0, 3], [1, 3, 0]
        dst = base.copy()
        rc, w = oracle.transfer(bf.to_oracle(src), s_, bf.to_oracle(dst), d_, lib=lib)
        assert rc == oracle.OK and w == 3 * L * R
        assert np.array_equal(dst.data, bf.transfer(src, s_, base, d_).data), (la, lb)
        for stop in range(L + 1):
            dst = base.copy()
            rc, w = oracle.transfer_layers(bf.to_oracle(src), s_, bf.to_oracle(dst), d_, stop,
                                           lib=lib)
            assert rc == oracle.OK and w == 3 * stop * R
            assert np.array_equal(dst.data, bf.transfer_layers(src, s_, base, d_, stop).data)
        rc, got, w = oracle.gather(bf.to_oracle(src), s_, lib=lib)
        want = bf.gather(src, s_)
        assert rc == oracle.OK and w == want.size * 2
        assert np.array_equal(got.view(np.uint16), want.ravel())
        dst = base.copy()
        rc, _ = oracle.scatter(bf.to_oracle(dst), d_, want.view(np.uint8), lib=lib)
        assert rc == oracle.OK and np.array_equal(dst.data, bf.scatter(base, d_, want).data)
    # K/V pools and latent pools do not mix
    a = bf.make_pool("planes", L, H, D, 4, _arange_fill(1))
    b = bf.make_pool("planes", L, H, D, 4, _sentinel_fill, kvp=1)
    rc, _ = oracle.transfer(bf.to_oracle(a), [0], bf.to_oracle(b), [1], lib=lib)
    assert rc == oracle.ERR_INVALID_ARG


def pin_bruteforce_hnd(lib):
    """Every page table of k <= 3 pages out of a 4-page pool (page size 3), every sequence
    length that ends in page k, for the page-table gather and the inverse rebuild."""
    ps = 3
    src = bf.make_pool("hnd", L, H, D, 4 * ps, _arange_fill(1), page_size=ps)
    base = bf.make_pool("hnd", L, H, D, 4 * ps, _sentinel_fill, page_size=ps)
    for k in range(1, 4):
        for pt in itertools.permutations(range(4), k):
            for seq in range((k - 1) * ps + 1, k * ps + 1):
                want = bf.hnd_gather(src, pt, seq)
                rc, buf = oracle.hnd_gather(bf.to_oracle(src), list(pt), seq, lib=lib)
                assert rc == oracle.OK
                assert np.array_equal(buf, _bytes_of(want)), (pt, seq)
                dst = base.copy()
                assert oracle.hnd_rebuild(bf.to_oracle(dst), list(pt), seq, want,
                                          lib=lib) == oracle.OK
                slots = [pt[s // ps] * ps + s % ps for s in range(seq)]
                assert np.array_equal(dst.data, bf.scatter(base, slots, want).data), (pt, seq)


def pin_roundtrip(lib):
    """[PD-budget] 5090 section: gather into staging, scatter back.  Scattering the gathered
    rows to the same slots leaves the pool unchanged; into a sentinel pool those slots equal
    the source and every other slot keeps its sentinel."""
    g = np.random.Generator(np.random.PCG64(7))
    for layout, ps in (("planes", 1), ("slot_major", 1), ("hnd", 4)):
        src = bf.make_pool(layout, 3, 2, 8, 64, lambda n: g.integers(0, 0x7C00, n), ps)
        slots = g.choice(64, 20, replace=False)
        rc, buf, _ = oracle.gather(bf.to_oracle(src), slots, lib=lib)
        assert rc == oracle.OK
        same = src.copy()
        assert oracle.scatter(bf.to_oracle(same), slots, buf, lib=lib)[0] == oracle.OK
        assert np.array_equal(same.data, src.data)
        sent = bf.make_pool(layout, 3, 2, 8, 64, _sentinel_fill, ps)
        ref = sent.copy()
        assert oracle.scatter(bf.to_oracle(sent), slots, buf, lib=lib)[0] == oracle.OK
        touched = set(int(s) for s in slots)
        for layer in range(3):
            for kv in range(2):
                for slot in range(64):
                    a = [sent.get(layer, kv, slot, h, d) for h in range(2) for d in range(8)]
                    b = [(src if slot in touched else ref).get(layer, kv, slot, h, d)
                         for h in range(2) for d in range(8)]
                    assert a == b, (layout, layer, kv, slot)


def pin_transfer_is_scatter_of_gather(lib):
    """[PD-budget]: the B300 direct write and the 5090 staging + scatter reach the same bytes."""
    g = np.random.Generator(np.random.PCG64(11))
    src = bf.make_pool("planes", 2, 2, 8, 50, lambda n: g.integers(0, 0x7C00, n))
    s = g.choice(50, 17, replace=False)
    d = g.choice(40, 17, replace=False)
    a = bf.make_pool("slot_major", 2, 2, 8, 40, _sentinel_fill)
    b = a.copy()
    assert oracle.transfer(bf.to_oracle(src), s, bf.to_oracle(a), d, lib=lib)[0] == oracle.OK
    rc, buf, _ = oracle.gather(bf.to_oracle(src), s, lib=lib)
    assert rc == oracle.OK
    assert oracle.scatter(bf.to_oracle(b), d, buf, lib=lib)[0] == oracle.OK
    assert np.array_equal(a.data, b.data)


def pin_hnd_roundtrip(lib):
    """[mini-infer]: permute on extract and the inverse permute on rebuild are the identity."""
    g = np.random.Generator(np.random.PCG64(13))
    ps = 4
    src = bf.make_pool("hnd", 2, 3, 8, 16 * ps, lambda n: g.integers(0, 0x7C00, n), ps)
    pt = g.choice(16, 5, replace=False)
    seq = 4 * ps + 2  # last page partial
    rc, buf = oracle.hnd_gather(bf.to_oracle(src), pt, seq, lib=lib)
    assert rc == oracle.OK
    dst = bf.make_pool("hnd", 2, 3, 8, 16 * ps, _sentinel_fill, ps)
    ref = dst.copy()
    assert oracle.hnd_rebuild(bf.to_oracle(dst), pt, seq, buf, lib=lib) == oracle.OK
    rc, buf2 = oracle.hnd_gather(bf.to_oracle(dst), pt, seq, lib=lib)
    assert np.array_equal(buf, buf2)
    # the tail of the last page and all other pages keep their sentinel
    touched = {int(pt[s // ps]) * ps + s % ps for s in range(seq)}
    for slot in range(16 * ps):
        if slot in touched:
            continue
        for layer in range(2):
            for kv in range(2):
                for h in range(3):
                    assert dst.get(layer, kv, slot, h, 0) == ref.get(layer, kv, slot, h, 0)


def pin_plane_locality(lib):
    """[DistServe] 第三步: layer j of P goes only to layer j of D (plane p only to plane p)."""
    P = 2 * 3
    src = bf.make_pool("planes", 3, 1, 8, 10, lambda n: np.repeat(np.arange(P) + 1, n // P))
    dst = bf.make_pool("planes", 3, 1, 8, 10, lambda n: np.zeros(n))
    assert oracle.transfer(bf.to_oracle(src), [1, 5, 9], bf.to_oracle(dst), [0, 2, 4],
                           lib=lib)[0] == oracle.OK
    for p in range(P):
        assert set(np.unique(dst.data[p])) <= {0, p + 1}
        assert (dst.data[p, [0, 2, 4]] == p + 1).all()


def pin_numpy_special_cases(lib):
    """Per-plane token rows: the gather is numpy fancy indexing pool[:, slots].  HND pages:
    it is transpose(1, 0, 2) of the page-table view [heads, seq, dim] ([mini-infer])."""
    g = np.random.Generator(np.random.PCG64(17))
    pool = bf.make_pool("planes", 3, 2, 8, 40, lambda n: g.integers(0, 0x7C00, n))
    slots = g.choice(40, 13, replace=False)
    rc, buf, _ = oracle.gather(bf.to_oracle(pool), slots, lib=lib)
    assert np.array_equal(buf, _bytes_of(pool.data[:, slots]))
    ps = 4
    hp = bf.make_pool("hnd", 3, 2, 8, 12 * ps, lambda n: g.integers(0, 0x7C00, n), ps)
    pt = g.choice(12, 3, replace=False)
    seq = 2 * ps + 3
    rc, buf = oracle.hnd_gather(bf.to_oracle(hp), pt, seq, lib=lib)
    s = np.arange(seq)
    planes = []
    for p in range(6):
        view = hp.data[p][pt[s // ps], :, s % ps, :]  # [seq, heads, dim] via fancy indexing
        hsd = np.transpose(view, (1, 0, 2))           # the [heads, seq, dim] cache view
        planes.append(np.transpose(hsd, (1, 0, 2)))   # permute(1, 0, 2)
    assert np.array_equal(buf, _bytes_of(np.stack(planes)))


def pin_validation(lib):
    """Out-of-range slots (== num_slots, negative) fail with OUT_OF_RANGE and write nothing;
    duplicate destinations fail only when checked."""
    pool = bf.make_pool("planes", L, H, D, 8, _sentinel_fill)
    keep = pool.data.copy()
    buf = np.arange(L * 2 * 3 * H * D, dtype=np.uint16)
    for bad in ([0, 8, 1], [0, -1, 1], [2147483647]):
        rc, _ = oracle.scatter(bf.to_oracle(pool), bad, buf[: L * 2 * len(bad) * H * D], lib=lib)
        assert rc == oracle.ERR_OUT_OF_RANGE
        assert np.array_equal(pool.data, keep)
    src = bf.make_pool("planes", L, H, D, 8, _arange_fill(0))
    assert oracle.gather(bf.to_oracle(src), [7, 8], lib=lib)[0] == oracle.ERR_OUT_OF_RANGE
    assert oracle.gather(bf.to_oracle(src), [7, 0], lib=lib)[0] == oracle.OK
    rc, _ = oracle.transfer(bf.to_oracle(src), [1, 2], bf.to_oracle(pool), [3, 8], lib=lib)
    assert rc == oracle.ERR_OUT_OF_RANGE and np.array_equal(pool.data, keep)
    rc, _ = oracle.scatter(bf.to_oracle(pool), [1, 1], buf[: L * 2 * 2 * H * D], check_dup=True,
                           lib=lib)
    assert rc == oracle.ERR_DUPLICATE_DST and np.array_equal(pool.data, keep)
    rc, _ = oracle.scatter(bf.to_oracle(pool), [1, 1], buf[: L * 2 * 2 * H * D], lib=lib)
    assert rc == oracle.OK
    hp = bf.make_pool("hnd", L, H, D, 8, _arange_fill(0), page_size=2)
    assert oracle.hnd_gather(bf.to_oracle(hp), [3, 4], 3, lib=lib)[0] == oracle.ERR_OUT_OF_RANGE
    assert oracle.hnd_gather(bf.to_oracle(hp), [3, 0], 3, lib=lib)[0] == oracle.OK


def pin_batch(lib):
    """[Mooncake] 6.1: a batch equals its requests applied one by one; a bad request reports
    its own status and moves nothing, the others still run."""
    g = np.random.Generator(np.random.PCG64(19))
    src = bf.make_pool("planes", L, H, D, 30, lambda n: g.integers(0, 0x7C00, n))
    dst0 = bf.make_pool("planes", L, H, D, 30, _sentinel_fill)
    R = H * D * 2
    P = 2 * L
    ss = g.choice(30, 12, replace=False).astype(np.int32)
    ds = g.choice(30, 12, replace=False).astype(np.int32)
    ss_bad = ss.copy()
    ss_bad[5] = 30  # request 1 (tokens 4..7 of the source list) goes out of range
    buf0 = np.zeros(2 * P * 4 * R, dtype=np.uint8)
    reqs = [(oracle.OP_TRANSFER, 4, 0, 0, 0), (oracle.OP_TRANSFER, 4, 4, 4, 0),
            (oracle.OP_GATHER, 4, 8, 0, 0), (oracle.OP_SCATTER, 4, 0, 8, P * 4 * R)]
    buf = buf0.copy()
    buf[P * 4 * R:] = g.integers(0, 255, P * 4 * R, dtype=np.uint8)
    dst = dst0.copy()
    st = oracle.batch(bf.to_oracle(src), bf.to_oracle(dst), reqs, ss_bad, ds, buf, lib=lib)
    assert list(st) == [oracle.ERR_OUT_OF_RANGE, 0, oracle.ERR_OUT_OF_RANGE, 0, 0]
    # expected: apply the good requests one by one with the element model
    exp = bf.transfer(src, ss[0:4], dst0, ds[0:4])
    want_gather = _bytes_of(bf.gather(src, ss[8:12]))
    assert np.array_equal(buf[: P * 4 * R], want_gather)
    sc = buf[P * 4 * R:].view(np.uint16).reshape(L, 2, 4, H, D)
    exp = bf.scatter(exp, ds[8:12], sc)
    assert np.array_equal(dst.data, exp.data)
    # bad records
    st = oracle.batch(bf.to_oracle(src), bf.to_oracle(dst), [(7, 1, 0, 0, 0), (0, -1, 0, 0, 0),
                      (0, 4, 10, 0, 0), (0, 4, 0, 0, 8)], ss, ds, buf, lib=lib)
    assert list(st) == [1, 1, 1, 1, 1]


def pin_batch_duplicates(lib):
    """The duplicate check of a batch, against a brute-force model written from its rule: the
    requests that pass their own checks and write into the pool are compared pairwise (and each
    with itself) for a shared destination slot; every request in such a pair fails with
    DUPLICATE_DST and moves nothing; the remaining requests are applied one by one with the
    element model.  Statuses, the destination pool and the buffer must all agree, on a fixed
    case (two transfers sharing a slot, a transfer repeating a slot, a refused transfer sharing
    a slot with one that must still move) and on random batches over a 12-slot pool."""
    g = np.random.Generator(np.random.PCG64(29))
    R = H * D * 2
    P = 2 * L

    def model(src, dst0, reqs, ss, ds, buf0):
        ok = []
        for op, n, so, do, bo in reqs:
            s_ok = op == oracle.OP_SCATTER or all(0 <= x < src.num_slots for x in ss[so:so + n])
            d_ok = op == oracle.OP_GATHER or all(0 <= x < dst0.num_slots for x in ds[do:do + n])
            ok.append(oracle.OK if (s_ok and d_ok) else oracle.ERR_OUT_OF_RANGE)
        writes = [q for q, r in enumerate(reqs) if ok[q] == oracle.OK and r[0] != oracle.OP_GATHER]
        dset = {q: list(ds[reqs[q][3]: reqs[q][3] + reqs[q][1]]) for q in writes}
        for a in writes:
            if len(set(dset[a])) < len(dset[a]):
                ok[a] = oracle.ERR_DUPLICATE_DST
            for b in writes:
                if a != b and set(dset[a]) & set(dset[b]):
                    ok[a] = oracle.ERR_DUPLICATE_DST
        dst, buf = dst0.copy(), buf0.copy()
        for q, (op, n, so, do, bo) in enumerate(reqs):
            if ok[q] != oracle.OK:
                continue
            if op == oracle.OP_TRANSFER:
                dst = bf.transfer(src, ss[so:so + n], dst, ds[do:do + n])
            elif op == oracle.OP_GATHER:
                buf[bo: bo + P * n * R] = _bytes_of(bf.gather(src, ss[so:so + n]))
            else:
                rows = buf[bo: bo + P * n * R].view(np.uint16).reshape(L, 2, n, H, D)
                dst = bf.scatter(dst, ds[do:do + n], rows)
        return [max(ok + [0])] + ok, dst, buf

    def check(src, dst0, reqs, ss, ds, buf0):
        dst, buf = dst0.copy(), buf0.copy()
        st = oracle.batch(bf.to_oracle(src), bf.to_oracle(dst), reqs, ss, ds, buf, check_dup=True,
                          lib=lib)
        want_st, want_dst, want_buf = model(src, dst0, reqs, ss, ds, buf0)
        assert list(st) == want_st, (list(st), want_st, reqs)
        assert np.array_equal(dst.data, want_dst.data)
        assert np.array_equal(buf, want_buf)
        return list(st)

    src = bf.make_pool("planes", L, H, D, 12, lambda n: g.integers(0, 0x7C00, n))
    dst0 = bf.make_pool("planes", L, H, D, 12, _sentinel_fill)
    buf0 = g.integers(0, 255, 4 * P * 3 * R, dtype=np.uint8)
    T, G, S = oracle.OP_TRANSFER, oracle.OP_GATHER, oracle.OP_SCATTER
    ss = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 99, 1, 2, 3], dtype=np.int32)
    ds = np.array([0, 1, 2, 2, 3, 4, 5, 6, 6, 7, 8, 9, 10, 11, 9], dtype=np.int32)
    reqs = [(T, 3, 0, 0, 0),       # dst 0 1 2: shares 2 with the next one
            (T, 3, 3, 3, 0),       # dst 2 3 4
            (T, 3, 6, 6, 0),       # dst 5 6 6: repeats a slot of its own
            (T, 3, 9, 9, 0),       # src 9 10 99 out of range; dst 7 8 9
            (S, 2, 0, 12, 0),      # dst 10 11
            (T, 1, 12, 14, 0),     # dst 9: shared only with the refused request, so it moves
            (G, 2, 13, 0, P * 2 * R)]
    st = check(src, dst0, reqs, ss, ds, buf0)
    D_, O_ = oracle.ERR_DUPLICATE_DST, oracle.ERR_OUT_OF_RANGE
    assert st == [D_, D_, D_, D_, O_, 0, 0, 0]
    # without the check every accepted request moves
    st = oracle.batch(bf.to_oracle(src), bf.to_oracle(dst0.copy()), reqs, ss, ds, buf0.copy(),
                      lib=lib)
    assert list(st) == [O_, 0, 0, 0, O_, 0, 0, 0]
    for trial in range(150):
        nreq = int(g.integers(1, 5))
        reqs, ss_l, ds_l, bo = [], [], [], 0
        for _ in range(nreq):
            op = int(g.choice([T, T, S, G]))
            n = int(g.integers(1, 4))
            reqs.append((op, n, len(ss_l), len(ds_l), bo))
            ss_l += list(g.integers(0, 13 if g.random() < 0.15 else 12, n))
            ds_l += list(g.integers(0, 12, n))
            bo += P * n * R
        buf0 = g.integers(0, 255, max(bo, 16), dtype=np.uint8)
        check(src, dst0, reqs, np.array(ss_l, np.int32), np.array(ds_l, np.int32), buf0)


def _expand(runs):
    src, dst = [], []
    for _, s, d, n in runs:
        src.extend(range(s, s + n))
        dst.extend(range(d, d + n))
    return src, dst


def _coarsest_segmentation(src, dst, reqs):
    """Brute force: among every way of cutting tokens 0..n-1 into consecutive pieces, keep the
    cuttings whose pieces lie in one request and step up by one on both lists, and return the
    one with the fewest pieces (as (req, src, dst, len) tuples).  [Mooncake] 7.6 merges every
    block that follows the previous one, so the plan is the coarsest such cutting."""
    n = len(src)
    req_of = [max(q for q, r in enumerate(reqs) if r <= i) for i in range(n)]
    best = None
    for mask in range(1 << (n - 1)):
        cuts = [0] + [i for i in range(1, n) if mask >> (i - 1) & 1] + [n]
        pieces = []
        ok = True
        for a, b in zip(cuts[:-1], cuts[1:]):
            for i in range(a + 1, b):
                if (src[i] != src[a] + (i - a) or dst[i] != dst[a] + (i - a)
                        or req_of[i] != req_of[a]):
                    ok = False
            pieces.append((req_of[a], src[a], dst[a], b - a))
        if ok and (best is None or len(pieces) < len(best)):
            best = pieces
    return best


def pin_plan(lib):
    """[Mooncake] 7.6 coalescing, by brute force: for every pair of index lists of up to three
    tokens over four values and every request split, the oracle's runs are the coarsest
    cutting of the tokens into pieces that stay in one request and step up by one on both
    lists (found by trying every cutting); the same on random four- and five-token cases and
    on lists holding INT32_MAX next to INT32_MIN.
    Invariants on long lists: the runs expand back to the index lists, the run count is
    1 + the number of places where either list stops stepping by one or a request starts, and
    a contiguous request of any length is a single run (nothing else, such as a tile or a page
    boundary, ends a run)."""
    import itertools
    for n in (1, 2, 3):
        lists = list(itertools.product(range(4), repeat=n))
        splits = [[0] + list(c) for k in range(n) for c in itertools.combinations(range(1, n), k)]
        for src in lists:
            for dst in lists:
                for reqs in splits:
                    got = oracle.runs(src, dst, reqs, lib=lib)
                    want = _coarsest_segmentation(src, dst, reqs)
                    assert [tuple(r) for r in got.tolist()] == want, (src, dst, reqs)
    g = np.random.Generator(np.random.PCG64(23))
    for trial in range(400):
        n = int(g.integers(4, 6))
        base = g.integers(0, 3, 2)
        src = (base[0] + np.cumsum(g.choice([0, 1, 1, 1, 2], n))).tolist()
        dst = (base[1] + np.cumsum(g.choice([0, 1, 1, 1, -1], n))).tolist()
        reqs = [0] + sorted(set(g.integers(1, n, int(g.integers(0, 3))).tolist()))
        got = oracle.runs(src, dst, reqs, lib=lib)
        assert [tuple(r) for r in got.tolist()] == _coarsest_segmentation(src, dst, reqs)
    # the extremes of int32: INT32_MAX followed by INT32_MIN does not step up by one (a step
    # test in wrapping 32-bit arithmetic would merge them)
    big, small = 2 ** 31 - 1, -2 ** 31
    for src, dst in (([big - 1, big, small], [0, 1, 2]), ([0, 1, 2], [big - 1, big, small]),
                     ([big, small, small + 1], [big, small, small + 1])):
        got = oracle.runs(src, dst, [0], lib=lib)
        assert [tuple(r) for r in got.tolist()] == _coarsest_segmentation(src, dst, [0])
    # a contiguous request is one run whatever its length (72 blocks on a fresh pool,
    # "穷人版 PD 分离", 5090 section: one block per layer and K/V)
    for n in (1, 2047, 2048, 2049, 100000):
        got = oracle.runs(np.arange(7, 7 + n), np.arange(n), [0], lib=lib)
        assert got.tolist() == [[0, 7, 0, n]]
    # long random lists with several requests
    for trial in range(40):
        n = int(g.integers(1, 3000))
        def runs_of(hi):  # an independent run structure for each list
            r = []
            while sum(r) < n:
                r.append(int(g.integers(1, hi)))
            return np.concatenate([np.arange(s, s + k) for s, k in
                                   zip(g.integers(0, 1000, len(r)), r)])[:n]
        src = runs_of(6) if trial % 3 else np.arange(40, 40 + n)
        dst = runs_of(9) if trial % 3 != 1 else np.arange(n)
        reqs = sorted(set([0] + list(g.integers(0, n, int(g.integers(0, 5))))))
        got = oracle.runs(src, dst, reqs, lib=lib)
        s2, d2 = _expand(got)
        assert s2 == src.tolist() and d2 == dst.tolist()
        assert (got[:, 3] >= 1).all()
        brk = np.zeros(n, bool)
        brk[0] = True
        brk[1:] |= (src[1:] != src[:-1] + 1) | (dst[1:] != dst[:-1] + 1)
        brk[reqs] = True
        assert len(got) == 1 + int(brk[1:].sum())
        starts = np.concatenate([[0], np.cumsum(got[:, 3])[:-1]])
        for (q, _, _, _), t0 in zip(got, starts):
            assert q == max(i for i, r in enumerate(reqs) if r <= t0)


ALL_PINS = [pin_sizes, pin_bytes_written, pin_bruteforce_gather, pin_bruteforce_scatter,
            pin_bruteforce_transfer, pin_bruteforce_transfer_layers, pin_bruteforce_transfer_owned,
            pin_bruteforce_move_heads, pin_bruteforce_reshard, pin_reshard_reassembles_model,
            pin_move_heads_full_range_is_transfer, pin_tp_slice, pin_mla, pin_bruteforce_hnd,
            pin_roundtrip,
            pin_transfer_is_scatter_of_gather, pin_hnd_roundtrip, pin_plane_locality,
            pin_numpy_special_cases, pin_validation, pin_batch, pin_batch_duplicates, pin_plan]
