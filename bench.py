#!/usr/bin/env python
"""Benchmark of libkvx on its headline workload.

Workload (a step = one pass of the whole hot path: index validation + run-length plan + copy):
a 2048-token prompt, 36 layers x K/V x 8 kv heads x head_dim 128 bf16 (144 KiB/token, 288 MiB),
moved pool-to-pool between two 65,536-slot token pools (72 per-plane tensors each, 9 GiB per
pool) in one GB300's HBM; source and destination slot lists are 2048 distinct uniformly random
slots each.  Inputs are resident in HBM before the timed region; L2 is flushed before every
timed step, outside the step's CUDA events: a write of 2x the L2 size, then a read of another
2x L2 buffer so that the flush's own dirty lines are written back before the step (the line
also reports the step after a write-only flush, and back to back without any flush).

Metric: GB/s moved = (payload read + payload written + index bytes) / device time per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

At N = 1 the line also summarises, each with its own clock record, the other workloads
(`config.workloads`: small gather + scatter-back, fragmented pools, a 64-request batch, the HND
permute and rebuild) and the streamed move, the TP reshards and the other formats
(`config.next_rows`); --workload NAME prints any one of them alone.

--impl reference times the CPU oracle (single-threaded, as it stands) on a bounded sample of
the same workload on the host cores.  Under torchrun (N > 1) every rank runs an independent
replica on its own GPU (no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV transfer GB/s (read+write) & µs/request at 288 MiB; % of GB300 HBM peak"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("2048-token prompt, 36 layers x K/V x 8 kv heads x 128 bf16 (144 KiB/token, "
            "288 MiB), pool-to-pool transfer between two 65536-slot per-plane token pools, "
            "2048 + 2048 distinct uniformly random slots")
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

L, H, D, SLOTS, N_TOK = 36, 8, 128, 65536, 2048
R = H * D * 2
P = 2 * L


def alg_bytes(n_tokens: int) -> int:
    """Payload read + payload written + the two int32 slot lists."""
    return 2 * n_tokens * P * R + 2 * 4 * n_tokens


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="headline line only: skip the other four workloads' summaries")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the summaries of the streamed, TP-reshard and format workloads")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--pool-slots", type=int, default=SLOTS,
                    help="slots per plane of both pools (smaller pools for profiler captures; "
                         "the request itself is unchanged)")
    ap.add_argument("--workload-slots", type=int, default=None,
                    help="--workload fragmented|batch|hnd_permute: slots per plane of its pools "
                         "(smaller pools for profiler captures; the request is unchanged)")
    ap.add_argument("--batch-requests", type=int, default=None,
                    help="--workload batch: only the first N of its 64 requests (profiler "
                         "captures)")
    ap.add_argument("--fused-max", type=int, default=None,
                    help="kvx_set_fused_max_tokens for this run (0: planner + copy launches only)")
    ap.add_argument("--workload", default="transfer",
                    help="transfer (default): the 2048-token, 288 MiB pool-to-pool transfer; "
                         "small_gather_scatter, fragmented, batch, hnd_permute: the other "
                         "workloads of tests/inputs.py; "
                         "stream: the headline transfer through kvx_stream (layer-streamed); "
                         "tp: the headline request resharded between TP groups (kvx_reshard, and "
                         "kvx_move_heads pair by pair); "
                         "formats: MLA, fp8, narrow rows and cross-kind transcoding; "
                         "comparators: other ways to move the headline bytes (context); "
                         "sizes: the transfer time against the request size (T_setup + B/BW)")
    ap.add_argument("--check-duplicates", action="store_true",
                    help="kvx_set_check_duplicates(1) for this run (the planner also checks "
                         "every destination slot for repeats)")
    ap.add_argument("--layer-us", type=float, default=100.0,
                    help="--workload stream: host cadence of the emulated producer, us/layer")
    ap.add_argument("--device-only", action="store_true",
                    help="--workload stream: only the device-timed parts (no host-raised "
                         "layers, no cancellation trials), e.g. for a profiler")
    return ap.parse_args()


# ---------------------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


COPY_SOURCES = ("kvx_copy.cu", "kvx_copy_ops.cuh", "kvx_internal.cuh")


def copy_source_sha256() -> str:
    """Hash of the sources the copy kernel is compiled from."""
    h = hashlib.sha256()
    for name in COPY_SOURCES:
        with open(os.path.join(ROOT, "disaggregated_paged_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic():
    """Per-launch DRAM bytes of the copy kernel from the committed ncu summary, if that summary
    was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "copy_row_kernel_transfer_2048_tokens.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h or copy_source_sha256() != h.group(1):
        return None
    return int(m.group(1))


class Clocks:
    def __init__(self, device_index: int, enabled: bool):
        self.proc = None
        self.lines = []
        if not enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


class L2Flush:
    """What runs on the stream between two timed steps so that no step finds the previous one's
    data in L2: a write of a buffer of 2x the L2 size (every line the previous step left is
    evicted), then a read of another 2x L2 buffer, so that the lines the write left dirty are
    written back here, outside the timed region, instead of inside the next step.  `write_only`
    keeps just the write (its dirty lines are then written back during the next step)."""

    def __init__(self, dev, l2_bytes: int, write_only: bool = False):
        import torch

        n = max(2 * l2_bytes, 256 << 20)
        self.w = torch.empty(n, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(n // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty(1, dtype=torch.int64, device=dev)
        self.write_only = write_only

    def fill_(self, v: int):
        import torch

        self.w.fill_(v)
        if not self.write_only:
            torch.sum(self.r, dim=0, keepdim=True, out=self.sink)


L2_NOTE = ("flushed before every timed step, outside the events: a write of 2x L2 (evicts the "
           "previous step's lines) then a read of another 2x L2 (writes the flush's dirty lines "
           "back before the step starts)")


def step_percentiles(step_ms):
    """p10, median and p90 of per-step times, in us (CUDA event timestamps tick in ~1-2 us
    steps on this GPU, so these are coarse; the mean is the headline)."""
    xs = sorted(step_ms)
    n = len(xs)
    return [xs[n // 10] * 1e3, xs[n // 2] * 1e3, xs[(9 * n) // 10] * 1e3]


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over all ranks (x itself without an initialised process group)."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput: every rank moved bytes_per_step per step; the slowest rank's time
    counts."""
    return world * bytes_per_step * steps / (max_total_ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------

def run_ours(args, rank: int, world: int, local_rank: int):
    import numpy as np
    import torch

    from disaggregated_paged_kv_gb300 import kvx
    from tests import inputs

    torch.cuda.set_device(local_rank)
    NS = args.pool_slots
    dev = torch.device("cuda", local_rank)
    kvx.lib()
    stream = torch.cuda.Stream(device=dev)
    sptr = int(stream.cuda_stream)

    # inputs resident in HBM: two 9 GiB pools of 72 per-plane [65536][8][128] bf16 tensors
    gen = torch.Generator(device=dev)
    gen.manual_seed(inputs.seed(2, inputs.ROLE_VALUES) + rank)
    src = torch.randn((P, NS, H, D), dtype=torch.bfloat16, device=dev, generator=gen)
    dst = torch.empty((P, NS, H, D), dtype=torch.bfloat16, device=dev)
    dst.view(torch.int16).fill_(0x7FC1)  # quiet-NaN sentinel
    s_np = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N_TOK, NS)
    d_np = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N_TOK, NS)
    s_dev = torch.from_numpy(s_np).to(dev)
    d_dev = torch.from_numpy(d_np).to(dev)
    src_l = kvx.Layout(L, H, D, kvx.BF16, NS, base=src, plane_stride=NS * R)
    dst_l = kvx.Layout(L, H, D, kvx.BF16, NS, base=dst, plane_stride=NS * R)
    ws = torch.empty(kvx.workspace_size(N_TOK, 0), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)
    torch.cuda.synchronize()

    def step():
        kvx.transfer(src_l, s_dev, dst_l, d_dev, N_TOK, ws, st, stream=sptr)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            step()
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    # the kernel did the work: sampled rows equal on the device
    k = torch.from_numpy(np.arange(0, N_TOK, 97)).to(dev)
    assert torch.equal(dst[:, d_dev[k]].view(torch.int16), src[:, s_dev[k]].view(torch.int16))

    # ---- timed region: K steps, each bracketed by events on the launching stream ----
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local_rank, not args.no_clocks)
    time.sleep(0.3 if clocks.proc else 0)
    with torch.cuda.stream(stream):
        for _ in range(3):  # untimed: the GPU back at full clocks after the pause above
            flush.fill_(1)
            step()
        for i in range(K):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)

    # ---- steady state without the flush: inputs larger than L2 (288 MiB each way per step),
    # consecutive steps moving two different sets of random rows in turn, so that no step finds
    # its rows in L2 and no flush buffer's dirty lines are written back inside a step ----
    s2 = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, 100 + inputs.ROLE_SRC_SLOTS), N_TOK, NS)).to(dev)
    d2 = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, 100 + inputs.ROLE_DST_SLOTS), N_TOK, NS)).to(dev)
    sets = [(s_dev, d_dev), (s2, d2)]
    ev4 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K + 2):
            if i >= 2:
                ev4[i - 2][0].record(stream)
            ss, dd = sets[i & 1]
            kvx.transfer(src_l, ss, dst_l, dd, N_TOK, ws, st, stream=sptr)
            if i >= 2:
                ev4[i - 2][1].record(stream)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    noflush_ms = statistics.mean(a.elapsed_time(b) for a, b in ev4)

    # ---- the same step captured once into a CUDA graph and replayed (same flushes) ----
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    ev5 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K + 3):
            flush.fill_(i & 0xFF)
            if i >= 3:
                ev5[i - 3][0].record(stream)
            graph.replay()
            if i >= 3:
                ev5[i - 3][1].record(stream)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    graph_ms = statistics.mean(a.elapsed_time(b) for a, b in ev5)
    del graph

    # ---- the same step after a write-only flush: L2 then holds up to its size in the flush's
    # dirty lines, which the step itself has to write back ----
    wflush = L2Flush(dev, l2, write_only=True)
    ev6 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K + 3):
            wflush.fill_(i & 0xFF)
            if i >= 3:
                ev6[i - 3][0].record(stream)
            step()
            if i >= 3:
                ev6[i - 3][1].record(stream)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.OK
    write_only_ms = statistics.mean(a.elapsed_time(b) for a, b in ev6)
    del wflush

    # ---- the copy kernel alone (plan and copy launched separately, same flushes) ----
    ev3 = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K):
            flush.fill_(i & 0xFF)
            ev3[i][0].record(stream)
            kvx.plan(kvx.OP_TRANSFER, src_l, s_dev, dst_l, d_dev, N_TOK, ws, st, stream=sptr)
            ev3[i][1].record(stream)
            kvx.execute(kvx.OP_TRANSFER, src_l, dst_l, None, 0, N_TOK, None, ws, st,
                        buf_bytes=0, stream=sptr)
            ev3[i][2].record(stream)
    torch.cuda.synchronize()
    plan_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in ev3)
    copy_ms = statistics.mean(b.elapsed_time(c) for _, b, c in ev3)

    # ---- the ceiling: the same payload as one contiguous device-to-device copy, same flushes ----
    ca = src.view(-1).view(torch.uint8)[: N_TOK * P * R]
    cb = dst.view(-1).view(torch.uint8)[: N_TOK * P * R]
    ev7 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K + 3):
            flush.fill_(i & 0xFF)
            if i >= 3:
                ev7[i - 3][0].record(stream)
            cb.copy_(ca)
            if i >= 3:
                ev7[i - 3][1].record(stream)
    torch.cuda.synchronize()
    contiguous_ms = statistics.mean(a.elapsed_time(b) for a, b in ev7)
    dst.view(torch.int16).fill_(0x7FC1)

    # ---- end to end through the C ABI with host buffers (kvx_submit) ----
    e2e = None
    if not args.no_e2e:
        hs = torch.from_numpy(s_np).pin_memory()
        hd = torch.from_numpy(d_np).pin_memory()
        hst = torch.full((1,), -1, dtype=torch.int32).pin_memory()
        ws2 = torch.empty(kvx.workspace_size(N_TOK, 0), dtype=torch.uint8, device=dev)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        with torch.cuda.stream(stream):
            for _ in range(3):  # untimed: the first calls look up the pinned buffers' mappings
                flush.fill_(1)
                kvx.submit(kvx.OP_TRANSFER, src_l, hs, dst_l, hd, N_TOK, None, ws2, hst,
                           buf_bytes=0, stream=sptr)
            for i in range(K):
                flush.fill_(i & 0xFF)
                ev2[i][0].record(stream)
                kvx.submit(kvx.OP_TRANSFER, src_l, hs, dst_l, hd, N_TOK, None, ws2, hst,
                           buf_bytes=0, stream=sptr)
                ev2[i][1].record(stream)
        torch.cuda.synchronize()
        assert int(hst[0]) == kvx.OK
        e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in ev2)
        e2e = {"value": alg_bytes(N_TOK) / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
               "us_per_request": e2e_ms * 1e3,
               "h2d_bytes_per_step": 2 * 4 * N_TOK, "d2h_bytes_per_step": 4,
               "how": "kvx_submit with pinned host slot lists and status word: the planner "
                      "and the copy read the 16 KiB of slot lists from host memory over "
                      "NVLink-C2C and the copy writes the 4-byte status back, all inside the "
                      "step's CUDA events"}

    total_ms = max_over_ranks(total_ms, device=dev)
    return dict(step_ms=step_ms, total_ms=total_ms, plan_ms=plan_ms, copy_ms=copy_ms, e2e=e2e,
                clocks=clk, device=torch.cuda.get_device_name(dev), noflush_ms=noflush_ms,
                graph_ms=graph_ms, write_only_ms=write_only_ms, contiguous_ms=contiguous_ms)


# ---------------------------------------------------------------------------------------
# the other workloads (--workload small_gather_scatter, fragmented, batch, hnd_permute): same
# timing rules, one JSON line each
# ---------------------------------------------------------------------------------------

def run_workload(args, name: str):
    print(json.dumps(measure_workload(args, name)), flush=True)


def measure_workload(args, name: str, min_seconds: float = 0.25):
    """Times every leg of the named workload (gather + scatter-back, fragmented gather +
    scatter, batch, fused-permute gather + rebuild) and returns its JSON line.  Pools, slot
    lists and page tables come from the same seeded recipe as the tests.  The timed steps are
    repeated until they span at least min_seconds, with the SM clocks sampled meanwhile."""
    import numpy as np
    import torch

    from disaggregated_paged_kv_gb300 import kvx
    from tests import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvx.lib()
    stream = torch.cuda.Stream(device=dev)
    sp = int(stream.cuda_stream)
    w = inputs.WORKLOADS[name]
    if args.workload_slots and name in ("fragmented", "batch", "hnd_permute"):
        w = dataclasses.replace(w, num_slots=args.workload_slots)
    sid = w.seed_id
    Pw, Hw, Dw, Rw = w.planes, w.kv_heads, w.head_dim, w.row_bytes
    tdt = torch.float16 if w.dtype == "fp16" else torch.bfloat16
    kdt = kvx.F16 if w.dtype == "fp16" else kvx.BF16
    gen = torch.Generator(device=dev)
    gen.manual_seed(inputs.seed(sid, inputs.ROLE_VALUES))
    sentinel = 0x7E01 if w.dtype == "fp16" else 0x7FC1

    def randn(shape):
        return torch.randn(shape, dtype=tdt, device=dev, generator=gen)

    def sentinel_pool(shape):
        t = torch.empty(shape, dtype=tdt, device=dev)
        t.view(torch.int16).fill_(sentinel)
        return t

    st = torch.zeros(65, dtype=torch.int32, device=dev)
    legs = []  # (name, fn, algorithmic bytes)
    requests = 1
    if name == "small_gather_scatter":
        pool = randn((w.num_slots, w.num_layers, 2, Hw, Dw))
        lay = kvx.Layout(w.num_layers, Hw, Dw, kdt, w.num_slots, base=pool, plane_stride=Rw,
                         slot_stride=Pw * Rw)
        slots = torch.from_numpy(inputs.distinct_slots(inputs.rng(sid, 1), w.n_tokens, w.num_slots)).to(dev)
        buf = torch.empty((Pw, w.n_tokens, Hw, Dw), dtype=tdt, device=dev)
        ws = torch.empty(kvx.workspace_size(w.n_tokens), dtype=torch.uint8, device=dev)
        nb = 2 * w.payload_bytes + 4 * w.n_tokens
        legs = [("gather", lambda: kvx.gather(lay, slots, w.n_tokens, buf, ws, st, stream=sp), nb),
                ("scatter_back_in_place",
                 lambda: kvx.scatter(lay, slots, w.n_tokens, buf, ws, st, stream=sp), nb)]
        desc = ("Qwen2.5-1.5B-shaped KV (28 x K/V x 2 x 128 fp16), slot-major pool of 4096 slots, "
                "128 random slots: gather to a 3.5 MiB [layer][K/V][seq][head][dim] buffer, then "
                "scatter back in place")
    elif name == "fragmented":
        src_planes = [randn((w.num_slots, Hw, Dw)) for _ in range(Pw)]
        dst_planes = [sentinel_pool((w.num_slots, Hw, Dw)) for _ in range(Pw)]
        s_np, runs = inputs.fragmented_slots(inputs.rng(sid, 1), w.n_tokens, w.num_slots, 1.6)
        d_np, _ = inputs.fragmented_slots(inputs.rng(sid, 2), w.n_tokens, w.num_slots, 1.6)
        s_d, d_d = torch.from_numpy(s_np).to(dev), torch.from_numpy(d_np).to(dev)
        sl = kvx.Layout(w.num_layers, Hw, Dw, kdt, w.num_slots, plane_ptrs=src_planes)
        dl = kvx.Layout(w.num_layers, Hw, Dw, kdt, w.num_slots, plane_ptrs=dst_planes)
        buf = torch.empty((Pw, w.n_tokens, Hw, Dw), dtype=tdt, device=dev)
        ws = torch.empty(kvx.workspace_size(w.n_tokens), dtype=torch.uint8, device=dev)
        nb = 2 * w.payload_bytes + 4 * w.n_tokens
        legs = [("gather", lambda: kvx.gather(sl, s_d, w.n_tokens, buf, ws, st, stream=sp), nb),
                ("scatter", lambda: kvx.scatter(dl, d_d, w.n_tokens, buf, ws, st, stream=sp), nb)]
        desc = (f"fragmented pools: 72 per-plane [131072][8][128] bf16 pools, 1536 tokens in "
                f"{len(runs)} runs ~Geometric(1.6): gather to a 216 MiB buffer, then scatter into a "
                f"fresh run layout")
    elif name == "batch":
        lens = inputs.batch_lengths()[: args.batch_requests or None]
        s_np, offs = inputs.paged_request_slots(inputs.rng(sid, 1), lens, w.page_size, w.num_slots)
        d_np, _ = inputs.paged_request_slots(inputs.rng(sid, 2), lens, w.page_size, w.num_slots)
        src = randn((Pw, w.num_slots, Hw, Dw))
        dst = sentinel_pool((Pw, w.num_slots, Hw, Dw))
        sl = kvx.Layout(w.num_layers, Hw, Dw, kdt, w.num_slots, base=src, plane_stride=w.num_slots * Rw)
        dl = kvx.Layout(w.num_layers, Hw, Dw, kdt, w.num_slots, base=dst, plane_stride=w.num_slots * Rw)
        reqs = [kvx.Request(kvx.OP_TRANSFER, L, int(o), int(o), 0) for L, o in zip(lens, offs[:-1])]
        dreq = torch.from_numpy(np.frombuffer(b"".join(bytes(r) for r in reqs), dtype=np.uint8).copy()).to(dev)
        total = int(sum(lens))
        s_d, d_d = torch.from_numpy(s_np).to(dev), torch.from_numpy(d_np).to(dev)
        ws = torch.empty(kvx.workspace_size(total, len(reqs)), dtype=torch.uint8, device=dev)
        nb = 2 * total * Pw * Rw + 8 * total + 32 * len(reqs)
        requests = len(reqs)
        legs = [("batch", lambda: kvx.batch(sl, dl, dreq, len(reqs), total, s_d, total, d_d, total,
                                             None, ws, st, buf_bytes=0, stream=sp), nb)]
        desc = (f"64 requests of U{{1000..2000}} tokens ({total} total), 36 x K/V x 8 x 128 bf16, "
                f"token-paged pools of 262144 slots with page size 16: one kvx_batch")
    elif name == "hnd_permute":
        ps = w.page_size
        pages = w.num_slots // ps
        n_pages = w.n_tokens // ps
        src = randn((Pw, pages, Hw, ps, Dw))
        dst = sentinel_pool((Pw, pages, Hw, ps, Dw))
        pt = inputs.random_pages(inputs.rng(sid, 1), n_pages, pages)
        pt2 = inputs.random_pages(inputs.rng(sid, 2), n_pages, pages)
        s_d = torch.from_numpy(inputs.page_table_slots(pt, w.n_tokens, ps)).to(dev)
        d_d = torch.from_numpy(inputs.page_table_slots(pt2, w.n_tokens, ps)).to(dev)
        sl = kvx.Layout(w.num_layers, Hw, Dw, kdt, w.num_slots, kind=kvx.HND_PAGED, page_size=ps,
                        base=src, plane_stride=w.num_slots * Rw)
        dl = kvx.Layout(w.num_layers, Hw, Dw, kdt, w.num_slots, kind=kvx.HND_PAGED, page_size=ps,
                        base=dst, plane_stride=w.num_slots * Rw)
        buf = torch.empty((Pw, w.n_tokens, Hw, Dw), dtype=tdt, device=dev)
        ws = torch.empty(kvx.workspace_size(w.n_tokens), dtype=torch.uint8, device=dev)
        nb = 2 * w.payload_bytes + 4 * w.n_tokens
        legs = [("gather_permute", lambda: kvx.gather(sl, s_d, w.n_tokens, buf, ws, st, stream=sp), nb),
                ("rebuild", lambda: kvx.scatter(dl, d_d, w.n_tokens, buf, ws, st, stream=sp), nb)]
        desc = ("Qwen2.5-7B-shaped KV (28 x K/V x 4 x 128 bf16), seq 32768 in HND pages of 16 "
                "(65536-page pools, random page tables): fused [heads,seq,dim] -> [seq,heads,dim] "
                "gather to a 1.75 GiB buffer, then the inverse rebuild")
    else:
        raise SystemExit(f"unknown workload {name}")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)

    def timed(K, flush_l2=True, legs=legs):
        evs = []
        with torch.cuda.stream(stream):
            for i in range(K):
                e = [torch.cuda.Event(enable_timing=True) for _ in range(len(legs) + 1)]
                if flush_l2:
                    flush.fill_(i & 0xFF)
                e[0].record(stream)
                for j, (_, fn, _) in enumerate(legs):
                    fn()
                    e[j + 1].record(stream)
                evs.append(e)
        torch.cuda.synchronize()
        return [[e[j].elapsed_time(e[j + 1]) for j in range(len(legs))] for e in evs]

    timed(max(3, args.warmup))
    assert int(st[0].item()) == kvx.OK, int(st[0].item())
    K = max(3, min(args.steps, 200 if name in ("batch", "hnd_permute") else args.steps))
    clocks = Clocks(0, not args.no_clocks)
    time.sleep(0.2 if clocks.proc else 0)
    timed(3)  # untimed: the GPU back at full clocks after the pause above
    res = []
    t_start = time.perf_counter()
    while not res or (time.perf_counter() - t_start < min_seconds and len(res) < 50 * K):
        res += timed(K)
    clk = clocks.stop()
    K = len(res)
    total_bytes = sum(b for _, _, b in legs)
    step_ms = statistics.mean(sum(r) for r in res)
    line = {"metric": METRIC, "value": total_bytes / (step_ms * 1e-3) / 1e9, "unit": UNIT,
            "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "dtype": "u8", "data": "synthetic",
            "config": {"workload": f"{name}: {desc}", "kv_dtype": w.dtype,
                       "alg_bytes_per_step": total_bytes, "requests_per_step": requests,
                       "us_per_request": step_ms * 1e3 / requests,
                       "l2": L2_NOTE},
            "legs": {name: {"us": statistics.mean(r[j] for r in res) * 1e3,
                            "GBs": b / (statistics.mean(r[j] for r in res) * 1e-3) / 1e9}
                     for j, (name, _, b) in enumerate(legs)},
            "clocks": clk}
    peaks, _ = measured_peaks()
    line["config"]["frac_of_measured_hbm"] = line["value"] / float(peaks["hbm_gbs"])
    line["config"]["frac_of_nominal_8tbs"] = line["value"] / NOMINAL_HBM_GBS
    # the floor of one leg: the same payload as one contiguous device-to-device copy, timed the
    # same way (flush outside the events)
    payload = total_bytes // (2 * len(legs))
    ca = torch.empty(payload, dtype=torch.uint8, device=dev)
    cb = torch.empty_like(ca)
    copy_leg = [("contiguous_copy", lambda: cb.copy_(ca), 2 * payload)]
    timed(3, legs=copy_leg)
    cres = timed(max(3, min(K, 200)), legs=copy_leg)
    line["contiguous_copy_us_per_leg"] = statistics.mean(r[0] for r in cres) * 1e3
    del ca, cb
    if name == "small_gather_scatter":
        # a launch-bound leg's floors under the same timing: an elementwise kernel reading and
        # writing the leg's bytes (the device copy above goes through the copy engine, whose
        # setup alone is longer here), and a kernel that touches one element
        ka = torch.zeros(payload // 2, dtype=torch.float16, device=dev)
        kb = torch.empty_like(ka)
        one = torch.zeros(1, dtype=torch.float32, device=dev)
        floors = {}
        for fname, fn in (("kernel_copy", lambda: torch.add(ka, 0, out=kb)),
                          ("one_element_kernel", lambda: one.add_(1))):
            leg = [(fname, fn, 0)]
            timed(3, legs=leg)
            floors[fname + "_us"] = statistics.mean(r[0] for r in timed(max(3, min(K, 200)), legs=leg)) * 1e3
        floors["how"] = ("event-to-event time of one torch kernel per step after the same flush: "
                         "an elementwise copy of one leg's bytes, and a one-element add")
        line["launch_floor_per_leg"] = floors
        del ka, kb, one
    if name == "fragmented":
        # the same request on the first 4 layers only (8 planes): ~7,700 fragments per direction
        L4 = 4
        sl4 = kvx.Layout(L4, Hw, Dw, kdt, w.num_slots, plane_ptrs=src_planes[:2 * L4])
        dl4 = kvx.Layout(L4, Hw, Dw, kdt, w.num_slots, plane_ptrs=dst_planes[:2 * L4])
        buf4 = buf[:2 * L4]
        nb4 = 2 * 2 * L4 * w.n_tokens * Rw + 4 * w.n_tokens
        legs4 = [("gather", lambda: kvx.gather(sl4, s_d, w.n_tokens, buf4, ws, st, stream=sp), nb4),
                 ("scatter", lambda: kvx.scatter(dl4, d_d, w.n_tokens, buf4, ws, st, stream=sp), nb4)]
        timed(3, legs=legs4)
        assert int(st[0].item()) == kvx.OK, int(st[0].item())
        r4 = timed(K, legs=legs4)
        ms4 = statistics.mean(sum(r) for r in r4)
        line["four_layers"] = {
            "planes": 2 * L4, "fragments_per_direction": 2 * L4 * len(runs),
            "us_per_step": ms4 * 1e3, "GBs": 2 * nb4 / (ms4 * 1e-3) / 1e9,
            "frac_of_measured_hbm": 2 * nb4 / (ms4 * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
            "legs_us": [statistics.mean(r[j] for r in r4) * 1e3 for j in range(2)],
            "how": "the same 1536-token request on 4 layers (8 planes), gather then scatter"}
    if name == "small_gather_scatter":  # launch-bound, L2-resident unless flushed: warm too
        warm = timed(K, flush_l2=False)
        wm = statistics.mean(sum(r) for r in warm)
        line["warm_l2"] = {"value": total_bytes / (wm * 1e-3) / 1e9, "us_per_step": wm * 1e3}
        # both legs captured once into a CUDA graph and replayed each step (same flushes)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for _, fn, _ in legs:
                    fn()
        torch.cuda.synchronize()

        def replayed(K, flush_l2):
            evs = []
            with torch.cuda.stream(stream):
                for i in range(K):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    if flush_l2:
                        flush.fill_(i & 0xFF)
                    e0.record(stream)
                    graph.replay()
                    e1.record(stream)
                    evs.append((e0, e1))
            torch.cuda.synchronize()
            return statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3

        replayed(3, True)
        assert int(st[0].item()) == kvx.OK
        gf, gw = replayed(K, True), replayed(K, False)
        line["cuda_graph"] = {"us_per_step": gf, "value": total_bytes / (gf * 1e-6) / 1e9,
                              "warm_l2_us_per_step": gw,
                              "warm_l2_value": total_bytes / (gw * 1e-6) / 1e9,
                              "how": "both legs captured once (one launch each: requests of up to 512 "
                                     "tokens skip the planner), replayed"}
    return line


OTHER_WORKLOADS = ("small_gather_scatter", "fragmented", "batch", "hnd_permute")


def workload_summaries(args):
    """The other four workloads, each timed as by --workload NAME, summarised for the headline
    line (their pools are allocated and freed one workload at a time)."""
    import torch

    out = {}
    for name in OTHER_WORKLOADS:
        torch.cuda.empty_cache()
        ln = measure_workload(args, name)
        cfg = ln["config"]
        out[name] = {"workload": cfg["workload"], "GBs": ln["value"],
                     "us_per_request": cfg["us_per_request"],
                     "us_per_step": ln["ms_per_step"] * 1e3,
                     "requests_per_step": cfg["requests_per_step"],
                     "alg_bytes_per_step": cfg["alg_bytes_per_step"],
                     "frac_of_measured_hbm": cfg["frac_of_measured_hbm"],
                     "frac_of_nominal_8tbs": cfg["frac_of_nominal_8tbs"],
                     "legs": ln["legs"], "steps": ln["steps"], "clocks": ln["clocks"],
                     "contiguous_copy_us_per_leg": ln["contiguous_copy_us_per_leg"]}
        for extra in ("four_layers", "warm_l2", "cuda_graph", "launch_floor_per_leg"):
            if extra in ln:
                out[name][extra] = ln[extra]
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------------------
# the oracle (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------------------

class OracleTransfer:
    """The single-threaded oracle on a transfer of n_tokens rows x 72 planes between two host
    pools of pool_slots slots per plane (both first-touched before any timing)."""

    def __init__(self, n_tokens: int, pool_slots: int):
        import numpy as np

        import oracle
        from tests import inputs

        g = inputs.rng(2, inputs.ROLE_VALUES)
        nbytes = P * pool_slots * R
        # the source pool: a seeded 1 MiB block of random bytes repeated (the copy never looks at
        # the values; every page is touched here, before any timing)
        block = 1 << 20
        self.src = np.empty(nbytes, dtype=np.uint8)
        self.src.reshape(-1, block)[:] = g.integers(0, 256, block, dtype=np.uint8)
        self.dst = np.zeros(nbytes, dtype=np.uint8)
        self.sp = oracle.Pool(L, H, D, 2, oracle.TOKEN_ROWS, pool_slots,
                              [(self.src, p * pool_slots * R) for p in range(P)], R)
        self.dp = oracle.Pool(L, H, D, 2, oracle.TOKEN_ROWS, pool_slots,
                              [(self.dst, p * pool_slots * R) for p in range(P)], R)
        self.s = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), n_tokens, pool_slots)
        self.d = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), n_tokens, pool_slots)
        self.lib = oracle.load()
        self.oracle = oracle
        self.pool_slots = pool_slots

    def run_all_cores(self, budget_s: float = 3.0):
        """The same transfer split by layers over every host core (one thread per layer range,
        the C oracle releasing the GIL), repeated for about budget_s.  Returns (seconds per
        transfer, threads).  Not the oracle as it stands: a labelled CPU line beside it."""
        import threading

        threads = max(1, min(os.cpu_count() or 1, L))
        bounds = [L * t // threads for t in range(threads + 1)]
        parts = []
        for t in range(threads):
            l0, l1 = bounds[t], bounds[t + 1]
            planes = slice(2 * l0, 2 * l1)
            sp = self.oracle.Pool(l1 - l0, H, D, 2, self.oracle.TOKEN_ROWS, self.pool_slots,
                                  self.sp.planes[planes], R)
            dp = self.oracle.Pool(l1 - l0, H, D, 2, self.oracle.TOKEN_ROWS, self.pool_slots,
                                  self.dp.planes[planes], R)
            parts.append((sp, dp))
        reps = [0]
        stop = time.perf_counter() + budget_s

        def work(sp, dp, out):
            n = 0
            while n < 1 or time.perf_counter() < stop:
                rc, _ = self.oracle.transfer(sp, self.s, dp, self.d, lib=self.lib)
                assert rc == self.oracle.OK
                n += 1
            out.append(n)

        counts = []
        t0 = time.perf_counter()
        ths = [threading.Thread(target=work, args=(sp, dp, counts)) for sp, dp in parts]
        for th in ths:
            th.start()
        for th in ths:
            th.join()
        wall = time.perf_counter() - t0
        return wall / min(counts), threads

    def run(self, reps: int = 0, budget_s: float = 0.0, min_reps: int = 1):
        """Runs reps transfers (or, with reps=0, at least min_reps and until budget_s).
        Returns (seconds per transfer, transfers run)."""
        n, t0 = 0, time.perf_counter()
        while (n < reps) if reps else (n < min_reps or time.perf_counter() - t0 < budget_s):
            rc, _ = self.oracle.transfer(self.sp, self.s, self.dp, self.d, lib=self.lib)
            assert rc == self.oracle.OK
            n += 1
        return (time.perf_counter() - t0) / max(n, 1), n


def _cudart():
    """The CUDA runtime library of the toolkit, for plain cudaMemcpyAsync calls."""
    import ctypes
    import glob
    cands = (glob.glob("/usr/local/cuda/lib64/libcudart.so*") +
             glob.glob("/usr/local/cuda/targets/*/lib/libcudart.so*"))
    for c in sorted(cands):
        try:
            lib = ctypes.CDLL(c)
            lib.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                            ctypes.c_int, ctypes.c_void_p]
            lib.cudaMemcpyAsync.restype = ctypes.c_int
            return lib
        except OSError:
            continue
    return None


def run_comparators(args):
    """Other ways to move the headline request's bytes on the same GB300 (context, not shipped):
    a contiguous device-to-device copy of the same byte count (the streaming ceiling), one
    cudaMemcpyAsync per 2 KiB fragment (the per-block path of the pages' first design, 147,456
    copies), and torch index_select + index_copy_ over the [72][slots][8][128] pools.  L2 flushed
    before each step; CUDA events on the launching stream."""
    import torch

    from disaggregated_paged_kv_gb300 import kvx
    from tests import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    NS = args.pool_slots
    stream = torch.cuda.Stream(device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(inputs.seed(2, inputs.ROLE_VALUES))
    src = torch.randn((P, NS, H, D), dtype=torch.bfloat16, device=dev, generator=gen)
    dst = torch.empty((P, NS, H, D), dtype=torch.bfloat16, device=dev)
    s_np = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N_TOK, NS)
    d_np = inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N_TOK, NS)
    s_dev = torch.from_numpy(s_np).to(dev).long()
    d_dev = torch.from_numpy(d_np).to(dev).long()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)
    flat_src = src.view(-1)[: N_TOK * P * H * D]
    flat_dst = dst.view(-1)[: N_TOK * P * H * D]

    def timed(fn, K):
        with torch.cuda.stream(stream):
            for _ in range(2):
                flush.fill_(1)
                fn()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            for i in range(K):
                flush.fill_(i & 0xFF)
                ev[i][0].record(stream)
                fn()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3

    res = {}
    res["contiguous_d2d_copy_us"] = timed(lambda: flat_dst.copy_(flat_src), args.steps)

    def index_path():
        dst.index_copy_(1, d_dev, src.index_select(1, s_dev))

    res["torch_index_select_index_copy_us"] = timed(index_path, max(3, args.steps // 20))

    rt = _cudart()
    if rt is not None:
        sp = stream.cuda_stream
        base_s, base_d = src.data_ptr(), dst.data_ptr()
        offs = [(p * NS + int(si)) * R for p in range(P) for si in s_np]
        offd = [(p * NS + int(di)) * R for p in range(P) for di in d_np]
        pairs = list(zip(offs, offd))

        def per_fragment():
            for a, b in pairs:
                rt.cudaMemcpyAsync(base_d + b, base_s + a, R, 3, sp)  # device to device

        res["per_fragment_memcpy_us"] = timed(per_fragment, 2)
        res["per_fragment_copies"] = len(pairs)
    else:
        res["per_fragment_memcpy_us"] = None
    kvx.lib()
    nb = alg_bytes(N_TOK)
    line = {
        "metric": "other ways to move the headline request's 288 MiB on the same GPU (context)",
        "value": res["contiguous_d2d_copy_us"], "unit": "us", "n_gpus": 1, "steps": args.steps,
        "warmup": 2, "higher_is_better": False, "dtype": "u8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "value": "contiguous D2D copy of the same bytes, us",
                   "l2": L2_NOTE},
        "comparators": res,
        "GBs": {k: (nb / (v * 1e-6) / 1e9 if isinstance(v, float) and k.endswith("_us") else None)
                for k, v in res.items()},
    }
    print(json.dumps(line), flush=True)


def run_sizes(args):
    """The transfer-time model T = T_setup + B / BW_eff on this GPU: one-shot kvx_transfer of n
    random tokens x 72 planes for n = 256 .. 16384, with 2 KiB rows (36 x K/V x 8 x 128 bf16)
    and with 1 KiB rows (the same shape in fp8), between 65536-slot per-plane pools, beside a
    contiguous device-to-device copy (torch copy_) of the same byte count.  L2 flushed before
    every step; CUDA events on the launching stream.  The fit (least squares over n >= 1024)
    splits each path's time into a fixed cost per call and a bandwidth."""
    import numpy as np
    import torch

    from disaggregated_paged_kv_gb300 import kvx
    from tests import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvx.lib()
    stream = torch.cuda.Stream(device=dev)
    sp = int(stream.cuda_stream)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)
    peaks, _ = measured_peaks()
    NS, K = 65536, max(10, min(args.steps, 100))
    sizes = [256, 512, 1024, 2048, 4096, 8192, 16384]

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K + 3)]
        with torch.cuda.stream(stream):
            for i, (a, b) in enumerate(ev):
                flush.fill_(i & 0xFF)
                a.record(stream)
                fn()
                b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev[3:]) * 1e3  # us

    def fit(pts):
        x = np.array([b for b, _ in pts], dtype=np.float64)
        y = np.array([t for _, t in pts], dtype=np.float64)
        slope, icpt = np.polyfit(x, y, 1)
        return {"t_setup_us": icpt, "bw_eff_gbs": 1e-3 / slope,
                "bw_eff_frac_of_measured_hbm": 1e-3 / slope / float(peaks["hbm_gbs"])}

    shapes = {"bf16_2KiB_rows": (2, kvx.BF16), "fp8_1KiB_rows": (1, kvx.FP8)}
    results, copy_pts = {}, {}
    for label, (e, dt) in shapes.items():
        R = H * D * e
        src = torch.randint(0, 255, (P * NS * R,), dtype=torch.uint8, device=dev)
        dst = torch.zeros(P * NS * R, dtype=torch.uint8, device=dev)
        sl = kvx.Layout(L, H, D, dt, NS, base=src, plane_stride=NS * R)
        dl = kvx.Layout(L, H, D, dt, NS, base=dst, plane_stride=NS * R)
        rows, pts = [], []
        for n in sizes:
            s_d = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), n, NS)).to(dev)
            d_d = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), n, NS)).to(dev)
            ws = torch.empty(kvx.workspace_size(n, 0), dtype=torch.uint8, device=dev)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            us = timed(lambda: kvx.transfer(sl, s_d, dl, d_d, n, ws, st, stream=sp))
            assert int(st.item()) == kvx.OK
            alg = 2 * n * P * R + 8 * n
            row = {"tokens": n, "alg_bytes": alg, "us": us, "GBs": alg / (us * 1e-6) / 1e9}
            row["frac_of_measured_hbm"] = row["GBs"] / float(peaks["hbm_gbs"])
            if n * P * R not in copy_pts:
                nb = n * P * R
                a, b = src[:nb], dst[:nb]
                cu = timed(lambda: b.copy_(a))
                copy_pts[nb] = cu
            row["contiguous_copy_us"] = copy_pts[n * P * R]
            rows.append(row)
            if n >= 1024:
                pts.append((alg, us))
        results[label] = {"row_bytes": R, "points": rows, "fit": fit(pts)}
        del src, dst, sl, dl
        torch.cuda.empty_cache()
    cfit = fit([(2 * nb, t) for nb, t in copy_pts.items() if nb >= 1024 * P * H * D])
    head = next(r for r in results["bf16_2KiB_rows"]["points"] if r["tokens"] == N_TOK)
    line = {
        "metric": METRIC, "value": head["GBs"], "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": 3, "ms_per_step": head["us"] * 1e-3, "higher_is_better": True,
        "dtype": "u8", "data": "synthetic (random bytes)",
        "config": {"workload": "sizes: one-shot kvx_transfer of 256 .. 16384 random tokens x 72 "
                               "planes (2 KiB bf16 and 1 KiB fp8 rows), 65536-slot per-plane "
                               "pools, beside a contiguous copy of the same bytes; value = the "
                               "2048-token 2 KiB-row point",
                   "l2": L2_NOTE},
        "sizes": results,
        "contiguous_copy_fit": cfit,
        "gpu_launches": 2 * K * len(sizes) * len(shapes),
    }
    print(json.dumps(line), flush=True)


def run_formats(args):
    print(json.dumps(measure_formats(args)), flush=True)


def measure_formats(args):
    """Pool-to-pool transfers of one request of random slots in other layouts and dtypes, each
    timed like the headline (L2 flushed before every step, CUDA events around kvx_transfer):
      mla_bf16   DeepSeek-V2-Lite-shaped MLA latent rows (27 layers x 576 bf16 = 1152 B),
                 16384 tokens, one plane per layer
      mla_fp8    the same latent rows in fp8 (576 B)
      gqa_fp8    the headline shape in fp8 (36 x K/V x 8 x 128: 1 KiB rows), 2048 tokens
      narrow     200-byte rows (one head of head_dim 100 fp16) through 8-byte accesses
      transcode  the headline shape from a slot-major pool into per-plane pools
      slot_major the headline shape between two slot-major pools ([slot][36][K/V][8][128]: each
                 token's 144 KiB contiguous)
    and, except the narrow rows, the same transfer through kvx_stream with every layer ready."""
    import numpy as np
    import torch

    from disaggregated_paged_kv_gb300 import kvx
    from tests import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvx.lib()
    stream = torch.cuda.Stream(device=dev)
    sp = int(stream.cuda_stream)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)
    peaks, _ = measured_peaks()
    # name: (layers, heads, head_dim, elem bytes, kv_planes, tokens, pool slots,
    #        source slot-major, destination slot-major)
    cases = {
        "mla_bf16": (27, 1, 576, 2, 1, 16384, 65536, False, False),
        "mla_fp8": (27, 1, 576, 1, 1, 16384, 65536, False, False),
        "gqa_fp8": (36, 8, 128, 1, 2, 2048, 65536, False, False),
        "narrow": (36, 1, 100, 2, 2, 16384, 65536, False, False),
        "transcode": (36, 8, 128, 2, 2, 2048, 32768, True, False),
        "slot_major": (36, 8, 128, 2, 2, 2048, 32768, True, True),
    }
    dts = {1: kvx.FP8, 2: kvx.BF16}
    results = {}
    for name, (Lc, Hc, Dc, e, kvp, n, NS, src_sm, dst_sm) in cases.items():
        Pc, Rc = kvp * Lc, Hc * Dc * e
        src = torch.randint(0, 255, (Pc * NS * Rc,), dtype=torch.uint8, device=dev)
        dst = torch.zeros(Pc * NS * Rc, dtype=torch.uint8, device=dev)

        def layout(base, slot_major):
            if slot_major:
                return kvx.Layout(Lc, Hc, Dc, dts[e], NS, base=base, plane_stride=Rc,
                                  slot_stride=Pc * Rc, kv_planes=kvp)
            return kvx.Layout(Lc, Hc, Dc, dts[e], NS, base=base, plane_stride=NS * Rc,
                              kv_planes=kvp)

        sl, dl = layout(src, src_sm), layout(dst, dst_sm)
        s_d = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), n, NS)).to(dev)
        d_d = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), n, NS)).to(dev)
        ws = torch.empty(kvx.workspace_size(n, 0), dtype=torch.uint8, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)

        def step():
            kvx.transfer(sl, s_d, dl, d_d, n, ws, st, stream=sp)

        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush.fill_(1)
                step()
        torch.cuda.synchronize()
        assert int(st.item()) == kvx.OK
        # spot check token 7, plane 1: bytes equal
        k = 7
        so = (int(s_d[k]) * Pc + 1) * Rc if src_sm else (NS + int(s_d[k])) * Rc
        do = (int(d_d[k]) * Pc + 1) * Rc if dst_sm else (NS + int(d_d[k])) * Rc
        assert torch.equal(dst[do:do + Rc], src[so:so + Rc])
        K = args.steps

        def timed(fn):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            with torch.cuda.stream(stream):
                for i in range(K):
                    flush.fill_(i & 0xFF)
                    ev[i][0].record(stream)
                    fn()
                    ev[i][1].record(stream)
            torch.cuda.synchronize()
            return statistics.mean(a.elapsed_time(b) for a, b in ev)

        ms = timed(step)
        alg = 2 * n * Pc * Rc + 8 * n
        gbs = alg / (ms * 1e-3) / 1e9

        def sector_bytes(slots, slot_major):
            """32-byte sectors every row of one side touches, in bytes: a row starting
            `o` bytes past a sector boundary covers ceil((o + R) / 32) sectors."""
            sl_ = slots.cpu().numpy().astype(np.int64)
            planes = np.arange(Pc, dtype=np.int64)
            if slot_major:
                off = (sl_[:, None] * Pc + planes[None, :]) * Rc
            else:
                off = planes[None, :] * NS * Rc + sl_[:, None] * Rc
            return int((((off % 32) + Rc + 31) // 32).sum()) * 32

        sect = sector_bytes(s_d, src_sm) + sector_bytes(d_d, dst_sm)
        results[name] = {"row_bytes": Rc, "planes": Pc, "tokens": n,
                         "payload_bytes_each_way": n * Pc * Rc, "us_per_request": ms * 1e3,
                         "GBs": gbs, "frac_of_measured_hbm": gbs / float(peaks["hbm_gbs"]),
                         "sector_rounded_bytes": sect,
                         "frac_of_measured_hbm_sector_rounded":
                             sect / (ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"])}
        if name != "narrow":  # the streamed kernels move 16-byte vectors only
            st4 = torch.zeros(4, dtype=torch.int32, device=dev)

            def step_stream():
                kvx.stream(kvx.OP_TRANSFER, sl, s_d, dl, d_d, n, None, ws, st4, buf_bytes=0,
                           stream=sp)

            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    flush.fill_(1)
                    step_stream()
            ms_s = timed(step_stream)
            assert st4.tolist()[:2] == [kvx.OK, 0], st4.tolist()
            gbs_s = alg / (ms_s * 1e-3) / 1e9
            results[name]["streamed_us_per_request"] = ms_s * 1e3
            results[name]["streamed_frac_of_measured_hbm"] = gbs_s / float(peaks["hbm_gbs"])
        del src, dst, sl, dl
        torch.cuda.empty_cache()
    head = results["mla_bf16"]
    line = {
        "metric": "KV transfer GB/s (read+write) in other layouts and dtypes",
        "value": head["GBs"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["us_per_request"] * 1e-3,
        "higher_is_better": True, "dtype": "u8", "data": "synthetic (random bytes)",
        "config": {"workload": "pool-to-pool transfers of random slots; value = MLA bf16 "
                               "(27 latent planes x 1152 B, 16384 tokens)",
                   "l2": L2_NOTE},
        "formats": results,
        "gpu_launches": 2 * args.steps,
    }
    return line


def run_tp(args):
    print(json.dumps(measure_tp(args)), flush=True)


def measure_tp(args):
    """The headline request (2048 random tokens, 36 layers x K/V x 8 kv heads x 128 bf16) moved
    between tensor-parallel groups of different sizes: for every (P rank, D rank) pair the heads
    kvx_tp_slice assigns it, one kvx_move_heads transfer each, each pair on its own stream
    (forked from and joined back into the timed stream; also timed with every pair on one
    stream).  A step is the whole reshard (every pair); L2 flushed before each step.  P pools are HND pages of 16
    tokens, D pools per-plane token rows."""
    import numpy as np
    import torch

    from disaggregated_paged_kv_gb300 import kvx
    from tests import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvx.lib()
    stream = torch.cuda.Stream(device=dev)
    sp = int(stream.cuda_stream)
    NS = min(args.pool_slots, 32768)
    gen = torch.Generator(device=dev)
    gen.manual_seed(inputs.seed(2, inputs.ROLE_VALUES))
    s_dev = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N_TOK, NS)).to(dev)
    d_dev = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N_TOK, NS)).to(dev)
    ws = torch.empty(kvx.workspace_size(N_TOK, 0), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)
    peaks, _ = measured_peaks()
    results = {}
    for p_tp, d_tp in ((1, 2), (2, 1), (4, 2), (2, 4), (8, 1)):
        hp, hd = H // p_tp, H // d_tp
        p_pools = [torch.randn((P, NS // 16, hp, 16, D), dtype=torch.bfloat16, device=dev,
                               generator=gen) for _ in range(p_tp)]
        d_pools = [torch.empty((P, NS, hd, D), dtype=torch.bfloat16, device=dev) for _ in range(d_tp)]
        p_l = [kvx.Layout(L, hp, D, kvx.BF16, NS, kind=kvx.HND_PAGED, page_size=16, base=t,
                          plane_stride=NS * hp * D * 2) for t in p_pools]
        d_l = [kvx.Layout(L, hd, D, kvx.BF16, NS, base=t, plane_stride=NS * hd * D * 2)
               for t in d_pools]
        plan = []
        for dr in range(d_tp):
            for pr in range(p_tp):
                sh0, dh0, nh = kvx.tp_slice(H, p_tp, pr, d_tp, dr)
                if nh:
                    plan.append((pr, dr, sh0, dh0, nh))

        # one stream, workspace and status per pair: independent pairs overlap on the GPU
        side = [torch.cuda.Stream(device=dev) for _ in plan]
        wss = [torch.empty(kvx.workspace_size(N_TOK, 0), dtype=torch.uint8, device=dev)
               for _ in plan]
        sts = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in plan]
        fork = torch.cuda.Event()
        joins = [torch.cuda.Event() for _ in plan]

        def step():
            fork.record(stream)
            for j, (pr, dr, sh0, dh0, nh) in enumerate(plan):
                side[j].wait_event(fork)
                kvx.move_heads(kvx.OP_TRANSFER, p_l[pr], s_dev, sh0, d_l[dr], d_dev, dh0, nh,
                               N_TOK, None, wss[j], sts[j], buf_bytes=0,
                               stream=int(side[j].cuda_stream))
                joins[j].record(side[j])
            for ev_j in joins:
                stream.wait_event(ev_j)

        def step_serial():
            for pr, dr, sh0, dh0, nh in plan:
                kvx.move_heads(kvx.OP_TRANSFER, p_l[pr], s_dev, sh0, d_l[dr], d_dev, dh0, nh,
                               N_TOK, None, ws, st, buf_bytes=0, stream=sp)

        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush.fill_(1)
                step()
                step_serial()
        torch.cuda.synchronize()
        assert int(st.item()) == kvx.OK and all(int(x.item()) == kvx.OK for x in sts)
        # spot check: token k, plane 0, first moved head of the first pair
        pr, dr, sh0, dh0, nh = plan[0]
        k = 97
        sslot, dslot = int(s_dev[k]), int(d_dev[k])
        got = d_pools[dr][0, dslot, dh0:dh0 + nh]
        want = p_pools[pr][0, sslot // 16, sh0:sh0 + nh, sslot % 16]
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
        K = args.steps

        def timed(fn):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            with torch.cuda.stream(stream):
                for i in range(K):
                    flush.fill_(i & 0xFF)
                    ev[i][0].record(stream)
                    fn()
                    ev[i][1].record(stream)
            torch.cuda.synchronize()
            return statistics.mean(a.elapsed_time(b) for a, b in ev)

        ms = timed(step)
        ms_serial = timed(step_serial)

        # the whole plan in one kvx_reshard call (one planner + one copy launch)
        def step_one():
            kvx.reshard(p_l, s_dev, d_l, d_dev, plan, N_TOK, ws, st, stream=sp)

        for t in d_pools:
            t.zero_()
        torch.cuda.synchronize()  # the zeroing ran on torch's current stream, not on `stream`
        with torch.cuda.stream(stream):
            step_one()
        torch.cuda.synchronize()
        assert int(st.item()) == kvx.OK
        for pr, dr, sh0, dh0, nh in plan:  # spot check: three tokens, two planes, every part
            for k, pl in ((0, 0), (1001, P - 1), (N_TOK - 1, 37 % P)):
                sslot, dslot = int(s_dev[k]), int(d_dev[k])
                got = d_pools[dr][pl, dslot, dh0:dh0 + nh]
                want = p_pools[pr][pl, sslot // 16, sh0:sh0 + nh, sslot % 16]
                assert torch.equal(got.view(torch.int16), want.view(torch.int16))
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush.fill_(1)
                step_one()
        ms_one = timed(step_one)
        assert int(st.item()) == kvx.OK

        # the same plan layer-streamed (kvx_stream_reshard), every layer's ready word raised
        words = torch.ones(L, dtype=torch.int32, device=dev)
        st4 = torch.zeros(4, dtype=torch.int32, device=dev)

        def step_streamed():
            kvx.stream_reshard(p_l, s_dev, d_l, d_dev, plan, N_TOK, ws, st4, layer_ready=words,
                               ready_value=1, stream=sp)

        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush.fill_(1)
                step_streamed()
        ms_streamed = timed(step_streamed)
        assert st4.tolist() == [kvx.OK, 0, 0, 1], st4.tolist()
        # ... and on a persistent grid capped at half the SMs (the rest left to a producer)
        half = torch.cuda.get_device_properties(dev).multi_processor_count // 2

        def step_capped():
            kvx.stream_reshard(p_l, s_dev, d_l, d_dev, plan, N_TOK, ws, st4, layer_ready=words,
                               ready_value=1, max_ctas=half, stream=sp)

        with torch.cuda.stream(stream):
            for _ in range(3):
                flush.fill_(1)
                step_capped()
        ms_capped = timed(step_capped)
        v4 = st4.tolist()
        assert v4[0:2] == [kvx.OK, 0] and v4[3] == 1, v4
        alg = alg_bytes(N_TOK) + 8 * N_TOK * (len(plan) - 1)  # every pair reads both lists
        gbs = alg / (ms * 1e-3) / 1e9
        gbs_one = alg_bytes(N_TOK) / (ms_one * 1e-3) / 1e9
        results[f"p{p_tp}_to_d{d_tp}"] = {
            "pairs": len(plan), "launches_per_reshard": 2 * len(plan),
            "us_per_reshard": ms * 1e3, "GBs": gbs,
            "frac_of_measured_hbm": gbs / float(peaks["hbm_gbs"]),
            "us_per_reshard_one_stream": ms_serial * 1e3,
            "us_per_reshard_one_call": ms_one * 1e3, "GBs_one_call": gbs_one,
            "frac_of_measured_hbm_one_call": gbs_one / float(peaks["hbm_gbs"]),
            "us_per_reshard_streamed_all_ready": ms_streamed * 1e3,
            "us_per_reshard_streamed_half_the_sms": ms_capped * 1e3,
            "slice_bytes": plan[0][4] * D * 2}
        del p_pools, d_pools, p_l, d_l
        torch.cuda.empty_cache()
    head = results["p8_to_d1"]
    line = {
        "metric": "KV reshard between TP groups in one kvx_reshard call at 288 MiB: GB/s "
                  "(read+write)",
        "value": head["GBs_one_call"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["us_per_reshard_one_call"] * 1e-3,
        "higher_is_better": True, "dtype": "u8", "data": "synthetic",
        "config": {"workload": "2048-token prompt, 36 layers x K/V x 8 kv heads x 128 bf16 "
                               "(288 MiB) moved from the HND pools (page 16) of a P TP group to "
                               "the token-row pools of a D TP group; value = P TP 8 -> D TP 1 "
                               "(each D row merged from eight 256-byte pieces) in one call; "
                               "every plan also timed pair by pair (kvx_move_heads)",
                   "pool_slots": NS,
                   "l2": L2_NOTE},
        "reshards": results,
        "gpu_launches": 2 * args.steps,
    }
    return line


def run_stream(args):
    print(json.dumps(measure_stream(args)), flush=True)


def measure_stream(args):
    """The headline transfer through kvx_stream.  (1) Every layer ready: device time of
    memset + planner + streamed copy per step, L2 flushed before each step.  (2) Layers raised
    by the host at a fixed cadence (an emulated prefill producing one layer every --layer-us):
    host time from raising the last layer to seeing the kernel's pinned "done" word.  (3) The
    same move started only after the last layer (no streaming): host time from the launch to
    the same word.  (4) Epoch-fenced writes: every layer ready with the request's epoch word or
    every destination page's owner word checked (device time), and a cancellation after half
    the layers (host time from changing the pinned epoch word to the "done" word)."""
    import numpy as np
    import torch

    from disaggregated_paged_kv_gb300 import kvx
    from tests import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvx.lib()
    NS = args.pool_slots
    stream = torch.cuda.Stream(device=dev)
    sp = int(stream.cuda_stream)
    gen = torch.Generator(device=dev)
    gen.manual_seed(inputs.seed(2, inputs.ROLE_VALUES))
    src = torch.randn((P, NS, H, D), dtype=torch.bfloat16, device=dev, generator=gen)
    dst = torch.empty((P, NS, H, D), dtype=torch.bfloat16, device=dev)
    dst.view(torch.int16).fill_(0x7FC1)
    s_dev = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, inputs.ROLE_SRC_SLOTS), N_TOK, NS)).to(dev)
    d_dev = torch.from_numpy(inputs.distinct_slots(inputs.rng(2, inputs.ROLE_DST_SLOTS), N_TOK, NS)).to(dev)
    src_l = kvx.Layout(L, H, D, kvx.BF16, NS, base=src, plane_stride=NS * R)
    dst_l = kvx.Layout(L, H, D, kvx.BF16, NS, base=dst, plane_stride=NS * R)
    ws = torch.empty(kvx.workspace_size(N_TOK, 0), dtype=torch.uint8, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(dev, l2)
    ready = torch.zeros(L, dtype=torch.int32).pin_memory()
    done = torch.zeros(1, dtype=torch.int32).pin_memory()

    def launch(**kw):
        kvx.stream(kvx.OP_TRANSFER, src_l, s_dev, dst_l, d_dev, N_TOK, None, ws, st,
                   buf_bytes=0, stream=sp, **kw)

    # (1) every layer ready
    K = args.steps
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            launch()
    torch.cuda.synchronize()
    assert st.tolist()[:2] == [kvx.OK, 0]
    k = torch.from_numpy(np.arange(0, N_TOK, 97)).to(dev)
    assert torch.equal(dst[:, d_dev[k]].view(torch.int16), src[:, s_dev[k]].view(torch.int16))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = Clocks(0, not args.no_clocks)
    time.sleep(0.3 if clocks.proc else 0)
    with torch.cuda.stream(stream):
        for i in range(K):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            launch()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    def timed(**kw):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        with torch.cuda.stream(stream):
            for i in range(K):
                flush.fill_(i & 0xFF)
                evs[i][0].record(stream)
                launch(**kw)
                evs[i][1].record(stream)
        torch.cuda.synchronize()
        assert st.tolist()[:2] == [kvx.OK, 0], st.tolist()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    # every layer ready, through device ready words already raised; and on a persistent grid
    words = torch.ones(L, dtype=torch.int32, device=dev)
    words_ms = timed(layer_ready=words, ready_value=1)
    # persistent grids capped at a fraction of the SMs (the rest left to a producer), in the
    # bulk (TMA) form and the register form
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    persistent = {"ctas": [], "mixed_us": [], "registers_us": [], "bulk_us": []}
    for ctas in (sms // 8, sms // 4, sms // 2, sms):
        persistent["ctas"].append(ctas)
        for key, engine in (("mixed_us", kvx.ENGINE_AUTO), ("registers_us", kvx.ENGINE_REGISTERS),
                            ("bulk_us", kvx.ENGINE_BULK)):
            kvx.set_copy_engine(engine)
            try:
                persistent[key].append(timed(max_ctas=ctas) * 1e3)
            finally:
                kvx.set_copy_engine(kvx.ENGINE_AUTO)

    # epoch-fenced writes: the request's epoch word checked, or every destination page's owner
    # word checked (nothing cancelled or reassigned: the cost of the checks alone)
    ep_word = torch.full((1,), 7, dtype=torch.int32, device=dev)
    epoch_ms = timed(epoch_word=ep_word, epoch=7)
    page_ep = torch.full(((NS + 15) // 16,), 7, dtype=torch.int32, device=dev)
    pages_ms = timed(dst_page_epochs=page_ep, epoch_page=16, epoch=7)

    # (2) layers raised by the host at a fixed cadence; (3) the move started after the last one
    cadence = args.layer_us * 1e-6
    trials = 0 if args.device_only else 30

    # numpy views of the pinned words: a poll or a store costs ~0.1 us instead of the ~1-2 us
    # of indexing a torch tensor from Python, so the host's own overhead stays out of the tails
    done_np, ready_np = done.numpy(), ready.numpy()

    def wait_done(t_from):
        while done_np[0] == 0 and time.perf_counter() < t_from + 2.0:
            pass
        return time.perf_counter()

    tails, unstreamed = [], []
    for trial in range(trials):
        v = trial + 1
        done[0] = 0
        flush.fill_(trial & 0xFF)
        torch.cuda.synchronize()
        launch(layer_ready=ready, ready_value=v, wait_ns=1_000_000_000, host_done=done)
        t0 = time.perf_counter()
        for layer in range(L):
            target = t0 + (layer + 1) * cadence
            while time.perf_counter() < target:
                pass
            ready_np[layer] = v
        t_last = time.perf_counter()
        tails.append((wait_done(t_last) - t_last) * 1e6)
        torch.cuda.synchronize()
        assert st.tolist()[:2] == [kvx.OK, 0], st.tolist()

        done[0] = 0
        flush.fill_(trial & 0xFF)
        torch.cuda.synchronize()
        t_last = time.perf_counter()
        launch(host_done=done)
        unstreamed.append((wait_done(t_last) - t_last) * 1e6)
        torch.cuda.synchronize()
        assert st.tolist()[:2] == [kvx.OK, 0], st.tolist()

    # (4) a cancellation: half the layers raised at the cadence, then the host changes the
    # request's epoch word (pinned); host time from the change to the "no further write" word
    ep_host = torch.zeros(1, dtype=torch.int32).pin_memory()
    ep_np = ep_host.numpy()
    cancels, pending = [], []
    for trial in range(trials):
        v = 1000 + trial  # above every ready value used so far
        ep_host[0] = v
        done[0] = 0
        flush.fill_(trial & 0xFF)
        torch.cuda.synchronize()
        launch(layer_ready=ready, ready_value=v, epoch_word=ep_host, epoch=v,
               wait_ns=1_000_000_000, host_done=done)
        t0 = time.perf_counter()
        for layer in range(L // 2):
            target = t0 + (layer + 1) * cadence
            while time.perf_counter() < target:
                pass
            ready_np[layer] = v
        t_c = time.perf_counter()
        ep_np[0] = v + 1
        cancels.append((wait_done(t_c) - t_c) * 1e6)
        torch.cuda.synchronize()
        s_ = st.tolist()
        assert s_[0] == kvx.ERR_CANCELLED and s_[3] == 1 and L - L // 2 <= s_[1] <= L, s_
        pending.append(s_[1])

    def pct(xs):
        if not xs:
            return None
        xs = sorted(xs)
        return {"median": xs[len(xs) // 2], "p10": xs[len(xs) // 10], "p90": xs[(9 * len(xs)) // 10]}

    peaks, peak_kind = measured_peaks()
    gbs = alg_bytes(N_TOK) / (step_ms * 1e-3) / 1e9
    line = {
        "metric": "layer-streamed KV transfer (kvx_stream) at 288 MiB: GB/s with every layer "
                  "ready; us from the last layer raised to the move acknowledged",
        "value": gbs, "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "dtype": "u8", "data": "synthetic",
        "config": {"workload": WORKLOAD + "; through kvx_stream", "pool_slots": NS,
                   "l2": L2_NOTE},
        "all_ready": {"us_per_request": step_ms * 1e3, "GBs": gbs,
                      "frac_of_measured_hbm": gbs / float(peaks["hbm_gbs"]),
                      "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
                      "includes": "planner + streamed copy + epilogue"},
        "all_ready_device_words_us": words_ms * 1e3,
        "all_ready_persistent_grid": dict(persistent, how=(
            "max_ctas CTAs for the whole move, one per SM at most; mixed (the default): 29 "
            "register warps and 3 warps of TMA bulk-copy threads per CTA (one 2 KiB shared-"
            "memory stage each); registers (KVX_ENGINE_REGISTERS): 32 register warps; bulk "
            "(KVX_ENGINE_BULK): 96 TMA bulk-copy threads")),
        "all_ready_request_epoch_checked_us": epoch_ms * 1e3,
        "all_ready_page_owners_checked_us": pages_ms * 1e3,
        "cancel_to_no_further_write_us": pct(cancels),
        "cancel_layers_pending": ({"min": min(pending), "max": max(pending),
                                   "of": L, "raised_before_cancel": L // 2} if pending else None),
        "streamed_tail_us": pct(tails),
        "unstreamed_us": pct(unstreamed),
        "producer": f"host raises one layer every {args.layer_us:g} us into pinned ready words; "
                    f"{trials} trials; times on the host clock (time.perf_counter), the kernel's "
                    "done word polled in pinned memory",
        "clocks": clk,
        "gpu_launches": 3 * K,  # validating planner, streamed row grid, epilogue
    }
    return line


def next_row_summaries(args):
    """The layer-streamed move, the TP reshards and the other formats, each measured as by
    --workload stream / tp / formats (at most 200 timed steps per measurement), with the SM
    clocks sampled over each, and summarised for the headline line."""
    import torch

    sub = argparse.Namespace(**vars(args))
    sub.steps = min(args.steps, 200)
    sub.warmup = max(3, min(args.warmup, 10))
    out = {}
    for name, fn in (("stream", measure_stream), ("tp", measure_tp), ("formats", measure_formats)):
        torch.cuda.empty_cache()
        clocks = Clocks(0, not args.no_clocks)
        ln = fn(sub)
        clk = clocks.stop()
        if name == "stream":
            ar = ln["all_ready"]
            pg = ln["all_ready_persistent_grid"]
            out[name] = {
                "all_ready_us": ar["us_per_request"], "GBs": ar["GBs"],
                "frac_of_measured_hbm": ar["frac_of_measured_hbm"],
                "all_ready_device_words_us": ln["all_ready_device_words_us"],
                "persistent_grid_mixed_us": dict(zip(map(str, pg["ctas"]), pg["mixed_us"])),
                "request_epoch_checked_us": ln["all_ready_request_epoch_checked_us"],
                "page_owners_checked_us": ln["all_ready_page_owners_checked_us"],
                "tail_after_last_layer_us": ln["streamed_tail_us"],
                "unstreamed_us": ln["unstreamed_us"],
                "cancel_to_no_further_write_us": ln["cancel_to_no_further_write_us"],
                "workload": ln["config"]["workload"]}
        elif name == "tp":
            out[name] = {k: {"one_call_us": v["us_per_reshard_one_call"],
                             "one_call_frac_of_measured_hbm": v["frac_of_measured_hbm_one_call"],
                             "pairs_us": v["us_per_reshard"],
                             "streamed_all_ready_us": v["us_per_reshard_streamed_all_ready"],
                             "streamed_half_the_sms_us": v["us_per_reshard_streamed_half_the_sms"]}
                         for k, v in ln["reshards"].items()}
            out[name]["workload"] = ln["config"]["workload"]
        else:
            out[name] = {k: {"row_bytes": v["row_bytes"], "us": v["us_per_request"],
                             "frac_of_measured_hbm": v["frac_of_measured_hbm"],
                             "frac_of_measured_hbm_sector_rounded":
                                 v["frac_of_measured_hbm_sector_rounded"],
                             **({"streamed_us": v["streamed_us_per_request"]}
                                if "streamed_us_per_request" in v else {})}
                         for k, v in ln["formats"].items()}
        out[name]["steps"] = sub.steps
        out[name]["clocks"] = clk
    torch.cuda.empty_cache()
    return out


def host_description():
    """nproc and the CPU model of this host."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.TimeoutExpired):
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model or "unknown"}


def workload_config() -> dict:
    """The headline workload, as both arms state it."""
    return {"workload": WORKLOAD, "kv_dtype": "bf16", "tokens": N_TOK, "planes": P,
            "row_bytes": R, "pool_slots": SLOTS, "payload_bytes_each_way": N_TOK * P * R,
            "alg_bytes_per_step": alg_bytes(N_TOK)}


def cpu_baseline(budget_s: float = 10.0):
    pool_slots = SLOTS
    ob = OracleTransfer(N_TOK, pool_slots)
    ob.run(reps=1)  # warm
    sec, reps = ob.run(budget_s=budget_s, min_reps=3)
    sec_all, threads = ob.run_all_cores()
    return {"value": alg_bytes(N_TOK) / sec / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "us_per_request": sec * 1e6,
            "sample": f"the full 2048-token x 72-plane transfer (288 MiB each way) between host "
                      f"pools of {pool_slots} slots per plane (2 x "
                      f"{P * pool_slots * R / 2**30:.2f} GiB, the GPU arm's pools), with the same "
                      f"slot lists, repeated {reps} times in {sec * reps:.1f} s; single thread",
            "host": host_description(),
            "all_cores": {"value": alg_bytes(N_TOK) / sec_all / 1e9, "unit": UNIT,
                          "threads": threads, "us_per_request": sec_all * 1e6,
                          "kind": "the oracle's transfer split by layer ranges over every core "
                                  "(a labelled CPU line, not the oracle as it stands)"}}


def run_reference(args, rank: int):
    """The reference arm: the oracle, as it stands, on the host cores, on the GPU arm's
    workload: each step is the whole 2048-token transfer between host pools of the GPU arm's
    size, with the same slot lists (~80 ms a step on one Neoverse-V2 core)."""
    if rank != 0:
        return
    ob = OracleTransfer(N_TOK, SLOTS)
    ob.run(reps=max(1, args.warmup))
    sec, _ = ob.run(reps=args.steps)
    value = alg_bytes(N_TOK) / sec / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic",
            "config": dict(workload_config(), parallelism="single host thread",
                           us_per_request=sec * 1e6),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "each step: the whole 2048-token x 72-plane transfer (288 MiB "
                                       "each way) between host pools of 65,536 slots per plane "
                                       "(2 x 9 GiB), the GPU arm's workload; single thread",
                             "host": host_description()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------

def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.fused_max is not None:
        from disaggregated_paged_kv_gb300 import kvx
        kvx.set_fused_max_tokens(args.fused_max)
    if args.check_duplicates:
        from disaggregated_paged_kv_gb300 import kvx
        kvx.set_check_duplicates(True)
    if args.workload == "stream":
        run_stream(args)
        return
    if args.workload == "tp":
        run_tp(args)
        return
    if args.workload == "formats":
        run_formats(args)
        return
    if args.workload == "comparators":
        run_comparators(args)
        return
    if args.workload == "sizes":
        run_sizes(args)
        return
    if args.workload != "transfer":
        run_workload(args, args.workload)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    K = args.steps
    ms_per_step = res["total_ms"] / K
    value = whole_job_gbs(alg_bytes(N_TOK), K, world, res["total_ms"])
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    copy_bytes = 2 * N_TOK * P * R
    achieved = copy_bytes / (res["copy_ms"] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {**workload_config(), "pool_slots": args.pool_slots,
                   "us_per_request": ms_per_step * 1e3,
                   "us_per_request_p10_median_p90": step_percentiles(res["step_ms"]),
                   "frac_of_measured_hbm": value / hbm,
                   "frac_of_nominal_8tbs": value / NOMINAL_HBM_GBS,
                   "plan_us": res["plan_ms"] * 1e3, "copy_us": res["copy_ms"] * 1e3,
                   "contiguous_copy_us": res["contiguous_ms"] * 1e3,
                   "l2": L2_NOTE,
                   "steady_state_no_flush": {
                       "us_per_request": res["noflush_ms"] * 1e3,
                       "GBs": alg_bytes(N_TOK) / (res["noflush_ms"] * 1e-3) / 1e9,
                       "frac_of_measured_hbm": alg_bytes(N_TOK) / (res["noflush_ms"] * 1e-3)
                       / 1e9 / hbm,
                       "how": "back-to-back requests, no flush: inputs larger than L2 (288 MiB "
                              "each way per step), two sets of random slot lists in turn"},
                   "write_only_flush": {
                       "us_per_request": res["write_only_ms"] * 1e3,
                       "GBs": alg_bytes(N_TOK) / (res["write_only_ms"] * 1e-3) / 1e9,
                       "how": "the same step after a flush that only writes 2x L2: the step "
                              "then also writes back the flush's dirty lines (up to the L2 "
                              "size)"},
                   "cuda_graph_replay": {
                       "us_per_request": res["graph_ms"] * 1e3,
                       "GBs": alg_bytes(N_TOK) / (res["graph_ms"] * 1e-3) / 1e9,
                       "how": "the one kvx_transfer call (planner + copy) captured once into a "
                              "CUDA graph and replayed each step, L2 flushed as above"},
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "duplicate_check": bool(args.check_duplicates),
                   "device": res["device"]},
        "clocks": res["clocks"],
        "e2e": res["e2e"],
        "gpu_launches": 2 * K,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": UNIT,
                     "frac": achieved / hbm, "traffic": profile_traffic(),
                     "traffic_over_alg": (profile_traffic() / copy_bytes
                                          if profile_traffic() else None),
                     "kernel": "copy_row_kernel (one warp per 2 KiB row)",
                     "peak_kind": f"{peak_kind} (burst copy)",
                     "achieved_bytes_per_launch": copy_bytes},
    }
    if world == 1 and not args.no_workloads:
        del res
        line["config"]["workloads"] = workload_summaries(args)
    if world == 1 and not args.no_next_rows:
        line["config"]["next_rows"] = next_row_summaries(args)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
