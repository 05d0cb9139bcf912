"""Throughput of the fused decode-time sampler on GB300.

One step = one strata_sample_rows call over one batch: the logprobs workload (8 fp32 rows, V=248,320,
N(0,3^2) logits with 1-5 spikes), every row a sampled request with the single-row request's keys
(penalties over a 64-token history, top_k 20, min_p 0.05, top_p 0.95, T 0.8, Philox draw), fused
with top_logprobs=20, the sampled token's log-probability and allowed_token_ids subsets of 5, 100 and
1000 ids.  That runs every step of the hot path in one launch.

  value      rows/s over exactly K timed steps: one CUDA graph holding the K calls, replayed once;
             inputs rotate over enough distinct batches to exceed 4x the L2 size (HBM serves reads).
             The steps alternate over S independent request groups (`--streams`, default 8): each
             group is its own context (own slots and counters) with its own stream, its calls
             chained in order, the groups' calls overlapping, with the concurrency launch hint.
             Call i writes output set i % R (`STRATA_FLAG_OWN_OUTPUTS`; `--no-own-outputs` gives
             each group one set), so no call waits for the previous one.
  single_group  the same K steps as one group alone into one set of buffers (one stream, the
             library's pipelined launch shape): each call waits for the previous call before its
             counters and writes.
  e2e        the same metric through the C ABI from pinned host buffers: every step copies its
             inputs host->device (the logits, and the small arrays packed into one copy), runs the
             call and copies every output back (one packed copy); copies run on their own streams
             into two buffer sets, so one step's inputs travel while the previous step samples; the
             calls stay in order on one stream; the K steps are one CUDA graph.
  roofline   algorithmic bytes per launch / average launch time, against the measured HBM copy
             bandwidth; `traffic` is the DRAM bytes per launch from the committed ncu summary when
             the kernel source still matches it.
  cpu_baseline  the CPU oracle (plain numpy) on a bounded sample of the same workload, 1 core.

Other workloads (`--workload`): `verify` (config 2's five-row verify windows, strata_sample_verify),
`verify-ring` (the same windows over histories kept on the device), `mask` (the default step with its
allowed ids as a sampling mask).  `--split N` forces N blocks per row (launch-shape sweeps).

`--impl reference` times the CPU oracle alone on the same workload (one row per step).
Multi-GPU (torchrun): every rank runs its own batch stream (weak scaling, no collective on the data
path); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "sampled rows/s and achieved HBM GB/s (fraction of GB300 peak) at V=248,320"
UNIT = "rows/s"
WORKLOAD = ("logprobs workload fused with sampling: B=8 fp32 rows x V=248,320, N(0,3^2)+1..5 spikes; "
            "per-row keys top_k=20 T=0.8 top_p=0.95 min_p=0.05 repeat=1.1 freq=0.1 presence=0.1 "
            "penalty_last_n=64; top_logprobs=20, chosen-token logprob, allowed_token_ids of 5/100/1000")
WORKLOAD_VERIFY = ("verify windows (strata_sample_verify): config 2's 5-row windows (4 drafts + head), 1 slot, "
                   "fp32 V=248,320, N(0,3^2)+1..5 spikes; keys T=0.7 top_k=20 top_p=0.9 min_p=0.05 repeat=1.1 "
                   "over a 64-token history; seeded draft ids; kept rows counted in the launch")
WORKLOAD_MASK = WORKLOAD + "; the allowed ids used as a sampling mask (STRATA_FLAG_ALLOWED_MASK)"
WORKLOAD_VERIFY_RING = (WORKLOAD_VERIFY + "; the 64-token window read from the slot's history kept on the device "
                        "(STRATA_FLAG_HISTORY_RING) and the kept picks appended in the launch")
KERNEL_SOURCES = ("request_token_sampling_gb300/csrc/strata_kernel.cuh",   # the device code the
                  "request_token_sampling_gb300/csrc/strata_device.cuh")   # ncu counters describe
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_config4_fused.json")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def algorithmic_bytes(w) -> int:
    """Bytes a launch must move at least: logits once, history windows, allowed ids, row arrays,
    slot keys and counters, and every output."""
    B, V = w["B"], w["V"]
    esz = 4 if w["dtype"] == "f32" else 2
    n = B * V * esz
    for s in range(w["n_hist_slots"]):
        ln = w["slot_params"][s]["penalty_last_n"]
        n += 4 * min(ln, int(w["hist_off"][s + 1] - w["hist_off"][s]))
    n_allowed = int(w["allowed_off"][-1]) if w.get("allowed_off") is not None else 0
    n += 4 * n_allowed + 4 * (B + 1) + 4 * (w["n_hist_slots"] + 1)          # allowed ids, offsets
    n += B * (4 + 8)                                                          # row slot + position
    n += len(w["slot_params"]) * (48 + 8 + 4)                                 # slot keys, counter
    n += B * (4 + 4 + w["top_n"] * 8) + 4 * n_allowed                         # outputs
    return n


def algorithmic_bytes_verify(w, ring=False) -> int:
    """Logits once, the history window, row arrays with drafts, slot keys and counter, picks and
    the kept count (with a kept history: its length read and written, the kept picks written;
    counted as the whole window)."""
    B, V = w["B"], w["V"]
    n = B * V * 4 + 4 * min(w["slot_params"][0]["penalty_last_n"], int(w["hist_off"][1] - w["hist_off"][0]))
    n += 4 * 2 + B * (4 + 8 + 4) + (48 + 8 + 4) + B * 4 + 4
    if ring:
        n += 16 + 4 * B
    return n


def oracle_windows_per_s(w, drafts, budget_s=15.0, max_windows=40, ring=False):
    """Time the unmodified oracle on whole verify windows (rows per second); with `ring`, windows
    whose history is kept between calls."""
    import oracle
    t0 = time.perf_counter()
    n = 0
    counters = dict(w["counters"])
    state = {0: [int(x) for x in w["hist"]]}
    while True:
        if ring:
            _, counters, state, _ = oracle.history_call(w, state, counters=counters, row_draft=drafts)
        else:
            _, counters, _ = oracle.verify_call(w, drafts, counters=counters)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= max_windows:
            return n * w["B"] / el, n, el


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank number over all ranks (the slowest rank sets the job's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job throughput: every rank processes its own rows (weak scaling)."""
    return world * rows_per_rank / seconds


# ------------------------------------------------------------------------------ clocks (NVML)
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str | None):
        self.ok = False
        self.samples = []
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            rc = -1
            if pci_bus_id:
                rc = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h))
            if rc != 0:
                return
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            pass

    def _read(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c))
        self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(r))
        return int(c.value), int(r.value)

    def _run(self):
        while not self._stop.is_set():
            self.samples.append(self._read())
            time.sleep(0.001)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self.t.join()
            self.samples.append(self._read())

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        mhz = [m for m, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = [n for b, n in self.REASONS.items() if bits & b]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples)}


# ------------------------------------------------------------------------------ CPU oracle timing
def oracle_rows_per_s(w, budget_s=15.0, max_rows=400, mask=False):
    """Time the unmodified oracle on rows of the workload (fused sample + logprobs + allowed)."""
    import oracle
    t0 = time.perf_counter()
    rows = 0
    counters = dict(w["counters"])
    while True:
        b = rows % w["B"]
        wb = dict(w)
        wb["B"] = 1
        wb["logits"] = w["logits"][b:b + 1]
        wb["row_slot"] = w["row_slot"][b:b + 1]
        wb["row_pos"] = w["row_pos"][b:b + 1]
        off = w["allowed_off"]
        wb["allowed"] = w["allowed"][off[b]:off[b + 1]]
        wb["allowed_off"] = np.array([0, off[b + 1] - off[b]], np.int32)
        _, counters = oracle.sample_call(wb, counters=counters, mask_allowed=mask)
        rows += 1
        el = time.perf_counter() - t0
        if el >= budget_s or rows >= max_rows:
            return rows / el, rows, el


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = synth.config4(fused=True)
    import oracle
    counters = dict(w["counters"])

    def step(i):
        nonlocal counters
        b = i % w["B"]
        wb = dict(w)
        wb["B"] = 1
        wb["logits"] = w["logits"][b:b + 1]
        wb["row_slot"] = w["row_slot"][b:b + 1]
        wb["row_pos"] = w["row_pos"][b:b + 1]
        off = w["allowed_off"]
        wb["allowed"] = w["allowed"][off[b]:off[b + 1]]
        wb["allowed_off"] = np.array([0, off[b + 1] - off[b]], np.int32)
        _, counters = oracle.sample_call(wb, counters=counters)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    v = args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32(penalty,ranking)+f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "rows_per_step": 1},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} timed rows of the 8-row batch, one row per step"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ GPU arm
def make_batches(w, R, dev):
    """R distinct device batches with the workload's recipe (batch 0 is the workload itself)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(0x5EED0004)
    out = [torch.from_numpy(w["logits"]).to(dev)]
    B, V = w["B"], w["V"]
    for _ in range(R - 1):
        x = torch.randn((B, V), generator=g, device=dev) * 3.0
        n = torch.randint(1, 6, (B,), generator=g, device=dev)
        for b in range(B):
            ids = torch.randint(0, V, (int(n[b]),), generator=g, device=dev)
            x[b, ids] = torch.rand((int(n[b]),), generator=g, device=dev) * 7.0 + 8.0
        out.append(x.contiguous())
    return out


def run_gpu(args, rank, world):
    import torch
    import torch.distributed as dist
    from request_token_sampling_gb300 import (STRATA_FLAG_ALLOWED_MASK, STRATA_FLAG_CONCURRENT, STRATA_FLAG_EARLY_LOAD,
                                              STRATA_FLAG_HISTORY_RING, STRATA_FLAG_OWN_OUTPUTS, STRATA_FLAG_PDL,
                                              STRATA_FLAG_SPLIT, Sampler)

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    verify = args.workload in ("verify", "verify-ring")
    ring = args.workload == "verify-ring"
    w = synth.config2_window(0) if verify else synth.config4(fused=True)
    B = w["B"]
    step_bytes = B * w["V"] * 4
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    R = max(2, -(-4 * l2 // step_bytes)) if args.batches <= 0 else args.batches
    flags = 0 if args.no_pdl else (STRATA_FLAG_PDL | (0 if args.no_early_load else STRATA_FLAG_EARLY_LOAD))
    if args.workload == "mask":
        flags |= STRATA_FLAG_ALLOWED_MASK
    if ring:
        flags |= STRATA_FLAG_HISTORY_RING
    if args.split > 0:
        flags |= STRATA_FLAG_SPLIT(args.split)
    elif args.streams > 1:  # other groups' calls run alongside: the launch shape for throughput
        flags |= STRATA_FLAG_CONCURRENT
    # every call writes its own output buffers (they rotate like the inputs), so no call waits for
    # the one before it; verify windows and kept histories depend on the previous call by nature
    own = (not args.no_own_outputs and (flags & STRATA_FLAG_EARLY_LOAD) != 0 and not verify)
    if own:
        flags |= STRATA_FLAG_OWN_OUTPUTS

    # S independent request groups: a context each (its own slots, counters and outputs), a stream
    # each; one group's calls are ordered, the groups' calls overlap
    S = max(1, args.streams)
    samplers = []
    for _ in range(S):
        sg = Sampler(device=local, max_slots=16, max_vocab=w["V"], max_rows=B)
        for slot, p in w["slot_params"].items():
            sg.restore_slot(slot, p, 0)
        samplers.append(sg)
    s = samplers[0]
    ten = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    row_slot, row_pos = ten(w["row_slot"]), ten(w["row_pos"])
    hist, hist_off = ten(w["hist"]), ten(w["hist_off"])
    if ring:  # the window lives in the slot's kept history; the call uploads none
        for sg in samplers:
            sg.history_enable()
            sg.history_set(0, w["hist"])
        hist = hist_off = None
    allowed = allowed_off = None
    if not verify:
        allowed, allowed_off = ten(w["allowed"]), ten(w["allowed_off"])
    drafts = np.random.default_rng(0x5EED0002).integers(0, w["V"], size=B).astype(np.int32)
    drafts[-1] = -1
    row_draft = ten(drafts)
    batches = make_batches(w, R, dev)
    outs = []
    for sg in samplers:
        if verify:
            outs.append(sg.verify(batches[0], row_slot, row_pos, row_draft, hist=hist, hist_off=hist_off, flags=flags))
        else:
            outs.append(sg.sample(batches[0], row_slot, row_pos, hist=hist, hist_off=hist_off, top_n=w["top_n"],
                                  chosen_lp=True, allowed=allowed, allowed_off=allowed_off, flags=flags))
    out = outs[0]
    # with own outputs, call i writes output set i % R: more sets than calls can be resident at once
    out_sets = [{k: torch.empty_like(v) for k, v in out.items()} for _ in range(R)] if own else None
    torch.cuda.synchronize()
    if any(sg.errors() != 0 for sg in samplers):
        raise RuntimeError("device error bits set")
    # the launch shape of a call with these flags (mode 2: verify windows)
    shape = s.shape(2 if verify else 0, 0, B, w["V"], w["top_n"], flags)

    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    gstreams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(S - 1)]

    def call_on(sg, st, o, fl, i):
        if verify:
            sg.verify(batches[i % R], row_slot, row_pos, row_draft, hist=hist, hist_off=hist_off, flags=fl,
                      stream=st, out=o)
        else:
            sg.sample(batches[i % R], row_slot, row_pos, hist=hist, hist_off=hist_off, top_n=w["top_n"],
                      chosen_lp=True, allowed=allowed, allowed_off=allowed_off, flags=fl, stream=st, out=o)

    def call(i):
        g = i % S
        call_on(samplers[g], gstreams[g], out_sets[i % R] if own else outs[g], flags, i)

    def calls(n):  # n steps spread over the groups' streams, forked from and joined back to `stream`
        for st in gstreams[1:]:
            st.wait_stream(stream)
        for i in range(n):
            call(i)
        for st in gstreams[1:]:
            stream.wait_stream(st)

    # the K timed steps as one CUDA graph (the calls advance the device counters on replay)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        calls(3 * S)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            calls(args.steps)
        warm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(warm, stream=stream):
            calls(max(args.warmup, 1))
    torch.cuda.synchronize()
    # untimed: bring clocks up, then exactly W warm-up steps
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 0.5
        while time.perf_counter() < t_end:
            warm.replay()
            stream.synchronize()
        warm.replay()
    stream.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    bus = getattr(props, "pci_bus_id", None)
    bus_str = None
    if bus is not None:
        bus_str = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus, getattr(props, "pci_device_id", 0))
    clk = ClockSampler(bus_str)
    with clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    if world > 1:
        dist.barrier()
    if any(sg.errors() != 0 for sg in samplers):
        raise RuntimeError("device error bits set after the timed region")
    per_launch_s = ms / 1e3 / args.steps
    value = job_rows_per_s(B * args.steps, world, ms / 1e3)

    # ---- one request group alone: its K calls chained on one stream with the library's launch
    # shape for that case (no concurrency hint), timed the same way and reported beside the value
    single = None
    if S > 1:
        flags1 = flags & ~(STRATA_FLAG_CONCURRENT | STRATA_FLAG_OWN_OUTPUTS)
        shape1 = s.shape(2 if verify else 0, 0, B, w["V"], w["top_n"], flags1)
        g1, warm1 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(3):
                call_on(s, stream, outs[0], flags1, i)
            stream.synchronize()
            with torch.cuda.graph(g1, stream=stream):
                for i in range(args.steps):
                    call_on(s, stream, outs[0], flags1, i)
            with torch.cuda.graph(warm1, stream=stream):
                for i in range(max(args.warmup, 1)):
                    call_on(s, stream, outs[0], flags1, i)
            warm1.replay()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            g1.replay()
            f1.record(stream)
        stream.synchronize()
        ms1 = max_over_ranks(f0.elapsed_time(f1), dev)
        if s.errors() != 0:
            raise RuntimeError("device error bits set in the single-group leg")
        single = {"value": job_rows_per_s(B * args.steps, world, ms1 / 1e3), "ms_per_step": ms1 / args.steps,
                  "split": shape1["split"], "smem_bytes": shape1["smem"], "grid": shape1["grid"]}

    # ---- e2e through the C ABI from pinned host buffers -------------------------------------
    # Every step copies its inputs in (the logits, plus the small arrays packed into one copy) and
    # its results out (packed into one copy).  Copies run on their own streams into and out of two
    # buffer sets, so step k+1's inputs travel while step k samples; the calls stay in order on
    # one stream (a context serves one stream at a time).
    K_e2e = max(3, min(args.steps, 200))
    small_keys = ("row_slot", "row_pos") + (() if ring else ("hist", "hist_off")) + \
        (() if verify else ("allowed", "allowed_off"))
    small_np = {k: np.ascontiguousarray(w[k]) for k in small_keys}
    if verify:
        small_np["row_draft"] = drafts

    def pack_layout(items):
        offs, o = {}, 0
        for k, (nbytes, dt, shp) in items.items():
            offs[k] = (o, nbytes, dt, shp)
            o = (o + nbytes + 15) // 16 * 16
        return offs, max(o, 16)

    in_offs, in_bytes = pack_layout({k: (a.nbytes, torch.from_numpy(a[:0]).dtype, a.shape) for k, a in small_np.items()})
    h_logits = torch.from_numpy(w["logits"]).pin_memory()
    h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    for k, (o, n, _dt, _shp) in in_offs.items():
        h_in[o:o + n].copy_(torch.from_numpy(small_np[k].reshape(-1).view(np.uint8)))
    out_items = {k: (v.numel() * v.element_size(), v.dtype, tuple(v.shape)) for k, v in out.items()}
    out_offs, out_bytes = pack_layout(out_items)

    def views(buf, offs):
        return {k: buf[o:o + n].view(dt).view(shp) for k, (o, n, dt, shp) in offs.items()}

    sets = []
    for _ in range(2):
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        d_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        sets.append(dict(logits=torch.empty_like(batches[0]), d_in=d_in, small=views(d_in, in_offs), d_out=d_out,
                         out=views(d_out, out_offs), h_out=torch.empty(out_bytes, dtype=torch.uint8).pin_memory(),
                         ev_in=torch.cuda.Event(), ev_call=torch.cuda.Event(), ev_out=torch.cuda.Event()))
    h2d = int(h_logits.numel() * h_logits.element_size() + in_bytes)
    d2h = int(out_bytes)
    copy_in = torch.cuda.Stream(device=dev)
    copy_out = torch.cuda.Stream(device=dev)

    # the e2e inputs are copied in right before each call, so those calls do not claim early loads
    flags_e2e = flags & ~(STRATA_FLAG_EARLY_LOAD | STRATA_FLAG_CONCURRENT | STRATA_FLAG_OWN_OUTPUTS)

    def e2e_step(k):
        st_ = sets[k % 2]
        if k >= 2:
            copy_in.wait_event(st_["ev_call"])   # the call two steps back has read this set
        with torch.cuda.stream(copy_in):
            st_["logits"].copy_(h_logits, non_blocking=True)
            st_["d_in"].copy_(h_in, non_blocking=True)
            st_["ev_in"].record(copy_in)
        stream.wait_event(st_["ev_in"])
        if k >= 2:
            stream.wait_event(st_["ev_out"])     # its results from two steps back have left
        d_small, o_ = st_["small"], st_["out"]
        if verify:
            s.verify(st_["logits"], d_small["row_slot"], d_small["row_pos"], d_small["row_draft"],
                     hist=d_small.get("hist"), hist_off=d_small.get("hist_off"), flags=flags_e2e, stream=stream,
                     out=o_)
        else:
            s.sample(st_["logits"], d_small["row_slot"], d_small["row_pos"], hist=d_small["hist"],
                     hist_off=d_small["hist_off"], top_n=w["top_n"], chosen_lp=True, allowed=d_small["allowed"],
                     allowed_off=d_small["allowed_off"], flags=flags_e2e, stream=stream, out=o_)
        st_["ev_call"].record(stream)
        copy_out.wait_event(st_["ev_call"])
        with torch.cuda.stream(copy_out):
            st_["h_out"].copy_(st_["d_out"], non_blocking=True)
            st_["ev_out"].record(copy_out)

    for k in range(4):
        e2e_step(k)
    torch.cuda.synchronize()
    # the K steps (copies, cross-stream events and calls) as one CUDA graph, like the timed calls
    # above, so that the host's per-step Python does not set the pace
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        copy_in.wait_stream(stream)
        copy_out.wait_stream(stream)
        for k in range(K_e2e):
            e2e_step(k)
        stream.wait_stream(copy_in)
        stream.wait_stream(copy_out)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a0.record(stream)
        e2e_graph.replay()
        a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a0.elapsed_time(a1), dev)
    e2e_value = job_rows_per_s(B * K_e2e, world, e2e_ms / 1e3)

    if rank != 0:
        for sg in samplers:
            sg.close()
        return
    alg = algorithmic_bytes_verify(w, ring) if verify else algorithmic_bytes(w)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peak, peak_src = float(json.load(open(peaks_path))["hbm_gbs"]), "measured"
    else:
        peak, peak_src = 6800.0, "fallback"
    achieved = alg / per_launch_s / 1e9
    if single is not None:
        single["roofline_frac"] = alg / (single["ms_per_step"] / 1e3) / 1e9 / peak
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        tj = json.load(open(TRAFFIC_FILE))
        if tj.get("kernel_hash") == kernel_hash() and args.workload == "fused":
            traffic = tj.get("dram_bytes_per_launch")
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        if verify:
            rps, nwin, el = oracle_windows_per_s(w, drafts.tolist(), budget_s=args.cpu_budget, ring=ring)
            cpu = {"value": rps, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{nwin} whole 5-row windows (sample + acceptance"
                             + (" + history update" if ring else "") + f"), {el:.1f} s on 1 host core"}
        else:
            rps, nrows, el = oracle_rows_per_s(w, budget_s=args.cpu_budget, mask=args.workload == "mask")
            cpu = {"value": rps, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{nrows} rows of the same 8-row workload (fused sample + logprobs + allowed), "
                             f"{el:.1f} s on 1 host core"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": {"verify": WORKLOAD_VERIFY, "mask": WORKLOAD_MASK,
                                "verify-ring": WORKLOAD_VERIFY_RING}.get(args.workload, WORKLOAD),
                   "rows_per_step": B, "V": w["V"],
                   "logits_dtype": "f32",
                   "l2_policy": f"inputs rotate over {R} distinct batches ({R * step_bytes / 1e6:.0f} MB, "
                                f"{R * step_bytes / l2:.1f}x the {l2 / 1e6:.0f} MB L2)",
                   "launch": "one CUDA graph of the K calls" + (", programmatic dependent launch" if flags & 1 else "")
                             + (", logit loads start before the previous call ends (inputs resident)"
                                if flags & 2 else "")
                             + (", each call writes its own output set (no wait for the previous call)"
                                if flags & STRATA_FLAG_OWN_OUTPUTS else ""),
                   "split": shape["split"], "chunk_elems": shape["chunk"], "smem_bytes": shape["smem"],
                   "grid": shape["grid"], "parallelism": f"replicas x{world}",
                   "streams": S},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": alg, "launch_us": per_launch_s * 1e6},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": K_e2e},
        "single_group": single,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    for sg in samplers:
        sg.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-early-load", action="store_true",
                    help="with PDL, wait for the previous kernel before loading logits (inputs produced by it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--split", type=int, default=0,
                    help="blocks per row (1..16; 0: the library's choice), for launch-shape sweeps")
    ap.add_argument("--no-own-outputs", action="store_true",
                    help="every call of a group writes the same output buffers, so each call waits for the "
                         "previous one before its counters and writes")
    ap.add_argument("--streams", type=int, default=8,
                    help="independent request groups, each its own context, slots and stream; the steps "
                         "alternate over them and the groups' calls overlap")
    ap.add_argument("--batches", type=int, default=0,
                    help="distinct input batches to rotate over (0: enough for 4x the L2 size)")
    ap.add_argument("--workload", choices=["fused", "verify", "mask", "verify-ring"], default="fused",
                    help="fused: the logprobs workload fused with sampling (the headline); verify: verify "
                         "windows; mask: the fused workload with its allowed ids as a sampling mask; "
                         "verify-ring: verify windows over histories kept on the device")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_gpu(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
