"""Throughput of the fused decode-time sampler on GB300.

One step = one strata_sample_rows call over one batch.  The default workload (`--workload fused`)
is the logprobs workload: 8 fp32 rows, V=248,320, N(0,3^2) logits with 1-5 spikes.  Every row is
a sampled request with the single-row request's keys: penalties over a 64-token history, top_k 20,
min_p 0.05, top_p 0.95, T 0.8 and a Philox draw.  It is fused with top_logprobs=20, the sampled
token's log-probability and allowed_token_ids subsets of 5, 100 and 1000 ids, so one launch runs
every step of the hot path.  The other workloads are `config1` (one fp32 row, V=32,000),
`config3` (8 bf16 batch slots, half greedy), `config5` (64 bf16 rows, top_k 64, 2048-id Zipf
histories, top_logprobs 20), `verify` (config 2's five-row verify windows), `verify-ring` (the same
windows over histories kept on the device) and `mask` (the default step with its allowed ids as a
sampling mask).

  value      rows/s over exactly K timed steps: one CUDA graph holding the K calls, replayed once.
             The steps alternate over S independent request groups (`--streams`).  Each group is its
             own context (own slots and counters) with its own stream.  A group's calls are chained
             in order; the groups' calls overlap.  Sampling calls write output set i of a rotation
             (`STRATA_FLAG_OWN_OUTPUTS`), so no call waits for the previous one.
  timing     CUDA events on the launching stream.  Right before the start event the stream writes
             a buffer several times the L2 size (the gate).  The write evicts every input from L2,
             and the host submits the timed graph while the GPU is still writing.  So neither L2
             hits nor the host's submission time fall inside the timed region.  Inputs rotate over
             enough distinct batches to exceed 4x the L2 size.  The timed steps start at the batch
             after the last warm-up step, so no timed batch was touched by the warm-up.
  single_group  the same K steps as one group alone (one stream, the library's pipelined launch
             shape): each call waits for the previous call before its counters and writes.
  single_call_us  one call alone (no programmatic dependent launch, inputs not in L2), the
             library's latency launch shape: the median over repeated gated calls.
  e2e        the same metric through the C ABI from pinned host buffers.  Every step copies its
             inputs host->device (the logits, plus the small arrays packed into one copy), runs the
             call and copies every output back (one packed copy).  Copies run on their own streams
             into two buffer sets, so one step's inputs travel while the previous step samples.
             The calls stay in order on one stream; the K steps are one CUDA graph.
  roofline   algorithmic bytes per launch / average launch time, against the measured HBM copy
             bandwidth.  `traffic` is the DRAM bytes per launch from the committed ncu summary,
             only when the kernel source still matches it.
  cpu_baseline  the CPU oracle (plain numpy) on whole batches of the same workload: rows spread
             over min(B, nproc) processes, and one core beside it.  The same leg compares the
             oracle's first batch with one GPU call on the same inputs and counters (`parity`).

`--impl reference` times the CPU oracle alone on the same workload (whole batches, one core).
Multi-GPU (torchrun): every rank runs its own batch stream (weak scaling, no collective on the data
path); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
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
_KEYS1 = ("per-row keys top_k=20 T=0.8 top_p=0.95 min_p=0.05 repeat=1.1 freq=0.1 presence=0.1 "
          "penalty_last_n=64")
DESCRIPTIONS = {
    "fused": ("logprobs workload fused with sampling: B=8 fp32 rows x V=248,320, N(0,3^2)+1..5 spikes; "
              + _KEYS1 + "; top_logprobs=20, chosen-token logprob, allowed_token_ids of 5/100/1000"),
    "config1": ("single row: B=1 fp32 row x V=32,000, N(0,2^2) + 3 spikes at +12; top_k=20 T=0.8 top_p=0.95 "
                "min_p=0.05 repeat=1.1 freq=0.1 presence=0.1 over a 64-id history; top_logprobs=5"),
    "config3": ("batch slots: B=8 bf16 rows x V=248,320, N(0,3^2)+1..5 spikes; slots 0-3 greedy (neutral, no "
                "history), slots 4-7 sampled with seeded keys (top_k 1..64, T 0.3..1.5, top_p 0.5..1, "
                "min_p 0..0.2, penalties over up to 256 history ids)"),
    "config5": ("stress: B=64 bf16 rows (8 slots x 8-token windows) x V=248,320, N(0,3^2)+1..5 spikes (bf16 "
                "ties); top_k=64 repeat=1.3 freq=0.5 presence=0.5 T=1 top_p=0.98 min_p=0.01 over 2048-id "
                "Zipf(1.1) histories; top_logprobs=20 on every row"),
    "verify": ("verify windows (strata_sample_verify): config 2's 5-row windows (4 drafts + head), 1 slot, "
               "fp32 V=248,320, N(0,3^2)+1..5 spikes; keys T=0.7 top_k=20 top_p=0.9 min_p=0.05 repeat=1.1 "
               "over a 64-token history; seeded draft ids; kept rows counted in the launch"),
}
DESCRIPTIONS["mask"] = DESCRIPTIONS["fused"] + "; the allowed ids used as a sampling mask (STRATA_FLAG_ALLOWED_MASK)"
DESCRIPTIONS["sliced"] = ("vocabulary slices: B=8 fp32 rows x V=248,320, N(0,3^2)+1..5 spikes; " + _KEYS1
                          + "; top_logprobs=20, chosen-token logprob (no allowed subsets); each row split into "
                          "{G} equal column slices reduced to records (strata_shard_rows, one launch per slice, "
                          "one after another on one GPU) and merged (strata_merge_shards)")
DESCRIPTIONS["verify-ring"] = (DESCRIPTIONS["verify"] + "; the 64-token window read from the slot's history kept on "
                               "the device (STRATA_FLAG_HISTORY_RING) and the kept picks appended in the launch")
KERNEL_SOURCES = ("request_token_sampling_gb300/csrc/strata_kernel.cuh",   # the device code the
                  "request_token_sampling_gb300/csrc/strata_device.cuh")   # ncu counters describe
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_config4_fused.json")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_workload(name: str):
    """(workload dict, kind) for a --workload name; kind is "sample" or "verify"."""
    if name in ("fused", "mask"):
        return synth.config4(fused=True), "sample"
    if name == "config1":
        return synth.config1(), "sample"
    if name == "config3":
        return synth.config3(), "sample"
    if name == "config5":
        return synth.config5(), "sample"
    if name in ("verify", "verify-ring"):
        return synth.config2_window(0), "verify"
    if name == "sliced":  # sliced rows carry no allowed subsets
        return dict(synth.config4(fused=True), allowed=None, allowed_off=None), "sample"
    raise SystemExit(f"unknown workload {name}")


def esize(w) -> int:
    return 4 if w["dtype"] == "f32" else 2


def algorithmic_bytes(w, kind="sample", ring=False, slices=0) -> int:
    """Bytes a launch must move at least: logits once, the history windows, allowed ids, row
    arrays, slot keys and counters, and every output (verify windows: drafts and the kept count;
    with a kept history its length read and written and the kept picks written, counted as the
    whole window; vocabulary slices: every slice's records written and read once)."""
    B, V = w["B"], w["V"]
    n = B * V * esize(w) + 2 * slices * B * 1280
    for s in range(w["n_hist_slots"]):
        ln = w["slot_params"][s]["penalty_last_n"]
        n += 4 * min(ln, int(w["hist_off"][s + 1] - w["hist_off"][s]))
    if w["n_hist_slots"]:
        n += 4 * (w["n_hist_slots"] + 1)                                      # history offsets
    n_allowed = int(w["allowed_off"][-1]) if w.get("allowed_off") is not None else 0
    if w.get("allowed_off") is not None:
        n += 4 * n_allowed + 4 * (B + 1)                                      # allowed ids, offsets
    n += B * (4 + 8)                                                          # row slot + position
    n += len(w["slot_params"]) * (48 + 8)                                     # slot keys, counter
    n += B * 4                                                                # picks
    if kind == "verify":
        n += B * 4 + 4 * len(w["slot_params"])                                # drafts, kept counts
        if ring:
            n += 16 + 4 * B
    else:
        n += B * (4 + w["top_n"] * 8) + 4 * n_allowed                         # chosen lp, top-N, allowed lps
    return n


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
            self.samples.append(self._read())
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


# ------------------------------------------------------------------------------ CPU oracle (baseline leg)
def slice_rows(w, rows):
    """The workload restricted to `rows` (the slots, histories and counters stay whole)."""
    rows = list(rows)
    wb = dict(w)
    wb["B"] = len(rows)
    wb["logits"] = np.ascontiguousarray(w["logits"][rows])
    wb["row_slot"] = w["row_slot"][rows]
    wb["row_pos"] = w["row_pos"][rows]
    if w.get("allowed_off") is not None:
        off = w["allowed_off"]
        parts = [w["allowed"][off[b]:off[b + 1]] for b in rows]
        wb["allowed"] = np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
        wb["allowed_off"] = np.concatenate([[0], np.cumsum([p.size for p in parts])]).astype(np.int32)
    return wb


def oracle_batch(w, kind, mask=False, ring_state=None, drafts=None):
    """One whole call of the oracle on workload `w` (what one GPU step computes)."""
    import oracle
    if kind == "verify":
        if ring_state is not None:
            rows, _, _, keep = oracle.history_call(w, ring_state, row_draft=drafts)
        else:
            rows, _, keep = oracle.verify_call(w, drafts)
        return rows, keep
    rows, _ = oracle.sample_call(w, mask_allowed=mask)
    return rows, None


_POOL_W = None


def _pool_init(w, kind, mask):
    global _POOL_W
    _POOL_W = (w, kind, mask)


def _pool_rows(rows):
    w, kind, mask = _POOL_W
    t0 = time.perf_counter()
    oracle_batch(slice_rows(w, rows), kind, mask)
    return time.perf_counter() - t0


def cpu_baseline_leg(w, kind, mask, drafts, budget_s, ring_state=None):
    """The oracle, as it stands, on whole batches of the workload: one core in this process
    (the first batch's rows are kept for the parity check), then the rows spread over
    min(B, nproc) spawned processes.  Returns (summary, first batch rows, kept counts)."""
    B = w["B"]
    t0 = time.perf_counter()
    first, keep = oracle_batch(w, kind, mask, ring_state, drafts)
    n1 = 1
    while time.perf_counter() - t0 < budget_s / 2 and n1 < 50:
        oracle_batch(w, kind, mask, ring_state, drafts)
        n1 += 1
    el1 = time.perf_counter() - t0
    one = {"value": n1 * B / el1, "unit": UNIT, "cores": 1,
           "sample": f"{n1} whole {B}-row calls, {el1:.1f} s on 1 host core"}
    nproc = os.cpu_count() or 1
    P = max(1, min(B, nproc))
    multi = None
    if P > 1 and kind == "sample":
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        groups = [list(range(i, B, P)) for i in range(P)]
        with ctx.Pool(P, initializer=_pool_init, initargs=(w, kind, mask)) as pool:
            pool.map(_pool_rows, groups)                         # workers import numpy and the oracle
            rounds = max(1, int(math.ceil((budget_s / 2) / max(1e-3, el1 / n1 / P * 1.0))))
            rounds = min(rounds, 50)
            t1 = time.perf_counter()
            for _ in range(rounds):
                pool.map(_pool_rows, groups)
            el = time.perf_counter() - t1
        multi = {"value": rounds * B / el, "unit": UNIT, "cores": P,
                 "sample": f"{rounds} whole {B}-row calls, rows spread over {P} processes, {el:.1f} s"}
    head = multi if multi is not None else one
    out = {"value": head["value"], "unit": UNIT, "cores": head["cores"], "kind": "oracle",
           "sample": head["sample"], "nproc": nproc, "one_core": one}
    return out, first, keep


def parity_summary(w, kind, rows, g, keep=None):
    """The GPU call's outputs `g` against the oracle's rows under the parity rules: greedy ids and
    the top_k sequence bit-exact, sampled ids exact outside rows the oracle flags (a top_p or draw
    decision within 1e-6 of a boundary), log-probabilities within 1e-5."""
    import oracle
    V, dtype = w["V"], w["dtype"]
    st = dict(rows=0, greedy_rows=0, greedy_mismatch=0, topk_mismatch=0, sampled_mismatch=0, flagged=0,
              flagged_and_different=0, max_dlp=0.0, lp_over_tol=0)
    for b, r in enumerate(rows):
        st["rows"] += 1
        gid = int(g["ids"][b])
        if r.get("invalid"):
            st["sampled_mismatch"] += int(gid != -1)
            continue
        if "topk_ids" in g:
            k = r["topk_ids"].size
            if g["topk_ids"][b, :k].tolist() != r["topk_ids"].tolist():
                st["topk_mismatch"] += 1
        flagged = r["flag_top_p"] or r["flag_draw"]
        if r["greedy"]:
            st["greedy_rows"] += 1
            st["greedy_mismatch"] += int(gid != r["id"])
        elif flagged:
            st["flagged"] += 1
            st["flagged_and_different"] += int(gid != r["id"])
        else:
            st["sampled_mismatch"] += int(gid != r["id"])
        raw = oracle.widen(w["logits"][b, :V], dtype)
        d = []
        if "chosen_lp" in g and gid >= 0:
            d.append(abs(float(g["chosen_lp"][b]) - float(oracle.log_softmax(raw)[gid])))
        if "top_ids" in g and w["top_n"]:
            if g["top_ids"][b].tolist() != r["top_ids"].tolist():
                st["topk_mismatch"] += 1
            a, e = np.asarray(g["top_lps"][b], np.float64), np.asarray(r["top_lps"], np.float64)
            fin = np.isfinite(e)
            d.extend(np.abs(a[fin] - e[fin]).tolist())
        if "allowed_lps" in g and w.get("allowed_off") is not None and "allowed_lps" in r:
            off = w["allowed_off"]
            a, e = np.asarray(g["allowed_lps"][off[b]:off[b + 1]], np.float64), np.asarray(r["allowed_lps"])
            d.extend(np.abs(a - e).tolist())
        if d:
            m = max(d)
            st["max_dlp"] = max(st["max_dlp"], m)
            st["lp_over_tol"] += int(m > 1e-5)
    if keep is not None and "keep" in g:
        st["keep_mismatch"] = int(sum(int(g["keep"][s]) != int(n) for s, n in keep.items()))
    return st


def run_reference(args, rank, world):
    if rank != 0:
        return
    w, kind = load_workload(args.workload)
    drafts = verify_drafts(w) if kind == "verify" else None
    mask = args.workload == "mask"
    ring_state = {0: [int(x) for x in w["hist"]]} if args.workload == "verify-ring" else None
    for _ in range(args.warmup):
        oracle_batch(w, kind, mask, ring_state, drafts)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_batch(w, kind, mask, ring_state, drafts)
    el = time.perf_counter() - t0
    v = args.steps * w["B"] / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32(penalty,ranking)+f64",
            "data": "synthetic", "config": {"workload": DESCRIPTIONS[args.workload].replace("{G}", str(args.slices)),
                                            "rows_per_step": w["B"], "V": w["V"], "logits_dtype": w["dtype"]},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} timed whole {w['B']}-row calls on 1 host core"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def verify_drafts(w):
    d = np.random.default_rng(0x5EED0002).integers(0, w["V"], size=w["B"]).astype(np.int32)
    d[-1] = -1
    return d


# ------------------------------------------------------------------------------ GPU arm
def make_batches(w, R, dev):
    """R distinct device batches with the workload's recipe (batch 0 is the workload itself)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(0x5EED0004)
    first = np.ascontiguousarray(w["logits"])
    if first.dtype == np.uint16:
        first = first.view(np.int16)
    out = [torch.from_numpy(first).to(dev)]
    B, V, ld = w["B"], w["V"], w["ld"]
    sigma = 2.0 if w["V"] < 100_000 else 3.0
    for _ in range(R - 1):
        x = torch.full((B, ld), -7.0, device=dev)
        x[:, :V] = torch.randn((B, V), generator=g, device=dev) * sigma
        n = torch.randint(1, 6, (B,), generator=g, device=dev).tolist()
        for b in range(B):
            ids = torch.randint(0, V, (n[b],), generator=g, device=dev)
            x[b, ids] = torch.rand((n[b],), generator=g, device=dev) * 7.0 + 8.0
        if w["dtype"] == "bf16":
            x = x.to(torch.bfloat16).view(torch.int16)
        out.append(x.contiguous())
    return out


class Gate:
    """A write of a buffer several times the L2 size, enqueued right before a start event: it
    evicts the inputs from L2, and the host submits the timed work while the GPU is still writing.
    Its length grows until it covers twice the host's submission time of what it guards."""

    def __init__(self, dev, l2, stream):
        import torch
        self.torch = torch
        self.stream = stream
        self.unit = torch.empty(max(4 * l2, 64 << 20) // 4, dtype=torch.float32, device=dev)
        self.reps = 1
        self.n = 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            self.unit.fill_(0.0)
            e0.record(stream)
            self.unit.fill_(1.0)
            e1.record(stream)
        stream.synchronize()
        self.unit_us = e0.elapsed_time(e1) * 1e3

    def cover(self, submit_us: float):
        self.reps = max(self.reps, int(math.ceil(2.0 * submit_us / max(self.unit_us, 1.0))))

    def time(self, fn, retry=True):
        """(device ms between the events around fn, host us spent submitting fn).  When the
        submission outlasted the gate, the gate grows and the measurement is taken again."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            for _ in range(self.reps):
                self.n += 1
                self.unit.fill_(float(self.n % 7))
            e0.record(self.stream)
            t0 = time.perf_counter()
            fn()
            host_us = (time.perf_counter() - t0) * 1e6
            e1.record(self.stream)
        self.stream.synchronize()
        if retry and host_us > 0.8 * self.reps * self.unit_us:
            self.cover(host_us)
            return self.time(fn, retry=False)
        return e0.elapsed_time(e1), host_us

    def describe(self):
        return (f"{self.reps} x {self.unit.numel() * 4 / 1e6:.0f} MB write ({self.reps * self.unit_us:.0f} us) "
                f"before the start event")


def run_gpu(args, rank, world):
    import torch
    import torch.distributed as dist
    from request_token_sampling_gb300 import (STRATA_FLAG_ALLOWED_MASK, STRATA_FLAG_CONCURRENT, STRATA_FLAG_EARLY_LOAD,
                                              STRATA_FLAG_HISTORY_RING, STRATA_FLAG_OWN_OUTPUTS, STRATA_FLAG_PDL,
                                              STRATA_FLAG_SPLIT, STRATA_SHARD_RECORD_BYTES, Sampler)

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    w, kind = load_workload(args.workload)
    verify = kind == "verify"
    ring = args.workload == "verify-ring"
    sliced = args.workload == "sliced"
    G = max(1, args.slices) if sliced else 0
    B, V = w["B"], w["V"]
    dtype_code = 0 if w["dtype"] == "f32" else 1
    step_bytes = B * w["ld"] * esize(w)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    R = max(2, -(-4 * l2 // step_bytes)) if args.batches <= 0 else args.batches
    W, K = args.warmup, args.steps
    flags = 0 if args.no_pdl else (STRATA_FLAG_PDL | (0 if args.no_early_load else STRATA_FLAG_EARLY_LOAD))
    if sliced:  # a slice call takes only the launch-shape flags
        flags = 0
    if args.workload == "mask":
        flags |= STRATA_FLAG_ALLOWED_MASK
    if ring:
        flags |= STRATA_FLAG_HISTORY_RING
    if args.split > 0:
        flags |= STRATA_FLAG_SPLIT(args.split)
    elif args.streams > 1 and not args.no_concurrent_hint:  # other groups' calls run alongside
        flags |= STRATA_FLAG_CONCURRENT
    # every call writes its own output buffers (they rotate like the inputs), so no call waits for
    # the one before it; verify windows and kept histories depend on the previous call by nature
    own = (not args.no_own_outputs and (flags & STRATA_FLAG_EARLY_LOAD) != 0 and not verify and not ring
           and not sliced)
    if own:
        flags |= STRATA_FLAG_OWN_OUTPUTS

    # S independent request groups: a context each (its own slots, counters and outputs), a stream
    # each; one group's calls are ordered, the groups' calls overlap
    S = max(1, args.streams)
    n_slots = max(16, len(w["slot_params"]))
    samplers = []
    for _ in range(S):
        sg = Sampler(device=local, max_slots=n_slots, max_vocab=V, max_rows=B)
        for slot, p in w["slot_params"].items():
            sg.restore_slot(slot, p, int(w["counters"].get(slot, 0)))
        samplers.append(sg)
    s = samplers[0]
    ten = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    row_slot, row_pos = ten(w["row_slot"]), ten(w["row_pos"])
    has_hist = w["hist"] is not None and w["hist"].size > 0
    hist = ten(w["hist"]) if has_hist else None
    hist_off = ten(w["hist_off"]) if has_hist else None
    if ring:  # the window lives in the slot's kept history; the call uploads none
        for sg in samplers:
            sg.history_enable()
            sg.history_set(0, w["hist"])
        hist = hist_off = None
    allowed = allowed_off = None
    if w.get("allowed_off") is not None:
        allowed, allowed_off = ten(w["allowed"]), ten(w["allowed_off"])
    drafts = verify_drafts(w)
    row_draft = ten(drafts)
    top_n = w["top_n"]
    batches = make_batches(w, R, dev)
    # vocabulary slices: G equal column ranges (multiples of 8 ids, so every slice starts on a
    # 16-byte boundary) and one record buffer per group
    bounds = [min(V, (V * g // max(G, 1) + 7) // 8 * 8) for g in range(G + 1)] if sliced else []
    recbufs = [torch.empty(G, B, STRATA_SHARD_RECORD_BYTES, dtype=torch.uint8, device=dev) for _ in samplers] \
        if sliced else []

    def sliced_call(sg, x, rs, rp, h, ho, st, o, fl, debug=False):
        rec = recbufs[samplers.index(sg)]
        for g in range(G):
            a, b = bounds[g], bounds[g + 1]
            sg.shard(x[:, a:b], rs, a, V=b - a, hist=h, hist_off=ho, top_n=top_n, flags=fl, stream=st, out=rec[g])
        return sg.merge(rec, rs, rp, top_n=top_n, chosen_lp=True, debug=debug, stream=st, out=o)

    def call_on(sg, st, o, fl, i, debug=False):
        x = batches[i % R]
        if sliced:
            return sliced_call(sg, x, row_slot, row_pos, hist, hist_off, st, o, fl, debug)
        if verify:
            return sg.verify(x, row_slot, row_pos, row_draft, V=V, hist=hist, hist_off=hist_off, top_n=top_n,
                             chosen_lp=True, flags=fl, stream=st, out=o)
        return sg.sample(x, row_slot, row_pos, V=V, hist=hist, hist_off=hist_off, top_n=top_n, chosen_lp=True,
                         allowed=allowed, allowed_off=allowed_off, flags=fl, stream=st, out=o, debug=debug)

    outs = [call_on(sg, None, None, flags, 0) for sg in samplers]
    out = outs[0]
    # with own outputs, call i writes output set i % R: more sets than calls can be resident at once
    out_sets = [{k: torch.empty_like(v) for k, v in out.items()} for _ in range(R)] if own else None
    torch.cuda.synchronize()
    if any(sg.errors() != 0 for sg in samplers):
        raise RuntimeError("device error bits set")
    shape = s.shape(2 if verify else 0, dtype_code, B, bounds[1] if sliced else V, top_n, flags)

    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    gstreams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(S - 1)]
    gate = Gate(dev, l2, stream)

    def calls(n, start):  # n steps from batch `start` on, spread over the groups' streams
        for st in gstreams[1:]:
            st.wait_stream(stream)
        for i in range(n):
            j = start + i
            g = i % S
            call_on(samplers[g], gstreams[g], out_sets[j % R] if own else outs[g], flags, j)
        for st in gstreams[1:]:
            stream.wait_stream(st)

    # the W warm-up steps and the K timed steps as two CUDA graphs (the calls advance the device
    # counters on replay); the timed steps take the batches after the warm-up's
    graph, warm = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        calls(3 * S, R - (3 * S) % R)
        torch.cuda.synchronize()
        with torch.cuda.graph(warm, stream=stream):
            calls(W, 0)
        with torch.cuda.graph(graph, stream=stream):
            calls(K, W)
    torch.cuda.synchronize()
    # untimed: bring clocks up, size the gate to the host's submission time, then W warm-up steps
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 0.5
        while time.perf_counter() < t_end:
            warm.replay()
            stream.synchronize()
        t0 = time.perf_counter()
        graph.replay()
        gate.cover((time.perf_counter() - t0) * 1e6)
        stream.synchronize()
        warm.replay()
    stream.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    bus = getattr(props, "pci_bus_id", None)
    bus_str = None
    if bus is not None:
        bus_str = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus, getattr(props, "pci_device_id", 0))
    clk = ClockSampler(bus_str)
    with clk:
        ms, submit_us = gate.time(graph.replay)
    torch.cuda.synchronize()
    ms = max_over_ranks(ms, dev)
    if world > 1:
        dist.barrier()
    if any(sg.errors() != 0 for sg in samplers):
        raise RuntimeError("device error bits set after the timed region")
    per_launch_s = ms / 1e3 / K
    value = job_rows_per_s(B * K, world, ms / 1e3)

    # ---- one request group alone: its K calls chained on one stream with the library's launch
    # shape for that case (no concurrency hint), timed the same way and reported beside the value
    single = None
    if S > 1:
        flags1 = flags & ~(STRATA_FLAG_CONCURRENT | STRATA_FLAG_OWN_OUTPUTS)
        shape1 = s.shape(2 if verify else 0, dtype_code, B, V, top_n, flags1)
        g1, warm1 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(3):
                call_on(s, stream, outs[0], flags1, i)
            stream.synchronize()
            with torch.cuda.graph(warm1, stream=stream):
                for i in range(W):
                    call_on(s, stream, outs[0], flags1, i)
            with torch.cuda.graph(g1, stream=stream):
                for i in range(K):
                    call_on(s, stream, outs[0], flags1, W + i)
            warm1.replay()
        stream.synchronize()
        ms1, _ = gate.time(g1.replay)
        ms1 = max_over_ranks(ms1, dev)
        if s.errors() != 0:
            raise RuntimeError("device error bits set in the single-group leg")
        single = {"value": job_rows_per_s(B * K, world, ms1 / 1e3), "ms_per_step": ms1 / K,
                  "split": shape1["split"], "smem_bytes": shape1["smem"], "grid": shape1["grid"]}

    # ---- one call alone: no programmatic dependent launch, inputs out of L2, the library's
    # latency shape; the median over repeated gated calls
    flags0 = flags & (STRATA_FLAG_ALLOWED_MASK | STRATA_FLAG_HISTORY_RING)
    shape0 = s.shape(2 if verify else 0, dtype_code, B, V, top_n, flags0)
    lone = []
    for i in range(args.lone_reps + 2):
        d_ms, _ = gate.time(lambda: call_on(s, stream, outs[0], flags0, W + K + i), retry=False)
        if i >= 2:
            lone.append(d_ms * 1e3)
    if s.errors() != 0:
        raise RuntimeError("device error bits set in the single-call leg")
    single_call = {"us": statistics.median(lone), "min_us": min(lone), "max_us": max(lone), "reps": len(lone),
                   "split": shape0["split"], "grid": shape0["grid"], "smem_bytes": shape0["smem"]}

    # ---- e2e through the C ABI from pinned host buffers -------------------------------------
    # Every step copies its inputs in (the logits, plus the small arrays packed into one copy) and
    # its results out (packed into one copy).  Copies run on their own streams into and out of two
    # buffer sets, so step k+1's inputs travel while step k samples; the calls stay in order on
    # one stream (a context serves one stream at a time).
    K_e2e = max(3, min(K, 200))
    small_keys = ["row_slot", "row_pos"]
    if has_hist and not ring:
        small_keys += ["hist", "hist_off"]
    if allowed is not None:
        small_keys += ["allowed", "allowed_off"]
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
    h_logits = batches[0].cpu().pin_memory()
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
        if sliced:
            sliced_call(s, st_["logits"], d_small["row_slot"], d_small["row_pos"], d_small.get("hist"),
                        d_small.get("hist_off"), stream, o_, flags_e2e)
        elif verify:
            s.verify(st_["logits"], d_small["row_slot"], d_small["row_pos"], d_small["row_draft"], V=V,
                     hist=d_small.get("hist"), hist_off=d_small.get("hist_off"), top_n=top_n, chosen_lp=True,
                     flags=flags_e2e, stream=stream, out=o_)
        else:
            s.sample(st_["logits"], d_small["row_slot"], d_small["row_pos"], V=V, hist=d_small.get("hist"),
                     hist_off=d_small.get("hist_off"), top_n=top_n, chosen_lp=True, allowed=d_small.get("allowed"),
                     allowed_off=d_small.get("allowed_off"), flags=flags_e2e, stream=stream, out=o_)
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
    e2e_ms, _ = gate.time(e2e_graph.replay)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e_value = job_rows_per_s(B * K_e2e, world, e2e_ms / 1e3)

    # ---- one GPU call on the workload's own batch at its stated counters, for the parity check
    # in the CPU-baseline leg (untimed)
    g_par = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        for slot, p in w["slot_params"].items():
            s.restore_slot(slot, p, int(w["counters"].get(slot, 0)), stream=stream)
        if ring:
            s.history_set(0, w["hist"], stream=stream)
        o = call_on(s, stream, None, flags0, 0, debug=not verify)
        stream.synchronize()
        g_par = {k: v.cpu().numpy() for k, v in o.items()}
        if s.errors() != 0:
            raise RuntimeError("device error bits set in the parity call")

    if rank != 0:
        for sg in samplers:
            sg.close()
        return
    alg = algorithmic_bytes(w, kind, ring, G)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peak, peak_src = float(json.load(open(peaks_path))["hbm_gbs"]), "measured"
    else:
        peak, peak_src = 6800.0, "fallback"
    achieved = alg / per_launch_s / 1e9
    if single is not None:
        single["roofline_frac"] = alg / (single["ms_per_step"] / 1e3) / 1e9 / peak
    single_call["roofline_frac"] = alg / (single_call["us"] / 1e6) / 1e9 / peak
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        tj = json.load(open(TRAFFIC_FILE))
        if tj.get("kernel_hash") == kernel_hash() and tj.get("workload") == args.workload:
            traffic = tj.get("dram_bytes_per_launch")
    cpu, parity = None, None
    if world == 1 and not args.no_cpu_baseline:
        ring_state = {0: [int(x) for x in w["hist"]]} if ring else None
        cpu, rows_o, keep_o = cpu_baseline_leg(w, kind, args.workload == "mask", drafts if verify else None,
                                               args.cpu_budget, ring_state)
        parity = parity_summary(w, kind, rows_o, g_par, keep_o)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.workload].replace("{G}", str(G)), "rows_per_step": B, "V": V,
                   "logits_dtype": w["dtype"],
                   "l2_policy": (f"inputs rotate over {R} distinct batches ({R * step_bytes / 1e6:.0f} MB, "
                                 f"{R * step_bytes / l2:.1f}x the {l2 / 1e6:.0f} MB L2); the timed steps take "
                                 f"batches {W}..{W + K - 1} (mod {R}), none of them the warm-up's 0..{W - 1}; "
                                 f"L2 flushed by the gate"),
                   "gate": gate.describe(), "graph_submit_us": submit_us,
                   "launch": "one CUDA graph of the K calls" + (", programmatic dependent launch" if flags & 1 else "")
                             + (", logit loads start before the previous call ends (inputs resident)"
                                if flags & 2 else "")
                             + (", each call writes its own output set (no wait for the previous call)"
                                if flags & STRATA_FLAG_OWN_OUTPUTS else "")
                             + (f"; a step is {G} slice launches and one merge launch" if sliced else ""),
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
        "single_call_us": single_call,
        "parity": parity,
        "gpu_launches": K * (G + 1) if sliced else K,
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
    ap.add_argument("--cpu-budget", type=float, default=16.0)
    ap.add_argument("--split", type=int, default=0,
                    help="blocks per row (1..16; 0: the library's choice), for launch-shape sweeps")
    ap.add_argument("--no-own-outputs", action="store_true",
                    help="every call of a group writes the same output buffers, so each call waits for the "
                         "previous one before its counters and writes")
    ap.add_argument("--no-concurrent-hint", action="store_true",
                    help="with several groups, leave the launch shape to the library's single-stream rule")
    ap.add_argument("--streams", type=int, default=8,
                    help="independent request groups, each its own context, slots and stream; the steps "
                         "alternate over them and the groups' calls overlap")
    ap.add_argument("--batches", type=int, default=0,
                    help="distinct input batches to rotate over (0: enough for 4x the L2 size)")
    ap.add_argument("--lone-reps", type=int, default=15, help="gated single calls timed for single_call_us")
    ap.add_argument("--slices", type=int, default=2, help="sliced workload: column slices per row (1..16)")
    ap.add_argument("--workload", choices=["fused", "config1", "config3", "config5", "verify", "mask",
                                           "verify-ring", "sliced"], default="fused",
                    help="fused: the logprobs workload fused with sampling (the headline); config1/3/5: those "
                         "workloads at their own shapes; verify: verify windows; mask: the fused workload with "
                         "its allowed ids as a sampling mask; verify-ring: verify windows over histories kept "
                         "on the device; sliced: the fused rows without allowed subsets over --slices "
                         "vocabulary slices, merged")
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
