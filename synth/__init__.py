"""Seeded synthetic inputs for the decode-time sampler.

This module is the only code shared by the two sides of every parity check:
the CPU oracle (``oracle/``) and the CUDA library (``request_token_sampling_gb300``)
both take their inputs from here.  It therefore holds *no* arithmetic of the
method itself: it draws logit rows, history windows, allowed-id subsets and
per-slot request parameters from numpy's PCG64 generator and returns plain
numpy arrays and dicts.  Nothing here penalises, ranks, cuts, softmaxes or
draws a token.

The five named workloads follow the five configurations the sampler is
specified on (vocabulary 32,000 or 248,320; fp32 or bf16 rows; one request's
verify window, batch slots, the logprobs path, and a tie-heavy stress batch).
Every quantity the specification leaves open is a choice of this module and is
listed in the design notes (spike placement, history streams, seeds, positions).

Logit rows are laid out as ``logits[B][ld]`` with ``ld >= V``; fp32 rows are
``float32`` arrays, bf16 rows are ``uint16`` arrays holding the bf16 bit
patterns (round-to-nearest-even from the fp32 draw).
"""
from __future__ import annotations

import numpy as np

V_SMALL = 32_000
V_FULL = 248_320

PARAM_FIELDS = (
    "temperature", "top_k", "top_p", "min_p",
    "penalty_repeat", "penalty_freq", "penalty_present", "penalty_last_n", "seed",
)


def make_params(temperature=0.0, top_k=0, top_p=1.0, min_p=0.0, penalty_repeat=1.0,
                penalty_freq=0.0, penalty_present=0.0, penalty_last_n=64, seed=0):
    """A request's sampling keys as a plain dict (values only, no defaults logic)."""
    return dict(temperature=float(temperature), top_k=int(top_k), top_p=float(top_p),
                min_p=float(min_p), penalty_repeat=float(penalty_repeat),
                penalty_freq=float(penalty_freq), penalty_present=float(penalty_present),
                penalty_last_n=int(penalty_last_n), seed=int(seed))


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the uint16 bit patterns.

    Input data preparation only: the stored rows of the bf16 workloads are these bits.
    """
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng(list(key))


def logit_rows(rng, B, V, sigma, spikes=(1, 5), spike_range=(8.0, 15.0), spike_value=None,
               ld=None, dtype="f32"):
    """B rows of N(0, sigma^2) logits with a few spikes overwritten at distinct seeded ids.

    Returns (rows, spike_ids) where rows is (B, ld) float32 (dtype "f32") or uint16 bf16 bits
    (dtype "bf16"); padding columns beyond V hold NaN-free garbage (-7.0) that no reader may use.
    """
    ld = V if ld is None else ld
    x = (rng.standard_normal((B, V)) * sigma).astype(np.float32)
    spike_ids = []
    for b in range(B):
        n = int(rng.integers(spikes[0], spikes[1] + 1))
        ids = rng.choice(V, size=n, replace=False)
        if spike_value is None:
            vals = rng.uniform(spike_range[0], spike_range[1], size=n).astype(np.float32)
        else:
            vals = np.full(n, spike_value, dtype=np.float32)
        x[b, ids] = vals
        spike_ids.append(ids.astype(np.int64))
    out = np.full((B, ld), -7.0, dtype=np.float32)
    out[:, :V] = x
    if dtype == "bf16":
        return to_bf16_bits(out), spike_ids
    return out, spike_ids


def zipf_ids(rng, n, V, s):
    """n ids drawn from a Zipf(s) law over ranks 1..V, ranks mapped through a seeded permutation."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    p = ranks ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    r = np.searchsorted(cdf, rng.random(n), side="right")
    r = np.minimum(r, V - 1)
    perm = rng.permutation(V)
    return perm[r].astype(np.int32)


def csr(lists):
    """Pack a list of int arrays as (flat int32, offsets int32[len+1])."""
    off = np.zeros(len(lists) + 1, dtype=np.int32)
    for i, a in enumerate(lists):
        off[i + 1] = off[i] + len(a)
    flat = np.concatenate([np.asarray(a, dtype=np.int32) for a in lists]) if lists else np.zeros(0, np.int32)
    if flat.size == 0:
        flat = np.zeros(0, dtype=np.int32)
    return flat.astype(np.int32), off


def _workload(name, dtype, V, logits, slot_params, row_slot, row_pos, hist_lists, top_n,
              allowed_lists=None, chosen=None, counters=None):
    hist, hist_off = csr(hist_lists)
    w = dict(name=name, dtype=dtype, B=int(logits.shape[0]), V=int(V), ld=int(logits.shape[1]),
             logits=logits, slot_params=slot_params, row_slot=np.asarray(row_slot, np.int32),
             row_pos=np.asarray(row_pos, np.int64), hist=hist, hist_off=hist_off,
             n_hist_slots=len(hist_lists), top_n=int(top_n),
             counters=dict(counters or {s: 0 for s in slot_params}))
    if allowed_lists is not None:
        w["allowed"], w["allowed_off"] = csr(allowed_lists)
    else:
        w["allowed"], w["allowed_off"] = None, None
    w["chosen"] = None if chosen is None else np.asarray(chosen, np.int32)
    return w


# ---------------------------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------------------------

def config1():
    """One row, V=32,000 fp32 ~N(0,2^2), three spikes at +12, one request's full chain, top_logprobs=5."""
    rng = _rng(0x5EED0001)
    V = V_SMALL
    logits, spikes = logit_rows(rng, 1, V, 2.0, spikes=(3, 3), spike_value=12.0)
    hist = rng.integers(0, V, size=64).astype(np.int32)
    hist[int(rng.integers(0, 64))] = spikes[0][0]          # one spike id is in the history
    p = make_params(temperature=0.8, top_k=20, top_p=0.95, min_p=0.05, penalty_repeat=1.1,
                    penalty_freq=0.1, penalty_present=0.1, penalty_last_n=64, seed=1234)
    return _workload("config1_single_row_v32000_f32", "f32", V, logits, {0: p}, [0], [0], [hist], 5)


CONFIG2_WINDOWS = 100


def config2_window(w, counter=None):
    """Window w (0..99) of one request's verify window: 5 rows (4 drafts + head), V=248,320 fp32."""
    V = V_FULL
    rng = _rng(0x5EED0002, w)
    logits, _ = logit_rows(rng, 5, V, 3.0, spikes=(1, 5))
    stream = _rng(0x5EED0002, 0xFFFF).integers(0, V, size=64 + CONFIG2_WINDOWS).astype(np.int32)
    hist = stream[w:w + 64]
    p = make_params(temperature=0.7, top_k=20, top_p=0.9, min_p=0.05, penalty_repeat=1.1,
                    penalty_last_n=64, seed=1234)
    pos = [100 + 5 * w + j for j in range(5)]
    c = {0: w if counter is None else counter}
    return _workload(f"config2_verify_window_w{w}", "f32", V, logits, {0: p}, [0] * 5, pos, [hist], 0,
                     counters=c)


def config3():
    """Eight batch slots, one bf16 row each, V=248,320: slots 0-3 greedy, 4-7 sampled with drawn params."""
    V = V_FULL
    rng = _rng(0x5EED0003)
    logits, _ = logit_rows(rng, 8, V, 3.0, spikes=(1, 5), dtype="bf16")
    prm, hists = {}, []
    for s in range(8):
        if s < 4:
            prm[s] = make_params(temperature=0.0, penalty_last_n=0)
            hists.append(np.zeros(0, np.int32))
        else:
            prm[s] = make_params(
                temperature=float(rng.uniform(0.3, 1.5)), top_k=int(rng.integers(1, 65)),
                top_p=float(rng.uniform(0.5, 1.0)), min_p=float(rng.uniform(0.0, 0.2)),
                penalty_repeat=float(rng.uniform(1.0, 1.5)), penalty_freq=float(rng.uniform(0.0, 0.5)),
                penalty_present=float(rng.uniform(0.0, 0.5)), penalty_last_n=int(rng.integers(0, 257)),
                seed=1000 + s)
            hists.append(rng.integers(0, V, size=256).astype(np.int32))
    return _workload("config3_batch_slots_s8_bf16", "bf16", V, logits, prm, list(range(8)),
                     [200 + 17 * s for s in range(8)], hists, 0)


def config4(fused=True):
    """Logprobs path: 8 fp32 rows, V=248,320, top_logprobs=20, allowed subsets of 5/100/1000 ids.

    With fused=True every row is also a sampled request (the single-row request's keys, one slot
    per row, seed 1234+row); with fused=False the chosen id of each row is given (its greedy argmax
    is not known to the generator, so the generator passes a seeded id instead).
    """
    V = V_FULL
    rng = _rng(0x5EED0004)
    logits, _ = logit_rows(rng, 8, V, 3.0, spikes=(1, 5))
    sizes = [5, 100, 1000]
    allowed = [rng.choice(V, size=sizes[b % 3], replace=False).astype(np.int32) for b in range(8)]
    hists = [rng.integers(0, V, size=64).astype(np.int32) for _ in range(8)]
    prm = {b: make_params(temperature=0.8, top_k=20, top_p=0.95, min_p=0.05, penalty_repeat=1.1,
                          penalty_freq=0.1, penalty_present=0.1, penalty_last_n=64, seed=1234 + b)
           for b in range(8)}
    chosen = None if fused else rng.integers(0, V, size=8).astype(np.int32)
    return _workload("config4_logprobs_b8_f32" + ("_fused" if fused else ""), "f32", V, logits, prm,
                     list(range(8)), list(range(8)), hists, 20, allowed_lists=allowed, chosen=chosen)


def config5():
    """Stress: 64 bf16 rows (8 slots x 8-token windows), top_k=64, 2048-id Zipf(1.1) histories."""
    V = V_FULL
    rng = _rng(0x5EED0005)
    logits, _ = logit_rows(rng, 64, V, 3.0, spikes=(1, 5), dtype="bf16")
    prm, hists = {}, []
    for s in range(8):
        prm[s] = make_params(temperature=1.0, top_k=64, top_p=0.98, min_p=0.01, penalty_repeat=1.3,
                             penalty_freq=0.5, penalty_present=0.5, penalty_last_n=2048, seed=5000 + s)
        hists.append(zipf_ids(rng, 2048, V, 1.1))
    row_slot = [b // 8 for b in range(64)]
    row_pos = [1000 * (b // 8) + (b % 8) for b in range(64)]
    return _workload("config5_stress_b64_bf16", "bf16", V, logits, prm, row_slot, row_pos, hists, 20)


# ---------------------------------------------------------------------------------------------
# Generic seeded cases for edge-case parity tests
# ---------------------------------------------------------------------------------------------

def random_case(seed, B, V, dtype="f32", ld=None, n_slots=None, sampled_frac=0.5, hist_len=64,
                top_n=5, allowed_sizes=None, ties=False, sigma=3.0, max_top_k=64):
    """A seeded batch with per-slot drawn params; `ties=True` quantises logits to a coarse grid."""
    rng = _rng(0xC0FFEE, seed)
    n_slots = B if n_slots is None else n_slots
    ld = V if ld is None else ld
    x = (rng.standard_normal((B, V)) * sigma).astype(np.float32)
    if ties:
        x = (np.round(x * 2.0) / 2.0).astype(np.float32)
        x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, -0.0, 0.0).astype(np.float32)
    rows = np.full((B, ld), -7.0, np.float32)
    rows[:, :V] = x
    logits = to_bf16_bits(rows) if dtype == "bf16" else rows
    prm, hists = {}, []
    for s in range(n_slots):
        if rng.random() < sampled_frac:
            prm[s] = make_params(
                temperature=float(rng.uniform(0.2, 2.0)), top_k=int(rng.integers(0, max_top_k + 1)),
                top_p=float(rng.choice([1.0, rng.uniform(0.3, 1.0)])),
                min_p=float(rng.choice([0.0, rng.uniform(0.0, 0.5)])),
                penalty_repeat=float(rng.choice([1.0, rng.uniform(0.5, 2.0)])),
                penalty_freq=float(rng.choice([0.0, rng.uniform(-0.5, 1.0)])),
                penalty_present=float(rng.choice([0.0, rng.uniform(-0.5, 1.0)])),
                penalty_last_n=int(rng.integers(0, hist_len + 8)), seed=int(rng.integers(0, 2**63)))
        else:
            prm[s] = make_params(temperature=float(rng.choice([0.0, -1.0])),
                                 penalty_repeat=float(rng.choice([1.0, 1.3])), penalty_last_n=hist_len,
                                 seed=int(rng.integers(0, 2**32)))
        n_h = int(rng.integers(0, hist_len + 1))
        h = rng.integers(-2, V + 2, size=n_h).astype(np.int32)       # a few out-of-range ids
        hists.append(h)
    row_slot = rng.integers(0, n_slots, size=B).astype(np.int32)
    row_pos = rng.integers(0, 2**40, size=B).astype(np.int64)
    allowed = None
    if allowed_sizes is not None:
        allowed = []
        for b in range(B):
            n = int(allowed_sizes[b % len(allowed_sizes)])
            a = rng.integers(0, V, size=n).astype(np.int32)       # duplicates allowed
            allowed.append(a)
    return _workload(f"random_case_{seed}", dtype, V, logits, prm, row_slot, row_pos, hists, top_n,
                     allowed_lists=allowed)


# ---------------------------------------------------------------------------------------------
# Decode runs: the same slots sampled step after step (for kept per-slot histories)
# ---------------------------------------------------------------------------------------------

class DecodeRun:
    """A seeded run of `steps` calls over `S` slots with penalties on, for histories kept between
    calls.  Each slot has its own keys, a prompt (its history before the first call) and a fixed
    set of `hot` ids that carry +5..+8 spikes in every row of the slot (redrawn each step), so the
    penalties over the history decide between them.  ``step(t)`` returns call t's workload:
    `rows_per_slot` rows per slot in a seeded interleaved order, positions advancing with t, and no
    history of its own (the kept histories supply the windows)."""

    def __init__(self, seed, S, V, dtype="f32", rows_per_slot=1, hot=24, prompt_len=(0, 40),
                 last_ns=(1, 8, 64, 300, 4096), greedy_frac=0.3):
        self.seed, self.S, self.V, self.dtype = seed, S, V, dtype
        self.rows_per_slot = rows_per_slot
        rng = _rng(0xD0C0DE, seed)
        self.slot_params, self.prompts, self.hot = {}, {}, {}
        for s in range(S):
            greedy = rng.random() < greedy_frac
            self.slot_params[s] = make_params(
                temperature=0.0 if greedy else float(rng.uniform(0.5, 1.5)),
                top_k=int(rng.integers(0, 65)), top_p=float(rng.choice([1.0, rng.uniform(0.6, 1.0)])),
                min_p=float(rng.choice([0.0, rng.uniform(0.0, 0.1)])),
                penalty_repeat=float(rng.uniform(1.2, 2.0)), penalty_freq=float(rng.uniform(0.2, 1.0)),
                penalty_present=float(rng.choice([0.0, rng.uniform(0.0, 0.5)])),
                penalty_last_n=int(rng.choice(last_ns)), seed=int(rng.integers(0, 2**63)))
            self.hot[s] = rng.choice(V, size=hot, replace=False).astype(np.int32)
            n = int(rng.integers(prompt_len[0], prompt_len[1] + 1))
            pick_hot = rng.random(n) < 0.5
            self.prompts[s] = np.where(pick_hot, rng.choice(self.hot[s], size=n),
                                       rng.integers(0, V, size=n)).astype(np.int32)

    def step(self, t, top_n=0, allowed_lists=None):
        rng = _rng(0xD0C0DE, self.seed, t)
        order = np.repeat(np.arange(self.S), self.rows_per_slot)
        order = order[rng.permutation(order.size)]                # slots interleave
        B = order.size
        x = (rng.standard_normal((B, self.V)) * 1.5).astype(np.float32)
        for b, s in enumerate(order):
            x[b, self.hot[s]] = rng.uniform(5.0, 8.0, size=self.hot[s].size).astype(np.float32)
        logits = to_bf16_bits(x) if self.dtype == "bf16" else x
        seen = {}
        pos = []
        for s in order:
            j = seen.get(int(s), 0)
            seen[int(s)] = j + 1
            pos.append(10_000 * int(s) + t * self.rows_per_slot + j)
        return _workload(f"decode_{self.seed}_t{t}", self.dtype, self.V, logits, dict(self.slot_params),
                         order.astype(np.int32), pos, [], top_n, allowed_lists=allowed_lists)
