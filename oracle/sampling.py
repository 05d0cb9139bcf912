"""Plain, slow CPU oracle of the decode-time sampling chain and the logprobs entry point.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this module.  It shares no code with the CUDA library and imports
nothing from it; both sides take their inputs from ``synth``.

Every step is the plain definition from the pages, cited by page title and section:

* "#19 serve: per-request temperature/top_p/top_k/min_p/penalties sampling" (the sampled chain),
  sections "What changed" -> "min_p and the penalties", "The sampled chain is one block per
  token", "A persistent per-request draw counter; sampled requests default top_k=20",
  "server.py forwards the block to the engine".
* "#3200 [Engine] OpenAI logprobs / top_logprobs / allowed_token_ids for the CUDA/HIP engine",
  sections "Problem and result" and "Approach" (logprobs on the raw head logits before
  penalties and temperature; top 0..20; allowed_token_ids renormalised over the named ids).
* "#1916 OpenAI logprobs on /v1/chat/completions for the CUDA/HIP engine", "What changed".
* "#559 Several conversations at once: batch slots, a pipelined layer split, per-stage dense
  weights", "What it adds" item 1 (one row per batch slot, each slot sampled with its own keys
  and Philox(seed, position)).

Precision: the penalty arithmetic, the ranking it feeds and the min_p cut are float32 (IEEE
round-to-nearest, no fused multiply-add), because they decide integers (which ids are kept and in
what order) and the pages state them on float logits with ``logf``.  Everything on the softmax
side (top_p mass, the draw's cumulative weights, log-sum-exp, log-probabilities) is float64.

Readings taken where the pages are silent (each is listed in the design notes):
  * the penalty applies to every vocabulary entry before top_k (the ~318M-compare figure is
    k * V * hlen, so every entry was evaluated in every round);
  * inside the penalty: repeat first (multiply if l <= 0, divide if l > 0), then subtract
    count*freq + [count>0]*present in one subtraction (the llama.cpp chain the page names);
  * top_p is measured on temperature-1 probabilities renormalised over the min_p survivors and
    keeps the smallest prefix whose mass reaches top_p; temperature applies after both cuts;
  * the draw picks the first survivor whose inclusive cumulative weight exceeds u * W;
  * greedy rows (temperature <= 0) take the first entry of the penalised order;
  * ties rank the lower index first; -0.0 equals +0.0; NaN ranks below -inf.
"""
from __future__ import annotations

import ctypes
import ctypes.util
from dataclasses import dataclass

import numpy as np

from .philox import row_uniform

BOUNDARY_EPS = 1e-6          # a top_p or draw decision this close to a boundary is "flagged"
DEFAULT_SAMPLED_TOP_K = 20   # "#19 ...": sampled requests default to the sampler's own top_k=20
MAX_TOP_K = 64               # "#19 ...": the sampled path requires top_k in 1..64
MAX_TOP_LOGPROBS = 20        # "#3200 ...": top_logprobs 0..20

_libm = ctypes.CDLL(ctypes.util.find_library("m"))
_libm.logf.restype = ctypes.c_float
_libm.logf.argtypes = [ctypes.c_float]


def c_logf(x: float) -> np.float32:
    """The host C library's single-precision logf, as the min_p formula names it."""
    return np.float32(_libm.logf(ctypes.c_float(x)))


# -------------------------------------------------------------------------------------------
# Request keys
# -------------------------------------------------------------------------------------------

@dataclass
class Params:
    temperature: float = 0.0
    top_k: int = 0
    top_p: float = 1.0
    min_p: float = 0.0
    penalty_repeat: float = 1.0
    penalty_freq: float = 0.0
    penalty_present: float = 0.0
    penalty_last_n: int = 64
    seed: int = 0

    @classmethod
    def from_dict(cls, d):
        return cls(**{k: d[k] for k in cls.__dataclass_fields__})

    @property
    def greedy(self) -> bool:
        # "#19 ...", "server.py forwards the block": an absent temperature keeps greedy and
        # temperature=0 means the same thing.
        return not (np.float32(self.temperature) > 0)

    @property
    def k(self) -> int:
        # "#19 ...", "A persistent per-request draw counter; sampled requests default top_k=20".
        return DEFAULT_SAMPLED_TOP_K if self.top_k == 0 else int(self.top_k)


def params_valid(p: Params) -> bool:
    """Whether the engine can honour these keys (it refuses the rest instead of changing them)."""
    vals = [p.temperature, p.top_p, p.min_p, p.penalty_repeat, p.penalty_freq, p.penalty_present]
    if not all(np.isfinite(np.float32(v)) for v in vals):
        return False
    if not (0 <= p.top_k <= MAX_TOP_K):
        return False
    if not (np.float32(p.penalty_repeat) > 0):
        return False
    if np.float32(p.min_p) < 0:
        return False
    if p.penalty_last_n < 0:
        return False
    return True


# -------------------------------------------------------------------------------------------
# Steps of the chain
# -------------------------------------------------------------------------------------------

def widen(row, dtype: str) -> np.ndarray:
    """bf16 -> fp32 is exact (the bf16 bits are the high half of the fp32 bits)."""
    if dtype == "bf16":
        return (np.asarray(row, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return np.asarray(row, dtype=np.float32)


def history_counts(hist_ids, last_n: int, V: int) -> dict:
    """Multiplicity of each id over the request's last `penalty_last_n` history tokens.

    "#19 ...", "min_p and the penalties": the serve loop uploads the request's last
    penalty_last_n tokens; ids outside [0, V) are not vocabulary entries and are skipped.
    """
    hist_ids = np.asarray(hist_ids, dtype=np.int64)
    h = min(int(last_n), hist_ids.size)
    window = hist_ids[hist_ids.size - h:] if h > 0 else hist_ids[:0]
    counts = {}
    for t in window.tolist():
        if 0 <= t < V:
            counts[t] = counts.get(t, 0) + 1
    return counts


def penalties_neutral(p: Params) -> bool:
    return (np.float32(p.penalty_repeat) == 1 and np.float32(p.penalty_freq) == 0
            and np.float32(p.penalty_present) == 0)


def apply_penalties(row32: np.ndarray, counts: dict, r: float, f: float, pres: float) -> np.ndarray:
    """The llama.cpp-style penalty set on every id with count c > 0, in float32.

    "#19 ...", "min_p and the penalties": the repeat penalty multiplies non-positive logits and
    divides positive ones; the frequency penalty is freq * count; the presence penalty is a
    boolean (present when the count is positive), not the count.
    """
    out = np.array(row32, dtype=np.float32, copy=True)
    if not counts:
        return out
    ids = np.fromiter(counts.keys(), dtype=np.int64)
    c = np.fromiter(counts.values(), dtype=np.int64)
    r32, f32_, p32 = np.float32(r), np.float32(f), np.float32(pres)
    x = out[ids]
    x = np.where(x <= np.float32(0), x * r32, x / r32).astype(np.float32)
    sub = (c.astype(np.float32) * f32_ + np.where(c > 0, p32, np.float32(0))).astype(np.float32)
    out[ids] = (x - sub).astype(np.float32)
    return out


def rank_order(values32: np.ndarray) -> np.ndarray:
    """All ids ordered by value descending, ties to the lowest index, NaN last.

    "#19 ...", "The sampled chain is one block per token": k argmax rounds whose ties resolve to
    the lowest index (a serial scan that only replaces on a strictly larger value); the first k entries of this order are the k
    rounds' winners in order.
    """
    v = np.asarray(values32, dtype=np.float32).astype(np.float64)
    idx = np.arange(v.size)
    return np.lexsort((idx, -v))


def min_p_cut(sel: np.ndarray, min_p: float) -> int:
    """Kept prefix length after min_p, in logit space, float32.

    "#19 ...", "min_p and the penalties": keep the prefix with sel_logit >= sel_logit[0] +
    logf(min_p); 0 disables; the top survivor is never cut, so at least one id is kept.
    """
    k = sel.size
    if not (np.float32(min_p) > 0):
        return k
    thr = np.float32(sel[0]) + c_logf(float(np.float32(min_p)))
    kept = int(np.count_nonzero(sel.astype(np.float32) >= np.float32(thr)))
    return max(1, kept)


def top_p_cut(sel: np.ndarray, m1: int, top_p: float):
    """Kept prefix length after top_p over the min_p survivors; returns (m2, flagged).

    Reading: probabilities at temperature 1 renormalised over the m1 survivors (min_p runs
    first and the page has the two cuts compose); keep the smallest prefix whose mass reaches top_p.
    """
    tp = float(np.float32(top_p))
    if tp >= 1.0:
        return m1, False
    if tp <= 0.0:
        return 1, False
    v = sel[:m1].astype(np.float64)
    q = np.exp(v - v[0])
    cum = np.cumsum(q) / np.sum(q)
    m2 = int(np.argmax(cum >= tp)) + 1 if np.any(cum >= tp) else m1
    flagged = bool(np.any(np.abs(cum - tp) < BOUNDARY_EPS))
    return m2, flagged


def draw_index(sel: np.ndarray, m2: int, temperature: float, u: float):
    """Index of the drawn survivor; returns (j, flagged).

    Temperature scales the kept logits, the weights are exp((l_i - l_0) / T), and the pick is the
    first survivor whose inclusive cumulative weight exceeds u * W.
    """
    v = sel[:m2].astype(np.float64)
    w = np.exp((v - v[0]) / float(np.float32(temperature)))
    cum = np.cumsum(w)
    W = cum[-1]
    hit = np.nonzero(cum > u * W)[0]
    j = int(hit[0]) if hit.size else m2 - 1
    flagged = bool(np.any(np.abs(cum / W - u) < BOUNDARY_EPS))
    return j, flagged


def log_softmax(raw32: np.ndarray) -> np.ndarray:
    """log-probabilities of the raw head logits in float64 (LSE with the max subtracted)."""
    l = np.asarray(raw32, dtype=np.float32).astype(np.float64)
    m = np.max(l)
    lse = m + np.log(np.sum(np.exp(l - m)))
    return l - lse


def allowed_renorm(raw32: np.ndarray, allowed) -> np.ndarray:
    """log-probabilities normalised over the caller's subset of ids only, in the caller's order.

    "#3200 ...", "Problem and result": allowed_token_ids returns a distribution renormalised over
    exactly the ids the caller named.  Reading: a repeated id counts once in the normaliser and is
    reported at every place it was named; an id outside [0, V) is reported as NaN and ignored.
    """
    l = np.asarray(raw32, dtype=np.float32).astype(np.float64)
    a = np.asarray(allowed, dtype=np.int64)
    V = l.size
    ok = (a >= 0) & (a < V)
    out = np.full(a.size, np.nan)
    if not np.any(ok):
        return out
    uniq = np.unique(a[ok])
    m = np.max(l[uniq])
    lse_a = m + np.log(np.sum(np.exp(l[uniq] - m)))
    out[ok] = l[a[ok]] - lse_a
    return out


# -------------------------------------------------------------------------------------------
# Whole rows
# -------------------------------------------------------------------------------------------

def sample_row(raw32, p: Params, hist_ids, position: int, counter: int, mask_ids=None):
    """One row of the sampled chain (or the greedy argmax); returns a dict of every decision.

    Chain order from "#19 ...": penalties over the history window -> top_k (ties to the lowest
    index) -> min_p -> top_p -> temperature -> Philox(seed, position) draw at the slot's counter.

    `mask_ids` (optional): the row's allowed_token_ids used as a sampling mask ("#3200 ...",
    "Problem and result" names constrained decoding as the client use).  Reading: the chain runs
    over the named ids only (out-of-range ids are ignored, a repeat counts once); an empty or
    absent list leaves the row unrestricted; with no named id inside [0, V) the row has no
    candidate (id -1).
    """
    V = raw32.size
    if penalties_neutral(p) or p.penalty_last_n <= 0 or hist_ids is None:
        counts = {}
    else:
        counts = history_counts(hist_ids, p.penalty_last_n, V)
    pen = apply_penalties(raw32, counts, p.penalty_repeat, p.penalty_freq, p.penalty_present)
    if mask_ids is not None and len(mask_ids) > 0:
        a = np.asarray(mask_ids, dtype=np.int64)
        keep = np.unique(a[(a >= 0) & (a < V)])
        if keep.size == 0:
            return dict(greedy=p.greedy, flag_top_p=False, flag_draw=False, u=None, id=-1, nocand=True,
                        topk_ids=np.zeros(0, np.int64), topk_vals=np.zeros(0, np.float32), m1=0, m2=0, j=0)
        order = keep[rank_order(pen[keep])]
    else:
        order = rank_order(pen)
    res = dict(greedy=p.greedy, flag_top_p=False, flag_draw=False, u=None)
    if p.greedy:
        res.update(id=int(order[0]), topk_ids=order[:1].copy(), topk_vals=pen[order[:1]],
                   m1=1, m2=1, j=0)
        return res
    k = min(p.k, order.size)
    sel_ids = order[:k]
    sel = pen[sel_ids]
    m1 = min_p_cut(sel, p.min_p)
    m2, f_tp = top_p_cut(sel, m1, p.top_p)
    u = row_uniform(p.seed, position, counter)
    j, f_dr = draw_index(sel, m2, p.temperature, u)
    res.update(id=int(sel_ids[j]), topk_ids=sel_ids.copy(), topk_vals=sel.copy(), m1=m1, m2=m2,
               j=j, u=u, flag_top_p=f_tp, flag_draw=f_dr)
    return res


def logprobs_row(raw32, chosen, top_n: int, allowed=None):
    """The logprobs of one row from its raw (pre-penalty, pre-temperature) logits.

    "#3200 ...", "Approach": the value comes from the verify window's head logits before
    sampling, penalties and temperature; one entry per token with up to 20 top alternatives.
    """
    lp = log_softmax(raw32)
    V = lp.size
    res = {}
    if chosen is not None:
        res["chosen_lp"] = float(lp[chosen]) if 0 <= chosen < V else float("nan")
    n = int(top_n)
    order = rank_order(raw32)[:n]
    ids = np.full(n, -1, dtype=np.int64)
    lps = np.full(n, -np.inf)
    ids[:order.size] = order
    lps[:order.size] = lp[order]
    res["top_ids"], res["top_lps"] = ids, lps
    if allowed is not None:
        res["allowed_lps"] = allowed_renorm(raw32, allowed)
    return res


# -------------------------------------------------------------------------------------------
# Whole calls, with the per-slot counter semantics
# -------------------------------------------------------------------------------------------

def _slot_history(w, s):
    if w.get("hist") is None or w.get("hist_off") is None or s >= w["n_hist_slots"]:
        return None
    off = w["hist_off"]
    return w["hist"][off[s]:off[s + 1]]


def sample_call(w, counters=None, top_n=None, with_allowed=True, mask_allowed=False):
    """One batched sampling call over workload dict `w` (see ``synth``); mirrors the library call.

    Every row reads its slot's draw counter as it stood before the call; afterwards each slot
    that had at least one sampled row advances by exactly one ("#19 ...": the Philox draw
    counter persists across a request's verify windows).  Returns (rows, new_counters).
    """
    counters = dict(w["counters"] if counters is None else counters)
    top_n = w["top_n"] if top_n is None else top_n
    V, dtype = w["V"], w["dtype"]
    rows = []
    sampled_slots = set()
    for b in range(w["B"]):
        s = int(w["row_slot"][b])
        raw = widen(w["logits"][b, :V], dtype)
        if s not in w["slot_params"]:
            rows.append(dict(id=-1, invalid=True))
            continue
        p = Params.from_dict(w["slot_params"][s])
        mask = None
        if mask_allowed and w.get("allowed_off") is not None:
            off = w["allowed_off"]
            mask = w["allowed"][off[b]:off[b + 1]]
        r = sample_row(raw, p, _slot_history(w, s), int(w["row_pos"][b]), counters.get(s, 0), mask)
        if not p.greedy:
            sampled_slots.add(s)
        allowed = None
        if with_allowed and w.get("allowed_off") is not None:
            off = w["allowed_off"]
            allowed = w["allowed"][off[b]:off[b + 1]]
        r.update(logprobs_row(raw, r["id"], top_n, allowed))
        rows.append(r)
    for s in sampled_slots:
        counters[s] = counters.get(s, 0) + 1
    return rows, counters


def logprobs_call(w, chosen=None, top_n=None):
    """One batched logprobs call (no sampling): chosen lp, top-N raw alternatives, allowed subset."""
    top_n = w["top_n"] if top_n is None else top_n
    V, dtype = w["V"], w["dtype"]
    chosen = w.get("chosen") if chosen is None else chosen
    out = []
    for b in range(w["B"]):
        raw = widen(w["logits"][b, :V], dtype)
        allowed = None
        if w.get("allowed_off") is not None:
            off = w["allowed_off"]
            allowed = w["allowed"][off[b]:off[b + 1]]
        c = None if chosen is None else int(chosen[b])
        out.append(logprobs_row(raw, c, top_n, allowed))
    return out


def accept_window(row_slot, row_ids, row_draft) -> dict:
    """Rows kept per slot of one verify window (the step right after sampling).

    "#19 ...", "What changed": the emitted tokens are always the target's own samples; the drafts
    only fill the verified window.  "#559 ...", "Not done (yet)": a sampled row is accepted when
    its pick equals the draft.  Reading: within one call, the rows of a slot are its window in row
    order; row j's pick is compared with `row_draft[j]`, the draft that the window placed right
    after row j's position (-1 for the window's last row, which has none).  Every row up to and
    including the first one whose pick differs from its draft (or that has no draft) is kept, so
    n_keep = 1 + the number of leading rows whose pick equals their draft; a row with pick -1
    (an out-of-range slot or no candidate) never matches.  Returns {slot: n_keep}.
    """
    keep, open_ = {}, {}
    for s, t, d in zip(row_slot, row_ids, row_draft):
        s, t, d = int(s), int(t), int(d)
        if s not in keep:
            keep[s], open_[s] = 0, True
        if not open_[s]:
            continue
        keep[s] += 1
        if d < 0 or t < 0 or t != d:
            open_[s] = False
    return keep


def verify_call(w, row_draft, counters=None, top_n=None):
    """A sampling call whose rows are verify windows: `sample_call` plus the kept count per slot."""
    rows, counters = sample_call(w, counters=counters, top_n=top_n, with_allowed=False)
    keep = accept_window(w["row_slot"], [r["id"] for r in rows], row_draft)
    return rows, counters, keep


# -------------------------------------------------------------------------------------------
# Per-slot histories kept between calls (the history-ring variant of the calls above)
# -------------------------------------------------------------------------------------------

HISTORY_RING_CAP = 4096   # ids a slot keeps: the largest penalty window ("#19 ...": penalty_last_n)


def _with_histories(w, state):
    """Workload `w` with each slot's penalty window taken from `state` ({slot: list of ids})."""
    slots = sorted(set(int(s) for s in w["row_slot"]) | set(int(s) for s in state))
    n = (max(slots) + 1) if slots else 0
    lists = [np.asarray(state.get(s, []), dtype=np.int32) for s in range(n)]
    off = np.zeros(n + 1, dtype=np.int32)
    for s, a in enumerate(lists):
        off[s + 1] = off[s] + a.size
    w2 = dict(w)
    w2["hist"] = np.concatenate(lists).astype(np.int32) if n else np.zeros(0, np.int32)
    w2["hist_off"] = off
    w2["n_hist_slots"] = n
    return w2


def history_call(w, state, counters=None, top_n=None, row_draft=None, mask_allowed=False):
    """One sampling call (a verify call when `row_draft` is given) whose penalty windows come from
    the slots' own run histories, followed by the history update.

    "#19 ...", "min_p and the penalties": before every window the serve loop hands the sampler the
    request's last penalty_last_n tokens, the consumed tail plus the fed-back head.  Kept on the
    device instead, each slot's history is its run so far: every row of the call counts over the
    same window, the last min(penalty_last_n, length) ids as they stood before the call; after it
    the slot's history grows by its rows' picks in row order (a verify call appends only the kept
    rows, "#19 ...", "What changed": the emitted tokens are the target's own samples), and a pick of
    -1 (no candidate, an out-of-range slot) appends nothing.  `state` is {slot: list of ids} and is
    not modified.  Returns (rows, new_counters, new_state, keep) with keep None for a plain call.
    """
    w2 = _with_histories(w, state)
    if row_draft is None:
        rows, counters = sample_call(w2, counters=counters, top_n=top_n, mask_allowed=mask_allowed)
        keep = None
    else:
        rows, counters, keep = verify_call(w2, row_draft, counters=counters, top_n=top_n)
    new = history_append(state, w["row_slot"], [r["id"] for r in rows], keep)
    return rows, counters, new, keep


def history_append(state, row_slot, ids, keep=None):
    """The history update that ends a call: each slot's picks in row order, only its first
    keep[slot] rows when `keep` is given (a verify call), picks of -1 skipped.  Returns a new
    {slot: list of ids}; `state` is not modified."""
    new = {s: list(v) for s, v in state.items()}
    taken = {}
    for s, t in zip(row_slot, ids):
        s, t = int(s), int(t)
        taken[s] = taken.get(s, 0) + 1
        if keep is not None and taken[s] > keep.get(s, 0):
            continue
        if t >= 0:
            new.setdefault(s, []).append(t)
    return new


def history_tail(state, slot, max_n=HISTORY_RING_CAP):
    """What a slot's history read returns: (the last min(length, capacity, max_n) ids, length)."""
    h = list(state.get(slot, []))
    m = min(len(h), HISTORY_RING_CAP, max(0, int(max_n)))
    return np.asarray(h[len(h) - m:], dtype=np.int32), len(h)


# -------------------------------------------------------------------------------------------
# Vocabulary shards: a row's vocabulary split into slices (devices or buffers), each reporting a
# record, the records merged into the row's result
# -------------------------------------------------------------------------------------------

def shard_record(raw32_shard, v0: int, p: Params, hist_ids, k: int, top_n: int) -> dict:
    """What one slice of a row (ids v0 .. v0 + len - 1) reports for the merge.

    The row's top_k list and top_n raw alternatives are each among the union of its slices' own
    lists, so a slice reports its k best penalised entries (value, id, raw logit), its top_n raw
    entries (value, id) and the log-sum-exp of its raw logits ("#19 ...": penalties over the
    history window, then top_k; "#3200 ...", "Approach": log-probabilities of the raw logits).
    History ids are the row's own (global) ids; a slice counts those that fall inside it.
    """
    raw = np.asarray(raw32_shard, dtype=np.float32)
    n = raw.size
    counts = {}
    if not (penalties_neutral(p) or p.penalty_last_n <= 0 or hist_ids is None):
        for t, c in history_counts(hist_ids, p.penalty_last_n, v0 + n).items():
            if t >= v0:
                counts[t - v0] = c
    pen = apply_penalties(raw, counts, p.penalty_repeat, p.penalty_freq, p.penalty_present)
    op = rank_order(pen)[:k]
    orr = rank_order(raw)[:top_n]
    l = raw.astype(np.float64)
    m = np.max(l) if n else -np.inf
    lse = float(m + np.log(np.sum(np.exp(l - m)))) if n and np.isfinite(m) else float("-inf")
    return dict(pen=[(float(pen[i]), v0 + int(i), float(raw[i])) for i in op],
                raw=[(float(raw[i]), v0 + int(i)) for i in orr], lse=lse)


def merge_records(records, p: Params, position: int, counter: int, top_n: int) -> dict:
    """A row's result from its slices' records: the same chain as sample_row and logprobs_row.

    The penalised entries of all slices, ordered by value descending with ties to the lowest id,
    give the top_k list; min_p, top_p, temperature and the Philox draw follow on it; the row's
    log-sum-exp is the log of the summed exponentials of the slices' log-sum-exps.
    """
    pen = sorted((e for r in records for e in r["pen"]), key=lambda e: (-e[0], e[1]))
    raw = sorted((e for r in records for e in r["raw"]), key=lambda e: (-e[0], e[1]))
    lses = np.array([r["lse"] for r in records], dtype=np.float64)
    mx = np.max(lses)
    lse = float(mx + np.log(np.sum(np.exp(lses - mx)))) if np.isfinite(mx) else float("-inf")
    res = dict(greedy=p.greedy, flag_top_p=False, flag_draw=False, u=None)
    k = 1 if p.greedy else min(p.k, len(pen))
    sel = pen[:k]
    sel_vals = np.array([e[0] for e in sel], dtype=np.float32)
    sel_ids = np.array([e[1] for e in sel], dtype=np.int64)
    if p.greedy:
        j, m1, m2 = 0, 1, 1
    else:
        m1 = min_p_cut(sel_vals, p.min_p)
        m2, f_tp = top_p_cut(sel_vals, m1, p.top_p)
        u = row_uniform(p.seed, position, counter)
        j, f_dr = draw_index(sel_vals, m2, p.temperature, u)
        res.update(u=u, flag_top_p=f_tp, flag_draw=f_dr)
    res.update(id=int(sel_ids[j]), topk_ids=sel_ids, topk_vals=sel_vals, m1=m1, m2=m2, j=j,
               chosen_lp=float(np.float64(sel[j][2]) - lse))
    top = raw[:top_n]
    ids = np.full(top_n, -1, dtype=np.int64)
    lps = np.full(top_n, -np.inf)
    for i, (v, t) in enumerate(top):
        ids[i] = t
        lps[i] = float(np.float64(v) - lse)
    res.update(top_ids=ids, top_lps=lps, lse=lse)
    return res
