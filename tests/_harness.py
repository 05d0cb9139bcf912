"""Helpers shared by the GPU tests: run a ``synth`` workload through the C ABI and compare it
with the CPU oracle under the parity rules (integers bit-exact; sampled ids exact except where the
oracle flags a top_p or draw decision within 1e-6 of a boundary; log-probabilities within 1e-5).
"""
from __future__ import annotations

import numpy as np

import oracle

LP_TOL = 1e-5


def dev_tensor(a, dtype=None):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.to(dtype)
    return t.to("cuda:0")


def upload(w):
    """Device tensors of a workload's inputs."""
    d = dict(logits=dev_tensor(w["logits"]), row_slot=dev_tensor(w["row_slot"]),
             row_pos=dev_tensor(w["row_pos"]))
    d["hist"] = dev_tensor(w["hist"]) if w["hist"] is not None and w["hist"].size else None
    d["hist_off"] = dev_tensor(w["hist_off"]) if d["hist"] is not None else None
    if w.get("allowed_off") is not None:
        a = w["allowed"] if w["allowed"].size else np.zeros(1, np.int32)   # a zero-size tensor has no address
        d["allowed"] = dev_tensor(a)
        d["allowed_off"] = dev_tensor(w["allowed_off"])
    else:
        d["allowed"] = d["allowed_off"] = None
    if w.get("chosen") is not None:
        d["chosen"] = dev_tensor(w["chosen"])
    return d


def shape_hint(kind):
    """Launch-shape flags of the parametrised tests: 0 the library's default, 1 the concurrency hint
    (one block per full row), 2 the concurrency hint with resident chunks (STRATA_FLAG_RESIDENT)."""
    from request_token_sampling_gb300 import STRATA_FLAG_CONCURRENT, STRATA_FLAG_RESIDENT
    return (0, STRATA_FLAG_CONCURRENT, STRATA_FLAG_CONCURRENT | STRATA_FLAG_RESIDENT)[kind]


def set_slots(sampler, w, counters=None):
    counters = w["counters"] if counters is None else counters
    for s, p in w["slot_params"].items():
        sampler.restore_slot(s, p, int(counters.get(s, 0)))


def gpu_sample(sampler, w, d=None, top_n=None, with_allowed=True, debug=True, flags=0, chosen_lp=True):
    import torch
    d = upload(w) if d is None else d
    top_n = w["top_n"] if top_n is None else top_n
    out = sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"],
                         hist_off=d["hist_off"], top_n=top_n, chosen_lp=chosen_lp,
                         allowed=d["allowed"] if with_allowed else None,
                         allowed_off=d["allowed_off"] if with_allowed else None, debug=debug, flags=flags)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def gpu_logprobs(sampler, w, d=None, top_n=None, flags=0):
    import torch
    d = upload(w) if d is None else d
    top_n = w["top_n"] if top_n is None else top_n
    out = sampler.logprobs(d["logits"], V=w["V"], chosen=d.get("chosen"), top_n=top_n, allowed=d["allowed"],
                           allowed_off=d["allowed_off"], flags=flags)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


# Parity counts per workload, gathered by the GPU tests and printed in pytest's terminal summary
# (and written as JSON to the file named by STRATA_PARITY_REPORT, when set).
REPORT = {}


def report(name, stats):
    """Record one workload's parity counts for the end-of-session summary."""
    REPORT[name] = stats.as_dict()


class Stats:
    def __init__(self):
        self.rows = 0
        self.flagged = 0
        self.flag_differs = 0
        self.max_dlp = 0.0

    def lp(self, a, b):
        a = np.asarray(a, np.float64)
        b = np.asarray(b, np.float64)
        both_nan = np.isnan(a) & np.isnan(b)
        both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
        ok = both_nan | both_inf
        with np.errstate(invalid="ignore"):     # inf - inf and NaN operands are settled by `ok`
            d = np.where(ok, 0.0, np.abs(a - b))
        d = np.nan_to_num(d, nan=np.inf)
        if d.size:
            self.max_dlp = max(self.max_dlp, float(d.max()))
        return d

    def as_dict(self):
        return {"rows": self.rows, "flagged": self.flagged, "flagged_and_different": self.flag_differs,
                "max_dlp": self.max_dlp}

    def __repr__(self):
        return (f"rows={self.rows} flagged={self.flagged} flagged_and_different={self.flag_differs} "
                f"max|dlp|={self.max_dlp:.3g}")


def check_flagged_pick(w, b, r, gid, m2g=None):
    """A row the oracle flags may differ from it only across the flagged boundary.

    Its top_k sequence and min_p count match exactly (checked by the caller).  The GPU's top_p
    count m2g must be one the cut gives for some top_p within 1e-6 of the key (the oracle's own
    count when the cut is not flagged).  Given that count, the pick must be one the oracle's draw
    (in double) makes for some uniform within 1e-6 of the row's: the oracle's own pick, or the
    survivor on the other side of the flagged boundary.  Without the debug outputs every count the
    cut allows is tried."""
    eps = oracle.BOUNDARY_EPS
    ids = r["topk_ids"].tolist()
    assert gid in ids, f"row {b}: flagged pick {gid} is not among the top_k survivors"
    jg = ids.index(gid)
    p = w["slot_params"][int(w["row_slot"][b])]
    sel, m1 = r["topk_vals"], r["m1"]
    if r["flag_top_p"]:
        lo = oracle.top_p_cut(sel, m1, p["top_p"] - eps)[0]
        hi = oracle.top_p_cut(sel, m1, p["top_p"] + eps)[0]
    else:
        lo = hi = r["m2"]
    if m2g is not None:
        assert lo <= m2g <= hi, f"row {b}: top_p survivors {m2g}, the cut allows {lo}..{hi}"
        lo = hi = m2g
    ok = False
    for m2 in range(lo, hi + 1):
        j_lo = oracle.draw_index(sel, m2, p["temperature"], max(0.0, r["u"] - eps))[0]
        j_hi = oracle.draw_index(sel, m2, p["temperature"], min(1.0 - 2.0 ** -24, r["u"] + eps))[0]
        ok = ok or j_lo <= jg <= j_hi
    assert ok, f"row {b}: flagged pick index {jg} is not the draw's decision (oracle {r['j']}, m2 {lo}..{hi})"


def compare_sample(w, rows, g, top_n=None, stats=None, debug=True):
    """Check GPU outputs `g` of one sample call against oracle `rows` (asserts)."""
    stats = Stats() if stats is None else stats
    top_n = w["top_n"] if top_n is None else top_n
    V, dtype = w["V"], w["dtype"]
    for b, r in enumerate(rows):
        stats.rows += 1
        gid = int(g["ids"][b])
        if r.get("invalid"):
            assert gid == -1, (b, gid)
            continue
        raw = oracle.widen(w["logits"][b, :V], dtype)
        k = r["topk_ids"].size
        if debug:
            assert g["topk_ids"][b, :k].tolist() == r["topk_ids"].tolist(), f"row {b}: top_k sequence"
            assert np.all(g["topk_ids"][b, k:] == -1)
            assert np.array_equal(g["topk_vals"][b, :k], r["topk_vals"]), f"row {b}: penalised values"
            assert int(g["kept"][b, 0]) == r["m1"], f"row {b}: min_p survivors"
            if not r["flag_top_p"]:
                assert int(g["kept"][b, 1]) == r["m2"], f"row {b}: top_p survivors"
        flagged = r["flag_top_p"] or r["flag_draw"]
        if flagged:
            stats.flagged += 1
            m2g = int(g["kept"][b, 1]) if debug else None
            check_flagged_pick(w, b, r, gid, m2g)
            if gid != r["id"]:
                stats.flag_differs += 1
        else:
            assert gid == r["id"], f"row {b}: sampled id {gid} vs oracle {r['id']}"
        lp_all = None
        if "chosen_lp" in g and gid < 0:
            assert np.isnan(g["chosen_lp"][b]), f"row {b}: a row without a pick has a NaN chosen lp"
        elif "chosen_lp" in g:
            lp_all = oracle.log_softmax(raw)
            d = stats.lp([g["chosen_lp"][b]], [lp_all[gid]])
            assert d.max() <= LP_TOL, f"row {b}: chosen lp off by {d.max()}"
        if top_n:
            assert g["top_ids"][b].tolist() == r["top_ids"].tolist(), f"row {b}: top_logprobs ids"
            d = stats.lp(g["top_lps"][b], r["top_lps"])
            assert d.max() <= LP_TOL, f"row {b}: top lps off by {d.max()}"
        if "allowed_lps" in g and w.get("allowed_off") is not None:
            off = w["allowed_off"]
            d = stats.lp(g["allowed_lps"][off[b]:off[b + 1]], r["allowed_lps"])
            if d.size:
                assert d.max() <= LP_TOL, f"row {b}: allowed lps off by {d.max()}"
    return stats


def compare_logprobs(w, ref, g, stats=None):
    stats = Stats() if stats is None else stats
    top_n = w["top_n"]
    for b, r in enumerate(ref):
        stats.rows += 1
        if "chosen_lp" in r and "chosen_lp" in g:
            d = stats.lp([g["chosen_lp"][b]], [r["chosen_lp"]])
            assert d.max() <= LP_TOL
        if top_n:
            assert g["top_ids"][b].tolist() == r["top_ids"].tolist(), f"row {b}: top ids"
            d = stats.lp(g["top_lps"][b], r["top_lps"])
            assert d.max() <= LP_TOL
        if "allowed_lps" in r:
            off = w["allowed_off"]
            d = stats.lp(g["allowed_lps"][off[b]:off[b + 1]], r["allowed_lps"])
            if d.size:
                assert d.max() <= LP_TOL
    return stats
