"""GPU parity of kept per-slot histories (STRATA_FLAG_HISTORY_RING): decode runs whose penalty
windows come from the context's rings match `oracle.history_call` step after step, and the rings
hold exactly the oracle's histories afterwards (read back with strata_history_get).

A sampled pick that the oracle flags as within 1e-6 of a top_p or draw boundary may differ; the
run then continues from the kernel's picks (`oracle.history_append` applied to them), so later
steps still compare like for like."""
import numpy as np
import pytest

import oracle
import synth

from _harness import Stats, compare_sample, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def S():
    import request_token_sampling_gb300 as mod
    return mod


@pytest.fixture(scope="module")
def sampler():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from request_token_sampling_gb300 import Sampler
    s = Sampler(device=0, max_slots=16, max_vocab=synth.V_FULL, max_rows=64)
    s.history_enable()
    yield s
    s.close()


def _start(sampler, run):
    """Keys, counters 0 and prompts of a run into the sampler; the oracle's initial state."""
    for s, p in run.slot_params.items():
        sampler.restore_slot(s, p, 0)
        sampler.history_set(s, run.prompts[s])
    return {s: [int(x) for x in run.prompts[s]] for s in run.slot_params}, {s: 0 for s in run.slot_params}


def _call(sampler, S, w, d, drafts=None, flags=0, mask=False, out=None, stream=None):
    fl = flags | S.STRATA_FLAG_HISTORY_RING | (S.STRATA_FLAG_ALLOWED_MASK if mask else 0)
    if drafts is None:
        return sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], top_n=w["top_n"],
                              chosen_lp=True, allowed=d["allowed"], allowed_off=d["allowed_off"],
                              debug=out is None, flags=fl, out=out, stream=stream)
    return sampler.verify(d["logits"], d["row_slot"], d["row_pos"], d["draft"], V=w["V"], top_n=w["top_n"],
                          chosen_lp=True, flags=fl, out=out, stream=stream)


def _host(o):
    return {k: v.cpu().numpy() for k, v in o.items()}


def _advance(w, state, counters, g, drafts=None, mask=False, stats=None, debug=True):
    """Compare one call's kernel outputs `g` with the oracle; return the next (state, counters)."""
    rows, ctr, new, keep = oracle.history_call(w, state, counters=counters, row_draft=drafts, mask_allowed=mask)
    compare_sample(w, rows, g, stats=stats, debug=debug)
    ids = g["ids"].tolist()
    keep_gpu = None
    if drafts is not None:
        keep_gpu = {s: int(g["keep"][s]) for s in set(int(x) for x in w["row_slot"])}
        assert keep_gpu == oracle.accept_window(w["row_slot"], ids, drafts)
    if ids == [r["id"] for r in rows]:
        assert keep_gpu is None or keep_gpu == keep
        return new, ctr
    return oracle.history_append(state, w["row_slot"], ids, keep_gpu), ctr


def _check_rings(sampler, state):
    for s, h in state.items():
        got, n = sampler.history_get(s)
        want, m = oracle.history_tail(state, s)
        assert n == m, f"slot {s}: length {n} vs {m}"
        assert got.tolist() == want.tolist(), f"slot {s}: kept ids differ"


def test_history_set_get_roundtrip(sampler, S):
    sampler.history_set(3, [5, 6, 7])
    got, n = sampler.history_get(3)
    assert got.tolist() == [5, 6, 7] and n == 3
    long = np.arange(5000, dtype=np.int32) * 7 % 1000
    sampler.history_set(3, long)
    got, n = sampler.history_get(3)
    assert n == 5000 and got.tolist() == long[-S.STRATA_HISTORY_CAP:].tolist()
    got, n = sampler.history_get(3, max_n=9)
    assert got.tolist() == long[-9:].tolist()
    sampler.history_set(3, [])
    assert sampler.history_get(3)[1] == 0 and sampler.history_get(3)[0].size == 0
    assert sampler.history_get(15)[1] == 0            # never set: empty
    with pytest.raises(S.StrataError) as ei:
        sampler.history_set(16, [1])
    assert ei.value.code == S.STRATA_ERANGE


def test_history_errors(sampler, S):
    from request_token_sampling_gb300 import Sampler
    run = synth.DecodeRun(3, 2, synth.V_SMALL)
    w = run.step(0)
    d = upload(w)
    with Sampler(device=0, max_slots=4, max_vocab=synth.V_SMALL, max_rows=8) as fresh:
        with pytest.raises(S.StrataError) as ei:
            fresh.history_set(0, [1, 2])
        assert ei.value.code == S.STRATA_EINVAL
        with pytest.raises(S.StrataError) as ei:
            _call(fresh, S, w, d)
        assert ei.value.code == S.STRATA_EINVAL       # the flag before strata_history_enable
    h = torch.zeros(4, dtype=torch.int32, device="cuda:0")
    ho = torch.tensor([0, 4], dtype=torch.int32, device="cuda:0")
    with pytest.raises(S.StrataError) as ei:
        sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=h, hist_off=ho,
                       flags=S.STRATA_FLAG_HISTORY_RING)
    assert ei.value.code == S.STRATA_EINVAL           # the flag replaces hist/hist_off
    with pytest.raises(S.StrataError) as ei:
        _call(sampler, S, w, d, flags=S.STRATA_FLAG_PDL | S.STRATA_FLAG_EARLY_LOAD | S.STRATA_FLAG_OWN_OUTPUTS)
    assert ei.value.code == S.STRATA_EINVAL           # kept histories depend on the previous call


@pytest.mark.parametrize("dtype,V,flags", [("f32", synth.V_SMALL, 0), ("bf16", 50_000, 0),
                                           ("f32", synth.V_SMALL, 3), ("bf16", synth.V_FULL, 1)])
def test_history_decode_loop(sampler, S, dtype, V, flags):
    """Six slots, one row each per call, twelve calls: every pick goes into its slot's history and
    steers the next call's penalties."""
    run = synth.DecodeRun(11 + V % 7, 6, V, dtype=dtype)
    state, counters = _start(sampler, run)
    stats = Stats()
    for t in range(12):
        w = run.step(t, top_n=3)
        g = _host(_call(sampler, S, w, upload(w), flags=flags))
        state, counters = _advance(w, state, counters, g, stats=stats)
    _check_rings(sampler, state)
    for s in run.slot_params:
        assert sampler.slot_state(s)[1] == counters[s]
    assert stats.flag_differs <= 1, stats


def test_history_rows_of_a_slot_and_masked_rows(sampler, S):
    """Three rows per slot per call, appended in row order; rows restricted to named ids, one row
    naming no id in range (its pick is -1 and appends nothing)."""
    run = synth.DecodeRun(5, 5, synth.V_SMALL, rows_per_slot=3)
    state, counters = _start(sampler, run)
    rng = np.random.default_rng(9)
    for t in range(6):
        lists = []
        for b in range(run.S * run.rows_per_slot):
            r = rng.random()
            lists.append([] if r < 0.5 else ([-1, synth.V_SMALL + 3] if r < 0.6
                                               else rng.integers(0, synth.V_SMALL, 12).tolist()))
        w = run.step(t, allowed_lists=lists)
        g = _host(_call(sampler, S, w, upload(w), mask=True))
        assert (g["ids"] == -1).sum() == sum(1 for a in lists if a and all(x < 0 or x >= w["V"] for x in a))
        state, counters = _advance(w, state, counters, g, mask=True)
    _check_rings(sampler, state)
    # the lists naming no id in range also report those ids (NaN allowed log-probabilities)
    assert sampler.errors() & ~(S.STRATA_DEVERR_NOCAND | S.STRATA_DEVERR_ALLOWED) == 0


def test_history_verify_windows(sampler, S):
    """Windows of four rows per slot: only the kept rows enter the history; drafts follow the
    oracle's own picks for a seeded number of rows, then turn wrong."""
    run = synth.DecodeRun(8, 4, synth.V_SMALL, rows_per_slot=4)
    state, counters = _start(sampler, run)
    rng = np.random.default_rng(4)
    kept_total = 0
    for t in range(8):
        w = run.step(t)
        rows, _, _, _ = oracle.history_call(w, state, counters=counters)
        picks = [r["id"] for r in rows]
        good = {s: int(rng.integers(0, run.rows_per_slot)) for s in run.slot_params}
        seen, drafts = {}, []
        for b, s in enumerate(w["row_slot"]):
            j = seen.get(int(s), 0)
            seen[int(s)] = j + 1
            if j == run.rows_per_slot - 1:
                drafts.append(-1)
            else:
                drafts.append(picks[b] if j < good[int(s)] else (picks[b] + 1) % w["V"])
        d = upload(w)
        d["draft"] = torch.from_numpy(np.asarray(drafts, np.int32)).to("cuda:0")
        g = _host(_call(sampler, S, w, d, drafts=drafts))
        state, counters = _advance(w, state, counters, g, drafts=drafts, debug=False)
        kept_total += sum(int(g["keep"][s]) for s in run.slot_params)
    _check_rings(sampler, state)
    assert kept_total > 8 * run.S                 # some windows kept more than one row


def test_history_long_windows_wrap_the_ring(sampler, S):
    """penalty_last_n 4096 over prompts longer than the ring: the window starts mid-ring."""
    run = synth.DecodeRun(21, 3, synth.V_SMALL, last_ns=(4096,), prompt_len=(4500, 6000))
    state, counters = _start(sampler, run)
    for t in range(4):
        w = run.step(t)
        g = _host(_call(sampler, S, w, upload(w)))
        state, counters = _advance(w, state, counters, g)
    _check_rings(sampler, state)


def test_history_back_to_back_early_loads(sampler, S):
    """Eight calls enqueued with no host synchronisation in between, with programmatic dependent
    launch and early loads: each call's windows must wait for the previous call's appends."""
    run = synth.DecodeRun(31, 6, synth.V_SMALL, greedy_frac=0.5)
    state, counters = _start(sampler, run)
    torch.cuda.synchronize()
    ws = [run.step(t) for t in range(8)]
    ds = [upload(w) for w in ws]
    outs = []
    for w, d in zip(ws, ds):
        outs.append(_call(sampler, S, w, d, flags=S.STRATA_FLAG_PDL | S.STRATA_FLAG_EARLY_LOAD, out={}))
    torch.cuda.synchronize()
    for w, o in zip(ws, outs):
        state, counters = _advance(w, state, counters, _host(o), debug=False)
    _check_rings(sampler, state)


def test_history_graph_replay(sampler, S):
    """One call captured in a CUDA graph and replayed five times on the same logits: every replay
    draws at the next counter and counts over the history the previous replay extended."""
    run = synth.DecodeRun(41, 5, synth.V_SMALL, greedy_frac=0.4)
    w = run.step(0)
    d = upload(w)
    out = {"ids": torch.empty(w["B"], dtype=torch.int32, device="cuda:0"),
           "chosen_lp": torch.empty(w["B"], dtype=torch.float32, device="cuda:0")}
    state, counters = _start(sampler, run)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        _call(sampler, S, w, d, out=out, stream=stream)            # an eager call first
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            _call(sampler, S, w, d, out=out, stream=stream)
    torch.cuda.synchronize()
    state, counters = _advance(w, state, counters, _host(out), debug=False)
    for rep in range(5):
        graph.replay()
        torch.cuda.synchronize()
        state, counters = _advance(w, state, counters, _host(out), debug=False)
    _check_rings(sampler, state)
    for s in run.slot_params:
        assert sampler.slot_state(s)[1] == counters[s]


@pytest.mark.parametrize("split", [0, 1, -1], ids=["concurrency-hint", "one-cta-per-row", "resident-hint"])
def test_history_verify_windows_full_vocab(sampler, S, split):
    """The verify-window shape at V=248,320 fp32 (5 rows: 4 drafts + head, one request, repeat 1.1
    over 64 ids) for ten consecutive windows, history kept on the device; with the concurrency hint
    (8 CTAs per row for these calls), forced to one CTA per row, and with resident chunks."""
    fl = S.STRATA_FLAG_SPLIT(split) if split > 0 else S.STRATA_FLAG_CONCURRENT
    if split == 0:
        assert sampler.shape(2, 0, 5, synth.V_FULL, 0, S.STRATA_FLAG_HISTORY_RING | fl)["split"] == 8
    if split < 0:
        fl |= S.STRATA_FLAG_RESIDENT
    run = synth.DecodeRun(51, 1, synth.V_FULL, rows_per_slot=5, last_ns=(64,), prompt_len=(64, 64),
                          greedy_frac=0.0)
    state, counters = _start(sampler, run)
    rng = np.random.default_rng(12)
    for t in range(10):
        w = run.step(t)
        rows, _, _, _ = oracle.history_call(w, state, counters=counters)
        picks = [r["id"] for r in rows]
        good = int(rng.integers(0, 5))
        drafts = [picks[j] if j < good else (picks[j] + 5) % w["V"] for j in range(4)] + [-1]
        d = upload(w)
        d["draft"] = torch.from_numpy(np.asarray(drafts, np.int32)).to("cuda:0")
        g = _host(_call(sampler, S, w, d, drafts=drafts, flags=fl))
        state, counters = _advance(w, state, counters, g, drafts=drafts, debug=False)
    _check_rings(sampler, state)
