"""GPU parity: the CUDA library through its C ABI against the CPU oracle on the same seeded inputs.

Rules (written in the comparisons of tests/_harness.py): greedy ids, the top_k id sequence, the
penalised values and the min_p survivor count bit-exact; top_p survivors and sampled ids exact
except rows the oracle flags (a top_p or draw decision within 1e-6 of a boundary, counted and
printed); log-probabilities within 1e-5 absolute.
"""
import numpy as np
import pytest

import oracle
import synth

from _harness import shape_hint, Stats, compare_logprobs, compare_sample, gpu_logprobs, gpu_sample, report, set_slots, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sampler():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from request_token_sampling_gb300 import Sampler
    s = Sampler(device=0, max_slots=64, max_vocab=synth.V_FULL, max_rows=256)
    yield s
    s.close()


def _check_no_errors(sampler, allowed_bits=0):
    bits = sampler.errors()
    assert bits & ~allowed_bits == 0, hex(bits)


def test_config1_single_row(sampler):
    w = synth.config1()
    set_slots(sampler, w)
    g = gpu_sample(sampler, w)
    rows, ctr = oracle.sample_call(w)
    st = compare_sample(w, rows, g)
    _check_no_errors(sampler)
    assert sampler.slot_state(0)[1] == ctr[0] == 1
    report("config1", st)


def test_config2_verify_windows_counter_persists(sampler):
    """100 consecutive 5-row windows of one request; the device counter carries across calls."""
    w0 = synth.config2_window(0)
    set_slots(sampler, w0, {0: 0})
    st = Stats()
    counters = {0: 0}
    for win in range(synth.CONFIG2_WINDOWS):
        w = synth.config2_window(win, counter=counters[0])
        g = gpu_sample(sampler, w, top_n=0, chosen_lp=False)
        rows, counters = oracle.sample_call(w, counters=counters)
        compare_sample(w, rows, g, top_n=0, stats=st)
    _check_no_errors(sampler)
    assert sampler.slot_state(0)[1] == counters[0] == synth.CONFIG2_WINDOWS
    report("config2", st)


@pytest.mark.parametrize("concurrent", [0, 1, 2], ids=["default-shape", "concurrency-hint", "resident-chunks"])
def test_config3_batch_slots_bf16(sampler, concurrent):
    w = synth.config3()
    set_slots(sampler, w)
    g = gpu_sample(sampler, w, top_n=0, chosen_lp=True, flags=shape_hint(concurrent))
    rows, ctr = oracle.sample_call(w)
    st = compare_sample(w, rows, g, top_n=0)
    _check_no_errors(sampler)
    for s in range(8):
        assert sampler.slot_state(s)[1] == ctr[s]
    report("config3", st)


def test_config4_logprobs_entry(sampler):
    w = synth.config4(fused=False)
    g = gpu_logprobs(sampler, w)
    ref = oracle.logprobs_call(w)
    st = compare_logprobs(w, ref, g)
    _check_no_errors(sampler)
    report("config4 logprobs", st)


@pytest.mark.parametrize("concurrent", [0, 1, 2], ids=["default-shape", "concurrency-hint", "resident-chunks"])
def test_config4_logprobs_entry_pipelined_own_outputs(sampler, concurrent):
    """strata_logprobs_rows back to back with early loads and own outputs: no call waits for the
    one before it; each call's log-probabilities against the oracle."""
    from request_token_sampling_gb300 import (STRATA_FLAG_CONCURRENT, STRATA_FLAG_EARLY_LOAD, STRATA_FLAG_OWN_OUTPUTS,
                                              STRATA_FLAG_PDL)
    base = synth.config4(fused=False)
    sampler.errors()  # drained: an earlier late-counter call would make these wait as usual
    fl = STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD | STRATA_FLAG_OWN_OUTPUTS
    fl |= shape_hint(concurrent)
    ws = []
    for c in range(5):
        w = dict(base)
        w["logits"] = np.roll(base["logits"], 2311 * c, axis=1) if c else base["logits"]
        ws.append((w, upload(w)))
    torch.cuda.synchronize()
    outs = [sampler.logprobs(d["logits"], V=w["V"], chosen=d.get("chosen"), top_n=w["top_n"], allowed=d["allowed"],
                             allowed_off=d["allowed_off"], flags=fl) for w, d in ws]
    torch.cuda.synchronize()
    for (w, _), o in zip(ws, outs):
        compare_logprobs(w, oracle.logprobs_call(w), {k: v.cpu().numpy() for k, v in o.items()})
    _check_no_errors(sampler)


def test_config4_fused_sample_and_logprobs(sampler):
    w = synth.config4(fused=True)
    set_slots(sampler, w)
    g = gpu_sample(sampler, w)
    rows, _ = oracle.sample_call(w)
    st = compare_sample(w, rows, g)
    _check_no_errors(sampler)
    report("config4 fused", st)


@pytest.mark.parametrize("concurrent", [0, 1, 2], ids=["default-shape", "concurrency-hint", "resident-chunks"])
def test_config5_stress_bf16_ties(sampler, concurrent):
    """Heavy ties and 2048-id histories: under the concurrency hint a bf16 row takes one CTA, so
    nearly every thread owns a history id and the threshold keys come from min(raw, penalised)
    over the batches that hold the thread maxima; tied ids at the threshold take the warp-wide
    rescan."""
    w = synth.config5()
    set_slots(sampler, w)
    g = gpu_sample(sampler, w, flags=shape_hint(concurrent))
    rows, ctr = oracle.sample_call(w)
    st = compare_sample(w, rows, g)
    _check_no_errors(sampler)
    for s in range(8):
        assert sampler.slot_state(s)[1] == ctr[s] == 1
    report("config5", st)


@pytest.mark.parametrize("seed", range(24))
def test_random_edge_cases(sampler, seed):
    """Small, ragged and tie-heavy cases across row splits, dtypes, strides and slot mixes."""
    rng = np.random.default_rng(1000 + seed)
    V = int(rng.choice([1, 3, 17, 64, 65, 300, 1023, 4099, 20011, 70001]))
    B = int(rng.integers(1, 12))
    dtype = "bf16" if seed % 3 == 1 else "f32"
    pad = int(rng.choice([0, 8, 24]))
    w = synth.random_case(seed, B=B, V=V, dtype=dtype, ld=V + (-V % 8) + pad, n_slots=int(rng.integers(1, 6)),
                          sampled_frac=0.7, hist_len=int(rng.choice([0, 5, 64, 300])),
                          top_n=int(rng.integers(0, 21)), allowed_sizes=[0, 3, 50] if seed % 2 else None,
                          ties=(seed % 4 == 0))
    if seed % 5 == 2:
        w["row_slot"][0] = 999          # an out-of-range slot: id -1 and the SLOT error bit
    set_slots(sampler, w)
    from request_token_sampling_gb300 import STRATA_FLAG_SPLIT
    split = int(rng.choice([0, 0, 1, 2, 3, 16]))
    g = gpu_sample(sampler, w, flags=STRATA_FLAG_SPLIT(split))
    rows, ctr = oracle.sample_call(w)
    compare_sample(w, rows, g)
    bits = sampler.errors()
    expect = 0x01 if seed % 5 == 2 else 0
    assert bits == expect, hex(bits)
    for s in w["slot_params"]:
        assert sampler.slot_state(s)[1] == ctr[s]


@pytest.mark.parametrize("resident", [False, True], ids=["streaming", "resident"])
def test_config4_pipelined_calls(sampler, resident):
    """Back-to-back calls with programmatic dependent launch and early loads, no host
    synchronisation in between; every call's picks, alternatives and log-probabilities against the
    oracle, the counters advancing call by call.  Streaming chunks take few, large chunks per row for
    such calls; resident chunks keep their size."""
    from request_token_sampling_gb300 import STRATA_FLAG_EARLY_LOAD, STRATA_FLAG_PDL, STRATA_FLAG_RESIDENT
    base = synth.config4(fused=True)
    set_slots(sampler, base)
    fl = STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD | (STRATA_FLAG_RESIDENT if resident else 0)
    one = sampler.shape(0, 0, base["B"], base["V"], base["top_n"], fl & STRATA_FLAG_RESIDENT)["split"]
    if resident:
        assert sampler.shape(0, 0, base["B"], base["V"], base["top_n"], fl)["split"] == one == 16
    else:
        assert sampler.shape(0, 0, base["B"], base["V"], base["top_n"], fl)["split"] < one
    ws, ds, outs = [], [], []
    for c in range(5):
        w = dict(base)
        w["logits"] = np.roll(base["logits"], 977 * c, axis=1) if c else base["logits"]
        ws.append(w)
        ds.append(upload(w))
    torch.cuda.synchronize()
    for w, d in zip(ws, ds):
        outs.append(sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"],
                                   hist_off=d["hist_off"], top_n=w["top_n"], chosen_lp=True, allowed=d["allowed"],
                                   allowed_off=d["allowed_off"], flags=fl))
    torch.cuda.synchronize()
    counters = dict(base["counters"])
    st = Stats()
    for w, o in zip(ws, outs):
        rows, counters = oracle.sample_call(w, counters=counters)
        compare_sample(w, rows, {k: v.cpu().numpy() for k, v in o.items()}, stats=st, debug=False)
    for s in base["slot_params"]:
        assert sampler.slot_state(s)[1] == counters[s]
    _check_no_errors(sampler)
    report("config4 pipelined" + (" resident" if resident else ""), st)


@pytest.mark.parametrize("concurrent", [0, 1, 2], ids=["default-shape", "concurrency-hint", "resident-chunks"])
def test_config4_pipelined_own_outputs(sampler, concurrent):
    """Back-to-back calls on one stream that each write their own outputs: no call waits for the
    one before it, each takes its counters at its start, and the draws still follow call order."""
    from request_token_sampling_gb300 import (STRATA_FLAG_CONCURRENT, STRATA_FLAG_EARLY_LOAD, STRATA_FLAG_OWN_OUTPUTS,
                                              STRATA_FLAG_PDL)
    base = synth.config4(fused=True)
    set_slots(sampler, base)
    sampler.errors()  # drained: an earlier waiting call would make these take their counters late
    fl = STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD | STRATA_FLAG_OWN_OUTPUTS
    fl |= shape_hint(concurrent)
    ws = []
    for c in range(8):
        w = dict(base)
        w["logits"] = np.roll(base["logits"], 613 * c, axis=1) if c else base["logits"]
        ws.append((w, upload(w)))
    torch.cuda.synchronize()
    outs = [sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"], hist_off=d["hist_off"],
                           top_n=w["top_n"], chosen_lp=True, allowed=d["allowed"], allowed_off=d["allowed_off"],
                           flags=fl) for w, d in ws]
    torch.cuda.synchronize()
    counters = dict(base["counters"])
    st = Stats()
    for (w, _), o in zip(ws, outs):
        rows, counters = oracle.sample_call(w, counters=counters)
        compare_sample(w, rows, {k: v.cpu().numpy() for k, v in o.items()}, stats=st, debug=False)
    for s in base["slot_params"]:
        assert sampler.slot_state(s)[1] == counters[s]
    _check_no_errors(sampler)
    report("config4 own outputs", st)


def test_config5_pipelined_own_outputs_rows_share_slots(sampler):
    """Config 5's 64 rows (8 per slot) in three back-to-back calls with own outputs: every row of a
    slot draws at the slot's counter from before its call, and each call advances it by one."""
    from request_token_sampling_gb300 import (STRATA_FLAG_CONCURRENT, STRATA_FLAG_EARLY_LOAD, STRATA_FLAG_OWN_OUTPUTS,
                                              STRATA_FLAG_PDL)
    base = synth.config5()
    set_slots(sampler, base)
    sampler.errors()  # drained: an earlier waiting call would make these take their counters late
    fl = STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD | STRATA_FLAG_OWN_OUTPUTS | STRATA_FLAG_CONCURRENT
    ws = []
    for c in range(3):
        w = dict(base)
        w["logits"] = np.roll(base["logits"], 4099 * c, axis=1) if c else base["logits"]
        ws.append((w, upload(w)))
    torch.cuda.synchronize()
    outs = [sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"], hist_off=d["hist_off"],
                           top_n=w["top_n"], chosen_lp=True, flags=fl) for w, d in ws]
    torch.cuda.synchronize()
    counters = dict(base["counters"])
    st = Stats()
    for (w, _), o in zip(ws, outs):
        rows, counters = oracle.sample_call(w, counters=counters, with_allowed=False)
        compare_sample(w, rows, {k: v.cpu().numpy() for k, v in o.items()}, stats=st, debug=False)
    for s in range(8):
        assert sampler.slot_state(s)[1] == counters[s] == 3
    _check_no_errors(sampler)
    report("config5 own outputs", st)


@pytest.mark.parametrize("resident", [False, True], ids=["streaming", "resident"])
def test_config4_concurrent_groups(resident):
    """Two request groups, each its own context and stream, their pipelined calls interleaved with
    the concurrency hint (one block per full row; resident chunks: 16 blocks per row): every call of
    each group matches the oracle, and each group's counters advance by its own calls only."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from request_token_sampling_gb300 import (STRATA_FLAG_CONCURRENT, STRATA_FLAG_EARLY_LOAD, STRATA_FLAG_PDL,
                                              STRATA_FLAG_RESIDENT, Sampler)
    base = synth.config4(fused=True)
    fl = STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD | STRATA_FLAG_CONCURRENT | (STRATA_FLAG_RESIDENT if resident else 0)
    groups = [Sampler(device=0, max_slots=16, max_vocab=synth.V_FULL, max_rows=64) for _ in range(2)]
    try:
        for g in groups:
            set_slots(g, base)
        assert groups[0].shape(0, 0, base["B"], base["V"], base["top_n"], fl)["split"] == (16 if resident else 2)
        streams = [torch.cuda.Stream() for _ in groups]
        ws, outs = [], []
        for c in range(6):
            w = dict(base)
            w["logits"] = np.roll(base["logits"], 1231 * c, axis=1) if c else base["logits"]
            ws.append((w, upload(w)))
        torch.cuda.synchronize()
        for c, (w, d) in enumerate(ws):
            g = c % 2
            outs.append(groups[g].sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"],
                                         hist_off=d["hist_off"], top_n=w["top_n"], chosen_lp=True,
                                         allowed=d["allowed"], allowed_off=d["allowed_off"], flags=fl,
                                         stream=streams[g]))
        torch.cuda.synchronize()
        counters = [dict(base["counters"]), dict(base["counters"])]
        st = Stats()
        for c, ((w, _), o) in enumerate(zip(ws, outs)):
            rows, counters[c % 2] = oracle.sample_call(w, counters=counters[c % 2])
            compare_sample(w, rows, {k: v.cpu().numpy() for k, v in o.items()}, stats=st, debug=False)
        for g, ctr in zip(groups, counters):
            for s in base["slot_params"]:
                assert g.slot_state(s)[1] == ctr[s]
            _check_no_errors(g)
        report("config4 concurrent groups" + (" resident" if resident else ""), st)
    finally:
        for g in groups:
            g.close()


@pytest.mark.parametrize("split", [1, 2, 4, 6, 8, 13, 16])
def test_full_vocab_every_split(sampler, split):
    """The 248,320-id rows give the same answer whatever the number of CTAs per row."""
    from request_token_sampling_gb300 import STRATA_FLAG_SPLIT
    w = synth.config4(fused=True)
    w["B"] = 3
    w["logits"] = w["logits"][:3]
    w["row_slot"], w["row_pos"] = w["row_slot"][:3], w["row_pos"][:3]
    w["allowed_off"] = w["allowed_off"][:4]
    set_slots(sampler, w)
    g = gpu_sample(sampler, w, flags=STRATA_FLAG_SPLIT(split))
    rows, _ = oracle.sample_call(w)
    compare_sample(w, rows, g)
    _check_no_errors(sampler)


def test_heavy_ties_fallback(sampler):
    """All-equal and two-level rows: more candidates than the per-CTA buffer (exact rounds path)."""
    V = 50000
    rows_np = np.zeros((4, V), np.float32)
    rows_np[1, ::7] = 1.0
    rows_np[2] = -0.0
    rows_np[3, 12345] = 2.0
    w = synth._workload("ties", "f32", V, rows_np,
                        {s: synth.make_params(temperature=1.0, top_k=64, seed=9 + s, penalty_repeat=1.5,
                                              penalty_last_n=8) for s in range(4)},
                        [0, 1, 2, 3], [0, 1, 2, 3],
                        [np.array([0, 7, 14, 40000], np.int32)] * 4, 20)
    set_slots(sampler, w)
    g = gpu_sample(sampler, w)
    rows, _ = oracle.sample_call(w)
    compare_sample(w, rows, g)
    _check_no_errors(sampler)


def test_logprobs_edge_cases(sampler):
    rng = np.random.default_rng(5)
    for V in (1, 7, 20, 21, 333, 40000):
        B = 3
        x = np.full((B, V + (-V % 4)), -7.0, np.float32)
        x[:, :V] = (rng.standard_normal((B, V)) * 4).astype(np.float32)
        allowed = [np.array([0, V - 1, 0], np.int32), np.zeros(0, np.int32),
                   np.concatenate([rng.integers(0, V, 40), [-1, V]]).astype(np.int32)]
        w = synth._workload("lp", "f32", V, x, {}, [0] * B, [0] * B, [], 20, allowed_lists=allowed,
                            chosen=np.array([0, V - 1, V], np.int32))
        g = gpu_logprobs(sampler, w)
        ref = oracle.logprobs_call(w)
        compare_logprobs(w, ref, g)
        assert sampler.errors() == 0x02 | 0x04     # out-of-range allowed and chosen ids flagged


def _boundary_case():
    """Rows built to sit on a top_p or draw boundary: the kernel's double-word fallbacks decide.

    Row 0: two equal logits, top_p 0.5 (the first prefix reaches it exactly).  Row 1: three equal
    logits, top_p = float32(2/3).  Rows 2-3: two survivors whose first cumulative weight equals the
    row's Philox uniform u (temperature 1, then 0.7): d = T * ln(1/u - 1), rounded to float32, for a
    position whose u is above 1/2 (the first survivor carries more than half the weight).
    """
    V, B = 1024, 4
    logits = np.full((B, V), -100.0, np.float32)
    logits[0, 10] = logits[0, 20] = 0.0
    logits[1, 10] = logits[1, 20] = logits[1, 30] = 1.5
    prm = {0: synth.make_params(temperature=1.0, top_k=8, top_p=0.5, seed=7),
           1: synth.make_params(temperature=1.0, top_k=8, top_p=float(np.float32(2.0 / 3.0)), seed=8)}
    pos = [100, 200, 0, 0]
    for b, (T, seed) in ((2, (1.0, 9)), (3, (0.7, 10))):
        p = 0
        while oracle.row_uniform(seed, p, 0) <= 0.5:
            p += 1
        u = oracle.row_uniform(seed, p, 0)
        pos[b] = p
        logits[b, 10] = 0.0
        logits[b, 20] = np.float32(T * np.log(1.0 / u - 1.0))
        prm[b] = synth.make_params(temperature=T, top_k=2, seed=seed)
    return synth._workload("boundary_rows", "f32", V, logits, prm, [0, 1, 2, 3], pos, [[], [], [], []], 3)


def test_rows_on_a_boundary_take_the_exact_fallback(sampler):
    """Every row sits within 1e-6 of a top_p or draw boundary (the oracle flags it): the kernel's
    fp32 decision is within 1e-5 of the boundary, so its double-word sums decide, and the pick must
    be one the oracle's draw makes for a top_p and a uniform within 1e-6 of the row's."""
    w = _boundary_case()
    set_slots(sampler, w)
    rows, _ = oracle.sample_call(w)
    assert all(r["flag_top_p"] or r["flag_draw"] for r in rows), [(r["flag_top_p"], r["flag_draw"]) for r in rows]
    g = gpu_sample(sampler, w, with_allowed=False)
    st = compare_sample(w, rows, g)
    _check_no_errors(sampler)
    assert st.flagged == 4
    report("boundary rows", st)
