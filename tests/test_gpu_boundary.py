"""GPU tests of the boundary: argument errors, the per-slot counter rule, save/restore, graph capture,
launch flags, and the invariants the pages state (greedy unchanged by neutral keys, same seed replays,
a batch row equals the row alone, logprobs off changes nothing)."""
import numpy as np
import pytest

import oracle
import synth

from _harness import compare_sample, dev_tensor, gpu_sample, set_slots, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sampler():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from request_token_sampling_gb300 import Sampler
    s = Sampler(device=0, max_slots=16, max_vocab=synth.V_FULL, max_rows=64)
    yield s
    s.close()


def _small(seed=0, B=6, V=5000, n_slots=3, **kw):
    return synth.random_case(seed, B=B, V=V, n_slots=n_slots, sampled_frac=1.0, hist_len=40, **kw)


def test_argument_errors_launch_nothing(sampler):
    import request_token_sampling_gb300 as S
    w = _small()
    d = upload(w)
    out = torch.full((w["B"],), 777, dtype=torch.int32, device="cuda:0")
    ctx = sampler.ctx
    cases = []
    raw = torch.zeros(w["B"] * w["ld"] + 4, dtype=torch.float32, device="cuda:0")
    misaligned = raw[1:1 + w["B"] * w["ld"]].view(w["B"], w["ld"])
    cases.append((dict(logits=misaligned), S.STRATA_EALIGN))
    cases.append((dict(top_n=21), S.STRATA_EINVAL))
    cases.append((dict(V=w["ld"] + 1), S.STRATA_EINVAL))
    big = torch.zeros((65, w["ld"]), dtype=torch.float32, device="cuda:0")
    cases.append((dict(logits=big, row_slot=torch.zeros(65, dtype=torch.int32, device="cuda:0"),
                       row_pos=torch.zeros(65, dtype=torch.int64, device="cuda:0"),
                       out_ids=torch.zeros(65, dtype=torch.int32, device="cuda:0")), S.STRATA_ERANGE))
    for over, code in cases:
        args = dict(logits=d["logits"], row_slot=d["row_slot"], row_pos=d["row_pos"], out_ids=out, V=w["V"])
        args.update(over)
        with pytest.raises(S.StrataError) as ei:
            S.strata_sample_rows(ctx, **args)
        assert ei.value.code == code
    torch.cuda.synchronize()
    assert (out == 777).all()                        # nothing ran
    bad = dict(synth.make_params(temperature=1.0, top_k=65))
    with pytest.raises(S.StrataError):
        sampler.set_slot(0, bad)
    with pytest.raises(S.StrataError):
        sampler.set_slot(99, synth.make_params())


def test_every_output_written(sampler):
    w = _small(1)
    set_slots(sampler, w)
    d = upload(w)
    o = {"ids": torch.full((w["B"],), 0x7EADBEEF, dtype=torch.int32, device="cuda:0")}
    sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"], hist_off=d["hist_off"], out=o)
    torch.cuda.synchronize()
    assert (o["ids"] >= 0).all() and (o["ids"] < w["V"]).all()


def test_counter_rule_and_restore(sampler):
    w = _small(2, B=7, n_slots=3)
    w["row_slot"] = np.array([0, 0, 1, 2, 0, 1, 2], np.int32)
    w["slot_params"][2]["temperature"] = 0.0         # greedy slot: its counter never moves
    set_slots(sampler, w, {0: 5, 1: 0, 2: 9})
    d = upload(w)
    counters = {0: 5, 1: 0, 2: 9}
    for _ in range(4):
        g = gpu_sample(sampler, w, d=d, top_n=0)
        rows, counters = oracle.sample_call(w, counters=counters)
        compare_sample(w, rows, g, top_n=0)
    assert counters == {0: 9, 1: 4, 2: 9}
    assert [sampler.slot_state(s)[1] for s in range(3)] == [9, 4, 9]
    # save slot 0, run two more calls, restore, replay: identical ids
    p0, c0 = sampler.slot_state(0)
    a = gpu_sample(sampler, w, d=d, top_n=0)["ids"]
    gpu_sample(sampler, w, d=d, top_n=0)
    sampler.restore_slot(0, p0, c0)
    sampler.restore_slot(1, w["slot_params"][1], 4)
    b = gpu_sample(sampler, w, d=d, top_n=0)["ids"]
    assert np.array_equal(a, b)
    # reset_counter sets 0
    sampler.set_slot(0, p0, reset_counter=True)
    assert sampler.slot_state(0)[1] == 0
    # set without reset keeps counting
    sampler.set_slot(1, w["slot_params"][1])
    assert sampler.slot_state(1)[1] == 5


def test_same_seed_replays_and_counter_moves_draws(sampler):
    w = synth.config1()
    p = dict(w["slot_params"][0], temperature=1.5, top_k=64, top_p=1.0, min_p=0.0)
    w["slot_params"][0] = p
    d = upload(w)
    set_slots(sampler, w, {0: 0})
    first = [int(gpu_sample(sampler, w, d=d, top_n=0)["ids"][0]) for _ in range(16)]
    set_slots(sampler, w, {0: 0})
    again = [int(gpu_sample(sampler, w, d=d, top_n=0)["ids"][0]) for _ in range(16)]
    assert first == again
    assert len(set(first)) > 1


def test_neutral_keys_are_greedy_byte_for_byte(sampler):
    w = synth.config4(fused=True)
    for s in w["slot_params"]:
        w["slot_params"][s] = synth.make_params(temperature=0.0, penalty_last_n=64, seed=s)
    set_slots(sampler, w)
    g = gpu_sample(sampler, w, top_n=0)
    raw = oracle.widen(w["logits"][:, :w["V"]], "f32")
    assert g["ids"].tolist() == [int(np.argmax(r)) for r in raw]
    # a sampled request with top_k=1 and no history is greedy too
    for s in w["slot_params"]:
        w["slot_params"][s] = synth.make_params(temperature=0.9, top_k=1, penalty_last_n=0, seed=s)
    set_slots(sampler, w)
    g1 = gpu_sample(sampler, w, top_n=0)
    assert g1["ids"].tolist() == g["ids"].tolist()


def test_batch_row_equals_solo_row(sampler):
    w = synth.config5()
    set_slots(sampler, w)
    batch = gpu_sample(sampler, w)
    for b in (0, 9, 33, 63):
        wb = dict(w)
        wb["B"] = 1
        wb["logits"] = w["logits"][b:b + 1]
        wb["row_slot"] = w["row_slot"][b:b + 1]
        wb["row_pos"] = w["row_pos"][b:b + 1]
        set_slots(sampler, w)
        solo = gpu_sample(sampler, wb)
        for k in ("ids", "chosen_lp", "top_ids", "top_lps", "topk_ids", "topk_vals", "kept"):
            assert np.array_equal(solo[k][0], batch[k][b], equal_nan=(k == "topk_vals")), (b, k)


def test_logprobs_off_changes_nothing(sampler):
    w = synth.config4(fused=True)
    set_slots(sampler, w)
    with_lp = gpu_sample(sampler, w)
    set_slots(sampler, w)
    without = gpu_sample(sampler, w, top_n=0, with_allowed=False, chosen_lp=False, debug=False)
    assert np.array_equal(with_lp["ids"], without["ids"])


@pytest.mark.parametrize("flags", [1, 3])
def test_pdl_flags_same_results(sampler, flags):
    w = synth.config3()
    set_slots(sampler, w)
    a = gpu_sample(sampler, w)
    set_slots(sampler, w)
    b = gpu_sample(sampler, w, flags=flags)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_graph_capture_replays_draw_fresh_numbers(sampler):
    """A captured call advances the device counters on every replay (the pages moved sampling out of
    the captured graph since a sampler baked into a graph draws identical numbers on every replay)."""
    w = synth.config4(fused=True)
    for s in w["slot_params"]:
        w["slot_params"][s] = dict(w["slot_params"][s], temperature=2.0, top_k=64, top_p=1.0, min_p=0.0)
    set_slots(sampler, w, {s: 0 for s in w["slot_params"]})
    d = upload(w)
    out = {"ids": torch.empty(w["B"], dtype=torch.int32, device="cuda:0")}
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"],
                       hist_off=d["hist_off"], out=out, stream=stream)   # warm-up call: counter 0
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"],
                           hist_off=d["hist_off"], out=out, stream=stream)
    torch.cuda.synchronize()
    counters = {s: 1 for s in w["slot_params"]}
    seen = []
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        rows, counters = oracle.sample_call(w, counters=counters, top_n=0, with_allowed=False)
        ids = out["ids"].cpu().numpy()
        for b, r in enumerate(rows):
            if not (r["flag_top_p"] or r["flag_draw"]):
                assert int(ids[b]) == r["id"]
        seen.append(ids.tolist())
    assert seen[0] != seen[1] or seen[1] != seen[2]
    assert sampler.slot_state(0)[1] == 4


@pytest.mark.parametrize("split", [0, 1])
def test_bounded_wait_runs_out_and_the_context_recovers(sampler, split):
    """Failure detection without a GPU fault: the leaders wait on an mbarrier nothing arrives at;
    the bounded wait runs out (about two seconds), the call reports STRATA_DEVERR_TIMEOUT, and the
    next call on the same context is exact again."""
    import request_token_sampling_gb300 as S
    w = synth.config1()
    set_slots(sampler, w)
    sampler.errors()
    gpu_sample(sampler, w, flags=S.STRATA_FLAG_TEST_STALL | S.STRATA_FLAG_SPLIT(split))
    assert sampler.errors() & S.STRATA_DEVERR_TIMEOUT
    set_slots(sampler, w)
    g = gpu_sample(sampler, w)
    rows, _ = oracle.sample_call(w)
    compare_sample(w, rows, g)
    assert sampler.errors() == 0


def test_trace_lines_on_stderr():
    """STRATA_SAMPLE_DEBUG=1: the library prints one line per call with the launch shape it chose."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys; sys.path.insert(0, %r); import torch, synth; from _harness import gpu_sample, set_slots; "
            "import request_token_sampling_gb300 as S; w = synth.config1(); s = S.Sampler(0, 4, w['V'], 4); "
            "set_slots(s, w); gpu_sample(s, w); gpu_sample(s, w, flags=S.STRATA_FLAG_CONCURRENT); "
            "gpu_sample(s, w, flags=S.STRATA_FLAG_PDL | S.STRATA_FLAG_EARLY_LOAD); s.close()") % os.path.join(root, "tests")
    env = dict(os.environ, STRATA_SAMPLE_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stderr.splitlines() if l.startswith("strata: sample_rows")]
    assert len(lines) == 3 and "V=32000" in lines[0] and "split=" in lines[0] and "smem=" in lines[0], r.stderr[-2000:]
    # one stream of calls takes the instance budgeted for two blocks per SM; the concurrency hint three
    assert [l.split("kernel=")[1].split()[0] for l in lines] == ["streaming-2", "streaming", "streaming-2"], lines


def test_own_outputs_after_a_waiting_call_take_counters_late():
    """A flagged call that follows an unflagged pipelined call on the same context takes its
    counters after its wait (the launch it gets carries no own-outputs bit) until the stream has
    drained; the trace shows the flags each launch got."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = """
import sys; sys.path.insert(0, %r)
import torch, synth
from _harness import set_slots, upload
import request_token_sampling_gb300 as S
w = synth.config1(); s = S.Sampler(0, 4, w['V'], 4); set_slots(s, w); d = upload(w)
own = S.STRATA_FLAG_PDL | S.STRATA_FLAG_EARLY_LOAD | S.STRATA_FLAG_OWN_OUTPUTS
def call(fl): s.sample(d['logits'], d['row_slot'], d['row_pos'], V=w['V'], hist=d['hist'], hist_off=d['hist_off'], flags=fl)
call(own); call(S.STRATA_FLAG_PDL | S.STRATA_FLAG_EARLY_LOAD); call(own); call(own)
assert s.errors() == 0
call(own)
torch.cuda.synchronize(); print('counter', s.slot_state(0)[1]); s.close()
""" % os.path.join(root, "tests")
    env = dict(os.environ, STRATA_SAMPLE_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    flags = [int(l.split("flags=")[1].split()[0], 16) for l in r.stderr.splitlines() if l.startswith("strata: sample_rows")]
    assert len(flags) == 5, r.stderr[-2000:]
    own_bits = [bool(f & 0x20) for f in flags]
    assert own_bits == [True, False, False, False, True], flags
    assert "counter 5" in r.stdout


def test_launch_shape_modes(sampler):
    """The shape query covers the three entry points (0 sampling, 1 logprobs, 2 verify windows) and
    refuses any other mode; the concurrency hint gives a full fp32 row two CTAs (512 KiB each) and
    a bf16 row one.
    Resident chunks (STRATA_FLAG_RESIDENT) hold at most 64 KiB of logits: a full fp32 row takes 16
    blocks, a bf16 row 8 under the concurrency hint."""
    import request_token_sampling_gb300 as S
    fl = S.STRATA_FLAG_PDL | S.STRATA_FLAG_EARLY_LOAD | S.STRATA_FLAG_CONCURRENT
    assert sampler.shape(0, 0, 8, synth.V_FULL, 20, fl)["split"] == 2
    assert sampler.shape(0, 1, 8, synth.V_FULL, 20, fl)["split"] == 1
    assert sampler.shape(1, 0, 8, synth.V_FULL, 20, fl)["split"] == 2
    assert sampler.shape(2, 0, 5, synth.V_FULL, 0, fl)["split"] == 2
    assert sampler.shape(2, 0, 5, synth.V_FULL, 0, fl | S.STRATA_FLAG_HISTORY_RING)["split"] == 8
    rs = fl | S.STRATA_FLAG_RESIDENT
    assert sampler.shape(0, 0, 8, synth.V_FULL, 20, rs)["split"] == 16
    assert sampler.shape(0, 1, 8, synth.V_FULL, 20, rs)["split"] == 8
    assert sampler.shape(0, 1, 8, synth.V_FULL, 20, S.STRATA_FLAG_RESIDENT)["split"] == 16
    assert sampler.shape(0, 0, 8, synth.V_FULL, 20, S.STRATA_FLAG_RESIDENT)["chunk"] * 4 <= 65536
    assert sampler.shape(2, 0, 5, synth.V_FULL, 0, rs)["split"] == 16
    for m in (0, 1, 2):
        sh = sampler.shape(m, 1, 3, synth.V_FULL, 5, 0)
        assert sh["grid"] == 3 * sh["split"] and sh["smem"] > 0
    with pytest.raises(S.StrataError) as ei:
        sampler.shape(3, 0, 8, synth.V_FULL, 20, 0)
    assert ei.value.code == S.STRATA_EINVAL
