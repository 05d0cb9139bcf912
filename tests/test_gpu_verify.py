"""GPU parity of verify windows (`strata_sample_verify`): the picks equal the oracle's, and every
slot keeps exactly the rows `oracle.accept_window` keeps.  Drafts are built by the test, from the
oracle's own picks (accepted prefixes of every length) or seeded ids (rejections)."""
import numpy as np
import pytest

import oracle
import synth

from _harness import set_slots, upload

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


def _verify(sampler, w, drafts, flags=0):
    d = upload(w)
    dr = torch.from_numpy(np.asarray(drafts, np.int32)).to("cuda:0")
    o = sampler.verify(d["logits"], d["row_slot"], d["row_pos"], dr, V=w["V"], hist=d["hist"],
                       hist_off=d["hist_off"], top_n=w["top_n"], chosen_lp=True, flags=flags)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


def _check(w, rows, g, drafts):
    flagged = any(r.get("flag_top_p") or r.get("flag_draw") for r in rows)
    ids = [r["id"] for r in rows]
    if not flagged:
        assert g["ids"].tolist() == ids
    # the kept counts are a function of the picks and the drafts: check the kernel's against the
    # oracle's rule applied to the picks the kernel made (and, unflagged, to the oracle's picks)
    keep_gpu = {s: int(g["keep"][s]) for s in set(int(x) for x in w["row_slot"])}
    assert keep_gpu == oracle.accept_window(w["row_slot"], g["ids"].tolist(), drafts)
    if not flagged:
        assert keep_gpu == oracle.accept_window(w["row_slot"], ids, drafts)


@pytest.mark.parametrize("accepted", [0, 1, 2, 3, 4])
def test_verify_window_every_prefix(sampler, accepted):
    """Config 2's five-row window (4 drafts + head): drafts equal the target's picks for the first
    `accepted` rows, then one wrong draft; `accepted` = 4 accepts the whole window."""
    w = synth.config2_window(11 + accepted)
    set_slots(sampler, w)
    rows, _ = oracle.sample_call(w, with_allowed=False)
    picks = [r["id"] for r in rows]
    drafts = picks[:-1] + [-1]
    if accepted < w["B"] - 1:
        drafts[accepted] = (picks[accepted] + 17) % w["V"]
    set_slots(sampler, w)
    g = _verify(sampler, w, drafts)
    rows2, ctr, keep = oracle.verify_call(w, drafts)
    assert keep == {0: accepted + 1}
    _check(w, rows2, g, drafts)
    assert sampler.slot_state(0)[1] == ctr[0]


@pytest.mark.parametrize("accepted", [0, 2, 4])
def test_verify_window_concurrency_hint(sampler, accepted):
    """The same windows with the concurrency hint (two CTAs per full row) and pipelined flags, as
    independent request groups run them; also with resident chunks, and one CTA per row, forced."""
    from request_token_sampling_gb300 import STRATA_FLAG_CONCURRENT, STRATA_FLAG_EARLY_LOAD, STRATA_FLAG_PDL
    w = synth.config2_window(31 + accepted)
    set_slots(sampler, w)
    rows, _ = oracle.sample_call(w, with_allowed=False)
    picks = [r["id"] for r in rows]
    drafts = picks[:-1] + [-1]
    if accepted < w["B"] - 1:
        drafts[accepted] = (picks[accepted] + 29) % w["V"]
    set_slots(sampler, w)
    from request_token_sampling_gb300 import STRATA_FLAG_RESIDENT, STRATA_FLAG_SPLIT
    fl = STRATA_FLAG_CONCURRENT | STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD
    assert sampler.shape(2, 0, w["B"], w["V"], w["top_n"], fl)["split"] == 2
    rows2, ctr, keep = oracle.verify_call(w, drafts)
    assert keep == {0: accepted + 1}
    for extra in (0, STRATA_FLAG_RESIDENT, STRATA_FLAG_SPLIT(1)):
        set_slots(sampler, w)
        g = _verify(sampler, w, drafts, flags=fl | extra)
        _check(w, rows2, g, drafts)
        assert sampler.slot_state(0)[1] == ctr[0]


def test_verify_batch_of_slots_mixed(sampler):
    """Eight slots of config 3 (greedy and sampled), each a window of three rows, drafts mixing the
    slot's own picks and seeded ids."""
    base = synth.config3()
    rng = np.random.default_rng(77)
    order = np.repeat(np.arange(8), 3)
    w = dict(base)
    w["B"] = order.size
    w["logits"] = np.stack([base["logits"][s] for s in order])
    w["row_slot"] = order.astype(np.int32)
    w["row_pos"] = np.array([300 + 10 * s + j for s, j in zip(order, np.tile(np.arange(3), 8))], np.int64)
    w["top_n"] = 3
    set_slots(sampler, w)
    rows, _ = oracle.sample_call(w, with_allowed=False)
    picks = [r["id"] for r in rows]
    drafts = []
    for b, s in enumerate(order):
        last = b + 1 == order.size or order[b + 1] != s
        if last:
            drafts.append(-1)
        elif rng.random() < 0.6:
            drafts.append(picks[b])
        else:
            drafts.append(int(rng.integers(0, w["V"])))
    set_slots(sampler, w)
    g = _verify(sampler, w, drafts)
    rows2, _, _ = oracle.verify_call(w, drafts)
    _check(w, rows2, g, drafts)


def test_verify_graph_replay_resets_the_window_words(sampler):
    """Captured once, replayed three times: every replay counts its windows afresh."""
    w = synth.config2_window(40)
    set_slots(sampler, w, {0: 0})
    d = upload(w)
    rows, _ = oracle.sample_call(w, counters={0: 1}, with_allowed=False)
    picks = [r["id"] for r in rows]
    drafts = picks[:2] + [(picks[2] + 1) % w["V"]] + picks[3:4] + [-1]   # keeps 3 at counter 1
    dr = torch.from_numpy(np.asarray(drafts, np.int32)).to("cuda:0")
    out = {"ids": torch.empty(w["B"], dtype=torch.int32, device="cuda:0"),
           "keep": torch.full((16,), -1, dtype=torch.int32, device="cuda:0")}
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        sampler.verify(d["logits"], d["row_slot"], d["row_pos"], dr, V=w["V"], hist=d["hist"],
                       hist_off=d["hist_off"], out=out, stream=stream)   # warm-up call: counter 0
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            sampler.verify(d["logits"], d["row_slot"], d["row_pos"], dr, V=w["V"], hist=d["hist"],
                           hist_off=d["hist_off"], out=out, stream=stream)
    torch.cuda.synchronize()
    counters = {0: 1}
    for rep in range(3):
        graph.replay()
        torch.cuda.synchronize()
        rows_r, counters, keep = oracle.verify_call(w, drafts, counters=counters, top_n=0)
        ids = out["ids"].cpu().numpy().tolist()
        assert int(out["keep"][0].item()) == oracle.accept_window(w["row_slot"], ids, drafts)[0]
        if not any(r["flag_top_p"] or r["flag_draw"] for r in rows_r):
            assert ids == [r["id"] for r in rows_r]
            assert int(out["keep"][0].item()) == keep[0]
    assert sampler.slot_state(0)[1] == 4


def test_verify_pipelined_windows(sampler):
    """Six windows of config 2 enqueued back to back with programmatic dependent launch and early
    loads: the five rows of a window share one slot (every row counts itself in, the last one
    advances the counter), and each window must see the counter the previous one left."""
    from request_token_sampling_gb300 import STRATA_FLAG_EARLY_LOAD, STRATA_FLAG_PDL
    w0 = synth.config2_window(60)
    set_slots(sampler, w0, {0: 0})
    rng = np.random.default_rng(3)
    ws, drafts, outs = [], [], []
    for k in range(6):
        w = synth.config2_window(60 + k, counter=k)
        ws.append(w)
        drafts.append([int(x) for x in rng.integers(0, w["V"], 4)] + [-1])
    ds = [upload(w) for w in ws]
    drs = [torch.from_numpy(np.asarray(d, np.int32)).to("cuda:0") for d in drafts]
    torch.cuda.synchronize()
    for w, d, dr in zip(ws, ds, drs):
        outs.append(sampler.verify(d["logits"], d["row_slot"], d["row_pos"], dr, V=w["V"], hist=d["hist"],
                                   hist_off=d["hist_off"], chosen_lp=True,
                                   flags=STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD))
    torch.cuda.synchronize()
    for k, (w, o) in enumerate(zip(ws, outs)):
        rows, _, _ = oracle.verify_call(w, drafts[k], counters={0: k})
        _check(w, rows, {key: v.cpu().numpy() for key, v in o.items()}, drafts[k])
    assert sampler.slot_state(0)[1] == 6


def test_verify_refuses_own_outputs(sampler):
    """Verify windows depend on the previous call (its kept counts): the own-outputs flag is an
    argument error there, and nothing is launched."""
    import request_token_sampling_gb300 as S
    w = synth.config2_window(3)
    set_slots(sampler, w)
    d = upload(w)
    dr = torch.full((w["B"],), -1, dtype=torch.int32, device="cuda:0")
    before = sampler.slot_state(0)[1]
    with pytest.raises(S.StrataError) as ei:
        sampler.verify(d["logits"], d["row_slot"], d["row_pos"], dr, V=w["V"], hist=d["hist"], hist_off=d["hist_off"],
                       flags=S.STRATA_FLAG_PDL | S.STRATA_FLAG_EARLY_LOAD | S.STRATA_FLAG_OWN_OUTPUTS)
    assert ei.value.code == S.STRATA_EINVAL
    assert sampler.slot_state(0)[1] == before


def test_verify_needs_drafts_and_keep(sampler):
    import request_token_sampling_gb300 as S
    w = synth.config1()
    d = upload(w)
    out = torch.empty(1, dtype=torch.int32, device="cuda:0")
    with pytest.raises(S.StrataError) as ei:
        S.strata_sample_verify(sampler.ctx, d["logits"], d["row_slot"], d["row_pos"], None, out, None, V=w["V"])
    assert ei.value.code == S.STRATA_EINVAL
