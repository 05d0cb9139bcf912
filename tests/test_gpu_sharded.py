"""GPU parity of vocabulary-sliced sampling (strata_shard_rows + strata_merge_shards) on one GPU.

Each slice's records are compared entry by entry with the oracle's record of the same slice
(penalised entries, raw entries and ids bit-exact, log-sum-exp within 1e-5); the merged outputs
are compared with the oracle on the whole rows under the usual parity rules, and with the
whole-row library call.  The slices run one after another on one GPU, standing in for ranks that
each hold one slice.
"""
import numpy as np
import pytest

import oracle
import synth

from _harness import LP_TOL, Stats, compare_sample, report, set_slots, upload

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


def _bounds(V, cuts):
    return [0] + list(cuts) + [V]


def _slice_records(sampler, w, d, bounds, top_n, flags=0):
    """Records of every slice [G, B, STRATA_SHARD_RECORD_BYTES] (slices in the order given)."""
    recs = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        part = d["logits"][:, a:b]
        recs.append(sampler.shard(part, d["row_slot"], a, V=b - a, hist=d["hist"], hist_off=d["hist_off"],
                                  top_n=top_n, flags=flags))
    return torch.stack(recs, 0)


def _check_records(w, recs, bounds, top_n):
    """Every slice's record against the oracle's record of that slice."""
    from request_token_sampling_gb300.sharded import unpack_record
    host = recs.cpu().numpy()
    V, dtype = w["V"], w["dtype"]
    worst = 0.0
    for b in range(w["B"]):
        s = int(w["row_slot"][b])
        if s not in w["slot_params"]:
            continue
        p = oracle.Params.from_dict(w["slot_params"][s])
        k = 1 if p.greedy else p.k
        raw = oracle.widen(w["logits"][b, :V], dtype)
        hist = oracle.sampling._slot_history(w, s)
        for g, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
            ref = oracle.shard_record(raw[lo:hi], lo, p, hist, k, top_n)
            got = unpack_record(host[g, b].tobytes())
            assert got["pen"] == ref["pen"], f"row {b} slice {g}: penalised entries"
            assert got["raw"] == ref["raw"], f"row {b} slice {g}: raw entries"
            d = abs(got["lse"] - ref["lse"])
            worst = max(worst, d)
            assert d <= LP_TOL, f"row {b} slice {g}: log-sum-exp off by {d}"
    return worst


def _merge(sampler, recs, d, top_n):
    out = sampler.merge(recs, d["row_slot"], d["row_pos"], top_n=top_n, chosen_lp=True, debug=True)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _run(sampler, w, cuts, name, order=None, flags=0):
    set_slots(sampler, w)
    d = upload(w)
    top_n = w["top_n"]
    bounds = _bounds(w["V"], cuts)
    recs = _slice_records(sampler, w, d, bounds, top_n, flags)
    torch.cuda.synchronize()
    _check_records(w, recs, bounds, top_n)
    if order is not None:
        recs = recs[list(order)].contiguous()
    g = _merge(sampler, recs, d, top_n)
    rows, ctr = oracle.sample_call(w, with_allowed=False)
    st = compare_sample(w, rows, g)
    assert sampler.errors() == 0
    for s in w["slot_params"]:
        assert sampler.slot_state(s)[1] == ctr.get(s, 0), f"slot {s}: counter"
    report(name, st)
    return g


def test_config4_two_slices(sampler):
    """Config 4's eight fp32 rows (sampled, penalised, top_logprobs 20) split at the middle."""
    w = synth.config4(fused=True)
    _run(sampler, w, [w["V"] // 2], "config4 two slices")


def test_config4_matches_whole_row_call(sampler):
    """The merged picks equal the whole-row call's on the same slots and counters."""
    w = synth.config4(fused=True)
    set_slots(sampler, w)
    d = upload(w)
    whole = sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=w["V"], hist=d["hist"],
                           hist_off=d["hist_off"], top_n=w["top_n"], chosen_lp=True, debug=True)
    torch.cuda.synchronize()
    whole = {k: v.cpu().numpy() for k, v in whole.items()}
    set_slots(sampler, w)
    recs = _slice_records(sampler, w, d, _bounds(w["V"], [62080, 124160, 186240]), w["top_n"])
    g = _merge(sampler, recs, d, w["top_n"])
    assert g["ids"].tolist() == whole["ids"].tolist()
    assert np.array_equal(g["topk_ids"], whole["topk_ids"])
    assert np.array_equal(g["kept"], whole["kept"])
    assert g["top_ids"].tolist() == whole["top_ids"].tolist()
    assert np.max(np.abs(g["top_lps"] - whole["top_lps"])) <= 2 * LP_TOL


def test_config5_uneven_slices_bf16(sampler):
    """Config 5's 64 bf16 rows (2048-id Zipf histories, top_k 64, heavy ties) over three uneven
    slices, merged in reverse slice order."""
    w = synth.config5()
    _run(sampler, w, [40000, 200000], "config5 three slices", order=[2, 1, 0])


def test_config3_four_slices_greedy_and_sampled(sampler):
    """Config 3's bf16 batch slots (half greedy) over four slices."""
    w = synth.config3()
    _run(sampler, w, [62080, 124160, 186240], "config3 four slices")


def test_config1_small_vocab_many_slices(sampler):
    """Config 1 (V=32,000, a history id on a spike) over sixteen slices, the library's maximum;
    the concurrency hint on the slices."""
    from request_token_sampling_gb300 import STRATA_FLAG_CONCURRENT
    w = synth.config1()
    cuts = [2000 * i for i in range(1, 16)]
    _run(sampler, w, cuts, "config1 sixteen slices", flags=STRATA_FLAG_CONCURRENT)


@pytest.mark.parametrize("seed", range(6))
def test_random_cases_slices(sampler, seed):
    """Seeded edge cases (ragged V, ties, drawn keys and histories) over 2-5 slices whose bounds
    are multiples of 8 ids."""
    rng = np.random.default_rng(seed)
    V = int(rng.choice([97, 1000, 4099, 32000]))
    w = synth.random_case(seed, B=int(rng.integers(1, 12)), V=V, dtype=str(rng.choice(["f32", "bf16"])),
                          ld=(V + 7) // 8 * 8, ties=bool(seed % 2), hist_len=48)
    G = int(rng.integers(2, 6))
    cuts = sorted(set(int(c) // 8 * 8 for c in rng.integers(8, V, size=G - 1)))
    cuts = [c for c in cuts if 0 < c < V]
    _run(sampler, w, cuts, f"random slices {seed}")


def test_slice_argument_checks(sampler):
    from request_token_sampling_gb300 import (STRATA_EALIGN, STRATA_EINVAL, STRATA_FLAG_PDL,
                                              STRATA_SHARD_RECORD_BYTES, StrataError)
    w = synth.config1()
    set_slots(sampler, w)
    d = upload(w)
    rec = torch.empty(1, STRATA_SHARD_RECORD_BYTES, dtype=torch.uint8, device="cuda:0")
    with pytest.raises(StrataError) as e:
        sampler.shard(d["logits"], d["row_slot"], -1, out=rec)
    assert e.value.code == STRATA_EINVAL
    with pytest.raises(StrataError) as e:
        sampler.shard(d["logits"], d["row_slot"], 0, flags=STRATA_FLAG_PDL, out=rec)
    assert e.value.code == STRATA_EINVAL
    big = torch.empty(2 * STRATA_SHARD_RECORD_BYTES + 8, dtype=torch.uint8, device="cuda:0")
    with pytest.raises(StrataError) as e:
        sampler.shard(d["logits"], d["row_slot"], 0, out=big[8:8 + STRATA_SHARD_RECORD_BYTES].view(1, -1))
    assert e.value.code == STRATA_EALIGN
    recs = torch.zeros(17, 1, STRATA_SHARD_RECORD_BYTES, dtype=torch.uint8, device="cuda:0")
    with pytest.raises(StrataError) as e:
        sampler.merge(recs, d["row_slot"], d["row_pos"])
    assert e.value.code == STRATA_EINVAL
    assert sampler.errors() == 0


def test_out_of_range_slot_row(sampler):
    """A row whose slot is outside the context: its records carry no penalised entries, the merge
    writes id -1 (NaN chosen lp) and sets STRATA_DEVERR_SLOT; the other rows are exact."""
    from request_token_sampling_gb300 import STRATA_DEVERR_SLOT
    w = synth.config4(fused=True)
    w = dict(w, allowed=None, allowed_off=None, row_slot=w["row_slot"].copy())
    w["row_slot"][3] = 1000                      # max_slots is 64
    sampler.errors()                              # clear earlier bits
    set_slots(sampler, w)
    d = upload(w)
    recs = _slice_records(sampler, w, d, _bounds(w["V"], [w["V"] // 2]), w["top_n"])
    g = _merge(sampler, recs, d, w["top_n"])
    assert sampler.errors() == STRATA_DEVERR_SLOT
    assert int(g["ids"][3]) == -1 and np.isnan(g["chosen_lp"][3])
    rows, _ = oracle.sample_call(w, with_allowed=False)
    compare_sample(w, rows, g)


def test_greedy_rows_with_penalties(sampler):
    """Greedy rows whose slots carry penalties (the penalised argmax) over four slices."""
    w = synth.random_case(11, B=6, V=20011, dtype="f32", ld=20016, sampled_frac=0.0, hist_len=40)
    for s in w["slot_params"]:
        w["slot_params"][s] = dict(w["slot_params"][s], penalty_repeat=1.7, penalty_freq=0.4, penalty_present=0.3)
    _run(sampler, w, [5000, 10000, 15000], "greedy penalised slices")


def test_one_slice_is_the_whole_row(sampler):
    """A single slice holding the whole vocabulary merges to the whole-row result (config 3's bf16
    slots, greedy and sampled)."""
    w = synth.config3()
    _run(sampler, w, [], "config3 one slice")


def test_sample_sliced_one_rank_nccl(sampler):
    """`sharded.sample_sliced` through a one-rank NCCL group on a side stream: the slice launch,
    the all-gather and the merge run in order on the GPU, and the picks and log-probabilities equal
    the whole-row call's (config 4's rows, the whole vocabulary as the one slice)."""
    import os
    import torch.distributed as dist
    from request_token_sampling_gb300.sharded import sample_sliced
    if not dist.is_available() or not dist.is_nccl_available():
        pytest.skip("torch.distributed without NCCL")
    w = synth.config4(fused=True)
    V, top_n = w["V"], w["top_n"]
    set_slots(sampler, w)
    d = upload(w)
    whole = sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=V, hist=d["hist"], hist_off=d["hist_off"],
                           top_n=top_n, chosen_lp=True)
    torch.cuda.synchronize()
    whole = {k: v.cpu().numpy() for k, v in whole.items()}
    set_slots(sampler, w)
    os.environ["NCCL_NVLS_ENABLE"] = "0"
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1)
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        out = sample_sliced(sampler, d["logits"][:, :V], 0, d["row_slot"], d["row_pos"], hist=d["hist"],
                            hist_off=d["hist_off"], top_n=top_n, chosen_lp=True, stream=side)
        side.synchronize()
        got = {k: v.cpu().numpy() for k, v in out.items()}
    finally:
        dist.destroy_process_group()
    assert sampler.errors() == 0
    assert got["ids"].tolist() == whole["ids"].tolist()
    assert got["top_ids"].tolist() == whole["top_ids"].tolist()
    assert np.max(np.abs(got["top_lps"] - whole["top_lps"])) <= 2 * LP_TOL
    assert np.max(np.abs(got["chosen_lp"] - whole["chosen_lp"])) <= 2 * LP_TOL
