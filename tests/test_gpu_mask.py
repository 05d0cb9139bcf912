"""GPU parity of allowed_token_ids as a sampling mask (STRATA_FLAG_ALLOWED_MASK): rows that name
allowed ids sample only among them, exactly as the oracle's masked chain; the log-probability
outputs keep describing the raw distribution."""
import numpy as np
import pytest

import oracle
import synth

from _harness import shape_hint, compare_sample, gpu_sample, set_slots

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


def _mask_flag():
    from request_token_sampling_gb300 import STRATA_FLAG_ALLOWED_MASK
    return STRATA_FLAG_ALLOWED_MASK


@pytest.mark.parametrize("concurrent", [0, 1, 2], ids=["default-shape", "concurrency-hint", "resident-chunks"])
def test_mask_config4_fused(sampler, concurrent):
    """Config 4's rows with their 5/100/1000-id lists used as masks (also with the concurrency hint:
    two CTAs per row, both id bitmaps as long as a half row)."""
    w = synth.config4(fused=True)
    set_slots(sampler, w)
    g = gpu_sample(sampler, w, flags=_mask_flag() | shape_hint(concurrent))
    rows, ctr = oracle.sample_call(w, mask_allowed=True)
    compare_sample(w, rows, g)
    off = w["allowed_off"]
    for b in range(w["B"]):
        assert int(g["ids"][b]) in set(w["allowed"][off[b]:off[b + 1]].tolist())
    assert sampler.errors() == 0
    for s in w["slot_params"]:
        assert sampler.slot_state(s)[1] == ctr[s]


@pytest.mark.parametrize("seed", range(8))
def test_mask_random_cases(sampler, seed):
    """Random small and ragged rows, ties, bf16, forced splits; masks of 0 (unrestricted), 3 and 50
    ids (repeats allowed) round-robin."""
    rng = np.random.default_rng(2000 + seed)
    V = int(rng.choice([17, 300, 4099, 20011, 70001]))
    B = int(rng.integers(1, 10))
    dtype = "bf16" if seed % 2 else "f32"
    w = synth.random_case(300 + seed, B=B, V=V, dtype=dtype, ld=V + (-V % 8), n_slots=int(rng.integers(1, 5)),
                          sampled_frac=0.8, hist_len=int(rng.choice([0, 64])), top_n=int(rng.integers(0, 8)),
                          allowed_sizes=[0, 3, 50], ties=(seed % 4 == 0))
    set_slots(sampler, w)
    from request_token_sampling_gb300 import STRATA_FLAG_SPLIT
    split = int(rng.choice([0, 2, 16]))
    esz = 2 if dtype == "bf16" else 4
    if split and -(-V // split) * esz > 190_000:
        split = 0
    g = gpu_sample(sampler, w, flags=_mask_flag() | STRATA_FLAG_SPLIT(split))
    rows, ctr = oracle.sample_call(w, mask_allowed=True)
    compare_sample(w, rows, g)
    assert sampler.errors() == 0
    for s in w["slot_params"]:
        assert sampler.slot_state(s)[1] == ctr[s]


def test_mask_without_any_id_in_range(sampler):
    """A masked sampled row whose ids all lie outside [0, V): id -1, the NOCAND bit, and its slot's
    counter still advances once (the row counted itself among the slot's arrivals)."""
    w = synth.config1()
    w["allowed"] = np.array([-5, w["V"], w["V"] + 9], np.int32)
    w["allowed_off"] = np.array([0, 3], np.int32)
    set_slots(sampler, w, {0: 7})
    g = gpu_sample(sampler, w, flags=_mask_flag())
    rows, ctr = oracle.sample_call(w, counters={0: 7}, mask_allowed=True)
    assert rows[0]["id"] == -1 and int(g["ids"][0]) == -1
    assert np.isnan(g["chosen_lp"][0])
    from request_token_sampling_gb300 import STRATA_DEVERR_ALLOWED, STRATA_DEVERR_NOCAND
    assert sampler.errors() == STRATA_DEVERR_NOCAND | STRATA_DEVERR_ALLOWED
    assert sampler.slot_state(0)[1] == ctr[0] == 8
    # and the next, unmasked call draws at counter 8 as usual
    g2 = gpu_sample(sampler, w, with_allowed=False)
    rows2, _ = oracle.sample_call(w, counters={0: 8}, with_allowed=False)
    if not (rows2[0]["flag_top_p"] or rows2[0]["flag_draw"]):
        assert int(g2["ids"][0]) == rows2[0]["id"]


def test_mask_off_matches_plain(sampler):
    """Without the flag the allowed lists only report (the draws equal a call without them)."""
    w = synth.config4(fused=True)
    set_slots(sampler, w)
    a = gpu_sample(sampler, w)
    set_slots(sampler, w)
    b = gpu_sample(sampler, w, with_allowed=False)
    assert a["ids"].tolist() == b["ids"].tolist()
