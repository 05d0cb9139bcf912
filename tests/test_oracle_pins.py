"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test fixes a value the pages or the mathematics determine: hand cases of every rule of the
chain, closed forms, invariants, known-answer vectors and a library generator for Philox, brute
force against a second formulation on tiny vocabularies, and a statistical check of the draw.
A plausible slip in the oracle (a dropped term, a flipped sign, a wrong index, a transposed
operand, the cuts in the wrong order) fails at least one of them.
"""
import ctypes
import math
import os

import numpy as np
import pytest

import oracle
import synth
from oracle import Params
from oracle.philox import philox4x32_10, row_uniform

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
f32 = np.float32


# ----------------------------------------------------------------------------- Philox
def _kat():
    rows = []
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(x, 16) for x in line.split()]
        rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answers():
    kat = _kat()
    assert len(kat) == 3
    for ctr, key, out in kat:
        assert list(philox4x32_10(ctr, key)) == out


def _curand_host():
    for name in ("libcurand.so", "libcurand.so.10", "/usr/local/cuda/lib64/libcurand.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


def test_philox_matches_curand_host_generator():
    """cuRAND's host Philox4_32_10 generator keys with the seed's two halves and starts at
    counter 0: its first four words must equal our Philox at counter (0,0,0,0)."""
    lib = _curand_host()
    if lib is None:
        pytest.skip("libcurand not loadable")
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:   # CURAND_RNG_PSEUDO_PHILOX4_32_10
        pytest.skip("cuRAND host generator unavailable")
    try:
        rng = np.random.default_rng(7)
        seeds = [0, 1, 1234, 2**32 - 1, 2**32, 2**64 - 1] + [int(x) for x in rng.integers(0, 2**63, 6)]
        for seed in seeds:
            assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(0)) == 0
            buf = (ctypes.c_uint32 * 4)()
            assert lib.curandGenerate(gen, buf, ctypes.c_size_t(4)) == 0
            mine = philox4x32_10((0, 0, 0, 0), (seed & 0xFFFFFFFF, seed >> 32))
            assert list(buf) == list(mine), hex(seed)
    finally:
        lib.curandDestroyGenerator(gen)


def test_row_uniform_layout():
    u = row_uniform(1234, 5, 7)
    assert 0.0 <= u < 1.0
    assert u * 2**24 == int(u * 2**24)
    x0 = philox4x32_10((5, 0, 7, 0), (1234, 0))[0]
    assert u == (x0 >> 8) / 2**24
    # position and counter occupy different counter words; the seed is the key
    big = (3 << 32) | 9
    x1 = philox4x32_10((9, 3, 11, 2), (0x89ABCDEF, 0x01234567))[0]
    assert row_uniform(0x0123456789ABCDEF, big, (2 << 32) | 11) == (x1 >> 8) / 2**24
    assert row_uniform(1, 0, 0) != row_uniform(1, 0, 1) != row_uniform(1, 1, 0)


def test_row_uniform_is_uniform():
    n = 40000
    us = np.array([row_uniform(99, 17, c) for c in range(n)])
    hist, _ = np.histogram(us, bins=20, range=(0.0, 1.0))
    chi2 = float(np.sum((hist - n / 20) ** 2 / (n / 20)))
    assert chi2 < 50.0          # 19 dof: p ~ 1e-4 at 43.8


# ----------------------------------------------------------------------------- penalties
def test_penalty_hand_cases():
    row = np.array([2.0, -2.0, 0.0, 5.0, 3.0], dtype=f32)
    cnt = {0: 1, 1: 1, 2: 1}
    out = oracle.apply_penalties(row, cnt, 2.0, 0.0, 0.0)
    assert out.tolist() == [1.0, -4.0, 0.0, 5.0, 3.0]       # divide positive, multiply non-positive
    out = oracle.apply_penalties(row, {3: 3}, 1.0, 0.5, 1.0)
    assert out[3] == f32(2.5)                                 # 5 - (3*0.5 + 1)
    out = oracle.apply_penalties(row, {3: 3}, 1.0, 0.0, 1.0)
    assert out[3] == f32(4.0)                                 # presence is boolean, not the count
    out = oracle.apply_penalties(row, {4: 1}, 1.5, 0.0, 0.0)
    assert out[4] == f32(2.0)
    # repeat first, then the subtraction: (4/2) - (1*1 + 1) = 0, not (4 - 2)/2 = 1
    out = oracle.apply_penalties(np.array([4.0], f32), {0: 1}, 2.0, 1.0, 1.0)
    assert out[0] == f32(0.0)
    # untouched ids stay bit-identical
    assert out.dtype == np.float32


def test_penalty_float32_rounding():
    """The chain is float32 with one rounding per operation (no fused multiply-add)."""
    x, r, c, fq, pr = f32(7.3), f32(1.1), 3, f32(0.1), f32(0.1)
    expect = f32(f32(x / r) - f32(f32(f32(c) * fq) + pr))
    got = oracle.apply_penalties(np.array([x], f32), {0: c}, float(r), float(fq), float(pr))[0]
    assert got == expect
    assert got.view(np.uint32) == expect.view(np.uint32)


def test_neutral_penalties_bit_identical():
    rng = np.random.default_rng(3)
    row = (rng.standard_normal(1000) * 3).astype(f32)
    row[5] = -0.0
    cnt = oracle.history_counts(rng.integers(0, 1000, 64), 64, 1000)
    out = oracle.apply_penalties(row, cnt, 1.0, 0.0, 0.0)
    assert np.array_equal(out.view(np.uint32), row.view(np.uint32))


def test_history_window_clamp():
    hist = [7, 7, 3, 9, 9, 9, -1, 12]
    assert oracle.history_counts(hist, 3, 10) == {9: 1}              # last 3: 9, -1, 12(out of range)
    assert oracle.history_counts(hist, 100, 10) == {7: 2, 3: 1, 9: 3}
    assert oracle.history_counts(hist, 0, 10) == {}
    assert oracle.history_counts([], 64, 10) == {}


# ----------------------------------------------------------------------------- ranking
def _argmax_rounds(vals, k):
    """Second formulation: k serial argmax rounds with a strict '>' (ties to the lowest index)."""
    taken = set()
    out = []
    for _ in range(k):
        best = None
        for i, v in enumerate(vals):
            if i in taken:
                continue
            if best is None or v > vals[best]:
                best = i
        taken.add(best)
        out.append(best)
    return out


@pytest.mark.parametrize("seed", range(40))
def test_rank_order_vs_argmax_rounds(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(1, 65))
    vals = rng.integers(-4, 5, size=V).astype(f32) * f32(0.5)          # many ties
    vals[rng.random(V) < 0.2] = -0.0
    vals[rng.random(V) < 0.2] = 0.0
    if seed % 3 == 0:
        vals = synth.to_bf16_bits((rng.standard_normal(V) * 3).astype(f32))
        vals = oracle.widen(vals, "bf16")
    k = int(rng.integers(1, V + 1))
    assert oracle.rank_order(vals)[:k].tolist() == _argmax_rounds([float(v) for v in vals], k)


# ----------------------------------------------------------------------------- widening
def test_widen_bf16_bit_patterns():
    """bf16 is the high half of an IEEE binary32: fixed bit patterns widen to known values."""
    bits = np.array([0x3F80, 0xC000, 0x8000, 0x0000, 0x7F80, 0xFF80, 0x0001, 0x4049, 0x3E80, 0xBF00,
                     0x0080, 0x7F7F], dtype=np.uint16)
    got = oracle.widen(bits, "bf16")
    assert got.dtype == np.float32
    want = [1.0, -2.0, -0.0, 0.0, math.inf, -math.inf, 2.0 ** -133, 3.140625, 0.25, -0.5, 2.0 ** -126,
            (2.0 - 2.0 ** -7) * 2.0 ** 127]
    assert [float(x) for x in got] == want
    assert math.copysign(1.0, float(got[2])) == -1.0 and math.copysign(1.0, float(got[3])) == 1.0
    # every pattern's low 16 fp32 bits are zero and the high 16 are the pattern itself
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    u = oracle.widen(allb, "bf16").view(np.uint32)
    assert np.array_equal(u >> 16, allb.astype(np.uint32)) and not np.any(u & 0xFFFF)


def test_widen_f32_is_the_row_itself():
    x = np.array([1.5, -0.0, np.inf, -3.25e-39], dtype=np.float32)
    assert oracle.widen(x, "f32").view(np.uint32).tolist() == x.view(np.uint32).tolist()


# ----------------------------------------------------------------------------- key validity
@pytest.mark.filterwarnings("ignore:overflow encountered in cast")
def test_params_valid_rules():
    """Keys the engine refuses rather than adjusts ("#19 ...", "server.py forwards the block"):
    top_k outside 0..64 (0 means 20; the sampled path needs 1..64), a repeat penalty that is not
    positive (the positive branch divides by it), a negative min_p, a negative window, any
    non-finite float.  Everything else is honoured (min_p above 1 keeps the head, top_p <= 0 keeps
    the head, top_p >= 1 disables the cut)."""
    ok = oracle.params_valid
    assert ok(Params())
    assert ok(Params(temperature=0.7, top_k=64, top_p=0.0, min_p=3.0, penalty_repeat=0.5,
                     penalty_freq=-1.0, penalty_present=-2.0, penalty_last_n=0))
    assert ok(Params(top_k=0)) and ok(Params(top_k=1)) and ok(Params(top_p=-1.0)) and ok(Params(temperature=-1.0))
    for bad in (dict(top_k=65), dict(top_k=-1), dict(penalty_repeat=0.0), dict(penalty_repeat=-1.0),
                dict(min_p=-0.01), dict(penalty_last_n=-1), dict(temperature=math.nan), dict(top_p=math.inf),
                dict(min_p=math.nan), dict(penalty_freq=-math.inf), dict(penalty_present=math.nan),
                dict(penalty_repeat=math.inf), dict(temperature=1e39)):
        assert not ok(Params(**bad)), bad


def test_rank_order_special_values():
    v = np.array([np.nan, -np.inf, 1.0, -0.0, 0.0, np.inf, 1.0], dtype=f32)
    assert oracle.rank_order(v).tolist() == [5, 2, 6, 3, 4, 1, 0]


# ----------------------------------------------------------------------------- cuts
def test_min_p_hand_case():
    sel = np.array([5.0, 4.0, 2.0], f32)
    assert oracle.min_p_cut(sel, 0.2) == 2                # thr = 5 + ln 0.2 = 3.3906
    assert oracle.min_p_cut(sel, 0.0) == 3                # disabled
    assert oracle.min_p_cut(sel, 0.05) == 2               # thr = 2.0043 > 2
    assert oracle.min_p_cut(sel, 0.04) == 3               # thr = 1.7811
    assert oracle.min_p_cut(sel, 0.9) == 1
    assert oracle.min_p_cut(np.array([5.0, 5.0, 4.0], f32), 1.0) == 2   # only the head's ties
    assert oracle.min_p_cut(sel, 3.0) == 1                # above 1: the head still survives
    # exact float32 boundary: an entry equal to the threshold is kept
    thr = f32(5.0) + oracle.c_logf(0.2)
    assert oracle.min_p_cut(np.array([5.0, thr, np.nextafter(thr, f32(-10))], f32), 0.2) == 2


def test_min_p_uses_c_logf():
    for x in (0.05, 0.2, 0.5, 0.9, 0.01, 1e-6):
        assert abs(float(oracle.c_logf(x)) - math.log(float(f32(x)))) < 4e-7 * max(1, abs(math.log(x)))


def test_top_p_hand_case():
    sel = np.array([5.0, 4.0], f32)
    assert oracle.top_p_cut(sel, 2, 0.7)[0] == 1          # e/(e+1) = 0.7311 >= 0.7
    assert oracle.top_p_cut(sel, 2, 0.75)[0] == 2
    assert oracle.top_p_cut(sel, 2, 1.0)[0] == 2
    assert oracle.top_p_cut(sel, 2, 0.0)[0] == 1
    assert oracle.top_p_cut(sel, 1, 0.99)[0] == 1


def test_min_p_then_top_p_compose():
    """min_p removes the tail first, which changes top_p's normaliser."""
    sel = np.array([0.0, -1.0] + [-3.0] * 18, f32)
    m1 = oracle.min_p_cut(sel, 0.2)                       # thr = -1.609: keeps [0, -1]
    assert m1 == 2
    assert oracle.top_p_cut(sel, m1, 0.7)[0] == 1         # 1/(1+e^-1) = 0.731 >= 0.7
    # applying top_p over all 20 first would keep far more (cum(0) = 0.44 < 0.7)
    assert oracle.top_p_cut(sel, 20, 0.7)[0] > 2


def test_draw_hand_cases():
    sel = np.array([5.0, 4.0], f32)
    assert oracle.draw_index(sel, 2, 1.0, 0.5)[0] == 0    # C/W = [0.7311, 1]
    assert oracle.draw_index(sel, 2, 1.0, 0.8)[0] == 1
    assert oracle.draw_index(sel, 2, 0.5, 0.8)[0] == 0    # T=0.5: C/W = [0.8808, 1]
    assert oracle.draw_index(sel, 1, 1.0, 0.999)[0] == 0  # one survivor
    j, flag = oracle.draw_index(sel, 2, 1.0, 1.0 / (1.0 + math.exp(-1.0)))
    assert flag                                            # exactly on the boundary
    assert oracle.draw_index(sel, 2, 1.0, 0.0)[0] == 0
    # the pick is the first survivor whose cumulative weight EXCEEDS u*W: on an exact tie of
    # u*W with a cumulative weight the next survivor is taken
    eq = np.array([0.0, 0.0, 0.0, 0.0], f32)
    assert oracle.draw_index(eq, 4, 1.0, 0.5)[0] == 2
    assert oracle.draw_index(eq, 4, 1.0, 0.25)[0] == 1


def test_draw_chi_square():
    """Draw frequencies over 30,000 counters match exp((l_i - l_0)/T) / W."""
    p = Params(temperature=0.9, top_k=5, top_p=1.0, min_p=0.0, seed=4242)
    raw = np.array([1.0, 0.5, 0.0, -0.5, -1.0, -9.0, -9.0], f32)
    n = 30000
    ids = [oracle.sample_row(raw, p, None, 3, c)["id"] for c in range(n)]
    counts = np.bincount(ids, minlength=7)[:5]
    w = np.exp((raw[:5].astype(np.float64) - 1.0) / 0.9)
    exp = n * w / w.sum()
    chi2 = float(np.sum((counts - exp) ** 2 / exp))
    assert chi2 < 25.0                                     # 4 dof: p ~ 5e-5 at 25
    assert np.bincount(ids, minlength=7)[5:].sum() == 0


def test_large_temperature_is_near_uniform_over_kept():
    p = Params(temperature=1e4, top_k=4, seed=5)
    raw = np.array([3.0, 2.0, 1.0, 0.0, -1.0], f32)
    ids = [oracle.sample_row(raw, p, None, 0, c)["id"] for c in range(8000)]
    counts = np.bincount(ids, minlength=5)
    assert counts[4] == 0 and all(abs(c - 2000) < 200 for c in counts[:4])


# ----------------------------------------------------------------------------- logprobs
def test_logprobs_sum_to_one_and_uniform():
    rng = np.random.default_rng(11)
    raw = (rng.standard_normal(5000) * 3).astype(f32)
    lp = oracle.log_softmax(raw)
    assert abs(math.fsum(np.exp(lp)) - 1.0) < 1e-12
    assert np.allclose(oracle.log_softmax(np.zeros(7, f32)), -math.log(7), atol=0, rtol=1e-15)
    # shift invariance
    assert np.allclose(oracle.log_softmax(raw + f32(100.0)), lp, atol=1e-9)


def test_allowed_renorm_rules():
    rng = np.random.default_rng(12)
    raw = (rng.standard_normal(300) * 3).astype(f32)
    full = oracle.allowed_renorm(raw, np.arange(300))
    assert np.allclose(full, oracle.log_softmax(raw), atol=1e-12)          # A = V: plain logprobs
    assert oracle.allowed_renorm(raw, [17]).tolist() == [0.0]              # |A| = 1
    a = [5, 9, 5, 299]
    out = oracle.allowed_renorm(raw, a)
    assert out[0] == out[2]                                                # repeat counted once
    assert abs(math.fsum(np.exp(out[[0, 1, 3]])) - 1.0) < 1e-12
    l = raw.astype(np.float64)
    assert abs(out[1] - (l[9] - math.log(math.exp(l[5]) + math.exp(l[9]) + math.exp(l[299])))) < 1e-12
    bad = oracle.allowed_renorm(raw, [3, -1, 300])
    assert np.isnan(bad[1]) and np.isnan(bad[2]) and bad[0] == 0.0


def test_p2_worked_example_round_trip():
    """Rebuild a row whose four head log-probabilities are the printed example; read them back."""
    vals = []
    for line in open(os.path.join(GOLDEN, "p2_top_logprobs_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        vals.append(float(line.split()[1]))
    assert len(vals) == 4
    V = 1000
    rest = 1.0 - sum(math.exp(v) for v in vals)
    assert 0.0068 < rest < 0.0070                     # the four printed entries hold 99.3% of the mass
    row = np.full(V, math.log(rest / (V - 4)), dtype=np.float64)
    ids = [400, 7, 655, 31]
    row[ids] = vals
    row32 = (row + 3.0).astype(f32)
    res = oracle.logprobs_row(row32, 400, 20)
    assert res["top_ids"][:4].tolist() == ids
    assert np.allclose(res["top_lps"][:4], vals, atol=2e-6)
    assert abs(res["chosen_lp"] - vals[0]) < 2e-6
    assert res["top_ids"][4] == 0                      # then the flat remainder, lowest index first


def test_logprobs_top_n_padding():
    res = oracle.logprobs_row(np.array([1.0, 2.0, 3.0], f32), 1, 5)
    assert res["top_ids"].tolist() == [2, 1, 0, -1, -1]
    assert np.isneginf(res["top_lps"][3:]).all()


def test_logprobs_chosen_outside_the_vocabulary():
    """An id outside [0, V) is no vocabulary entry and has no log-probability (NaN), at either end;
    the ends inside have the closed form log(e^l / sum e^l)."""
    row = np.array([1.0, 2.0, 3.0], f32)
    for c in (-1, -3, 3, 10):
        assert math.isnan(oracle.logprobs_row(row, c, 0)["chosen_lp"])
    z = math.log(math.e + math.e ** 2 + math.e ** 3)
    assert abs(oracle.logprobs_row(row, 0, 0)["chosen_lp"] - (1.0 - z)) < 1e-12
    assert abs(oracle.logprobs_row(row, 2, 0)["chosen_lp"] - (3.0 - z)) < 1e-12


# ----------------------------------------------------------------------------- full chain
def test_feature_visibility_config1():
    """Each feature of the single-row request changes the oracle's answer when it is switched on."""
    w = synth.config1()
    raw = oracle.widen(w["logits"][0, :w["V"]], "f32")
    p = Params.from_dict(w["slot_params"][0])
    hist = w["hist"]
    base = oracle.sample_row(raw, p, hist, 0, 0)
    # penalties: the forced spike id in the history loses its place in the order
    nopen = oracle.sample_row(raw, Params(**{**p.__dict__, "penalty_repeat": 1.0, "penalty_freq": 0.0,
                                             "penalty_present": 0.0}), hist, 0, 0)
    assert base["topk_ids"].tolist() != nopen["topk_ids"].tolist() or \
        not np.array_equal(base["topk_vals"], nopen["topk_vals"])
    # min_p: the cut keeps fewer survivors than top_k
    assert base["m1"] < p.k
    # greedy is the penalised argmax
    g = oracle.sample_row(raw, Params(**{**p.__dict__, "temperature": 0.0}), hist, 0, 0)
    assert g["id"] == base["topk_ids"][0]


def test_sampled_top_k_default_is_20():
    """top_k=0 on a sampled request means the sampler's own default of 20 survivors."""
    raw = np.linspace(5.0, -5.0, 100).astype(f32)
    r = oracle.sample_row(raw, Params(temperature=1.0, top_k=0, seed=3), None, 0, 0)
    assert r["topk_ids"].tolist() == list(range(20))
    assert Params(top_k=0).k == 20 and Params(top_k=7).k == 7
    assert oracle.sample_row(raw, Params(temperature=1.0, top_k=64, seed=3), None, 0, 0)["m1"] == 64


def test_feature_visibility_min_p_fixtures():
    """min_p at 0 / 0.5 / 0.9 gives three different kept counts on a graded row."""
    raw = np.array([3.0, 2.8, 2.5, 2.2, 1.9, 1.0, 0.0] + [-5.0] * 30, f32)
    m = [oracle.sample_row(raw, Params(temperature=1.0, top_k=20, min_p=mp, seed=1), None, 0, 0)["m1"]
         for mp in (0.0, 0.5, 0.9)]
    assert m[0] == 20 and m[0] > m[1] > m[2] >= 1


def test_invariants_random():
    rng = np.random.default_rng(21)
    for t in range(60):
        V = int(rng.integers(1, 300))
        raw = (rng.standard_normal(V) * 2).astype(f32)
        p = Params(temperature=float(rng.uniform(0.1, 2)), top_k=int(rng.integers(0, 65)),
                   top_p=float(rng.uniform(0, 1.2)), min_p=float(rng.uniform(0, 1.2)),
                   penalty_repeat=float(rng.uniform(0.5, 2)), penalty_freq=float(rng.uniform(-1, 1)),
                   penalty_present=float(rng.uniform(-1, 1)), penalty_last_n=int(rng.integers(0, 40)),
                   seed=int(rng.integers(0, 2**63)))
        hist = rng.integers(-3, V + 3, size=int(rng.integers(0, 50)))
        r = oracle.sample_row(raw, p, hist, t, 3)
        assert 1 <= r["m2"] <= r["m1"] <= min(p.k, V)
        assert r["id"] in r["topk_ids"][:r["m2"]].tolist()
        assert r["id"] == oracle.sample_row(raw, p, hist, t, 3)["id"]          # deterministic
        # top_k = 1 with no history is the greedy argmax
        p1 = Params(temperature=0.7, top_k=1, seed=p.seed)
        assert oracle.sample_row(raw, p1, None, t, 0)["id"] == int(np.argmax(raw))
        # neutral keys reproduce greedy byte for byte
        g = oracle.sample_row(raw, Params(), hist, t, 0)
        assert g["id"] == int(np.argmax(raw))


def test_seed_replay_and_counter_advance():
    w = synth.config1()
    raw = oracle.widen(w["logits"][0, :w["V"]], "f32")
    p = Params(temperature=1.5, top_k=64, top_p=1.0, seed=99)
    a = [oracle.sample_row(raw, p, None, 0, c)["id"] for c in range(64)]
    b = [oracle.sample_row(raw, p, None, 0, c)["id"] for c in range(64)]
    assert a == b                                           # same seed, same counters: same output
    assert len(set(a)) > 1                                  # the counter moves the draw
    p2 = Params(temperature=1.5, top_k=64, top_p=1.0, seed=100)
    assert [oracle.sample_row(raw, p2, None, 0, c)["id"] for c in range(64)] != a


def test_call_counter_semantics():
    """A call reads each slot's counter once and advances each sampled slot by exactly one."""
    w = synth.random_case(5, B=6, V=50, n_slots=3, sampled_frac=1.0)
    w["slot_params"][2]["temperature"] = 0.0               # slot 2 greedy: never advances
    w["row_slot"] = np.array([0, 0, 1, 2, 0, 1], np.int32)
    w["counters"] = {0: 10, 1: 0, 2: 5}
    rows, ctr = oracle.sample_call(w)
    assert ctr == {0: 11, 1: 1, 2: 5}
    rows2, _ = oracle.sample_call(w, counters={0: 10, 1: 0, 2: 5})
    assert [r["id"] for r in rows] == [r["id"] for r in rows2]
    for b in (0, 1, 4):
        p = Params.from_dict(w["slot_params"][0])
        assert rows[b]["u"] == row_uniform(p.seed, int(w["row_pos"][b]), 10)


def _chain_bruteforce(raw, p, hist, pos, ctr):
    """Second, loop-based formulation of the whole chain (float32 scalars, math.exp, k rounds)."""
    V = len(raw)
    counts = {}
    if hist is not None and p.penalty_last_n > 0:
        h = list(hist)[-p.penalty_last_n:] if p.penalty_last_n < len(hist) else list(hist)
        for t in h:
            if 0 <= t < V:
                counts[t] = counts.get(t, 0) + 1
    pen = [f32(x) for x in raw]
    r, fq, pr = f32(p.penalty_repeat), f32(p.penalty_freq), f32(p.penalty_present)
    for t, c in counts.items():
        x = pen[t]
        x = f32(x * r) if x <= 0 else f32(x / r)
        pen[t] = f32(x - f32(f32(f32(c) * fq) + pr))
    if p.greedy:
        return _argmax_rounds(pen, 1)[0], None
    k = min(20 if p.top_k == 0 else p.top_k, V)
    ids = _argmax_rounds(pen, k)
    vals = [pen[i] for i in ids]
    m1 = k
    if f32(p.min_p) > 0:
        thr = f32(vals[0] + oracle.c_logf(float(f32(p.min_p))))
        m1 = max(1, sum(1 for v in vals if v >= thr))
    tp = float(f32(p.top_p))
    if tp >= 1:
        m2 = m1
    elif tp <= 0:
        m2 = 1
    else:
        q = [math.exp(float(v) - float(vals[0])) for v in vals[:m1]]
        tot, acc, m2 = sum(q), 0.0, m1
        for i, x in enumerate(q):
            acc += x
            if acc / tot >= tp:
                m2 = i + 1
                break
    T = float(f32(p.temperature))
    wts = [math.exp((float(v) - float(vals[0])) / T) for v in vals[:m2]]
    W = sum(wts)
    u = row_uniform(p.seed, pos, ctr)
    acc, j = 0.0, m2 - 1
    for i, x in enumerate(wts):
        acc += x
        if acc > u * W:
            j = i
            break
    return ids[j], (ids, m1, m2)


@pytest.mark.parametrize("seed", range(30))
def test_chain_vs_bruteforce(seed):
    w = synth.random_case(seed, B=4, V=int(np.random.default_rng(seed).integers(2, 80)), n_slots=4,
                          sampled_frac=0.8, hist_len=30, ties=(seed % 2 == 0))
    rows, _ = oracle.sample_call(w)
    for b in range(w["B"]):
        s = int(w["row_slot"][b])
        p = Params.from_dict(w["slot_params"][s])
        raw = oracle.widen(w["logits"][b, :w["V"]], "f32")
        off = w["hist_off"]
        hist = w["hist"][off[s]:off[s + 1]]
        nb, extra = _chain_bruteforce(raw, p, hist if not oracle.sampling.penalties_neutral(p) else None,
                                      int(w["row_pos"][b]), w["counters"][s])
        r = rows[b]
        if extra is not None:
            ids, m1, m2 = extra
            assert r["topk_ids"].tolist() == ids
            assert r["m1"] == m1
            if not r["flag_top_p"]:
                assert r["m2"] == m2
        if not (r["flag_top_p"] or r["flag_draw"]):
            assert r["id"] == nb


def test_configs_generate_and_run():
    """The five workloads generate with the stated shapes; the small one runs through the oracle."""
    w1 = synth.config1()
    assert (w1["B"], w1["V"], w1["dtype"]) == (1, 32000, "f32")
    rows, ctr = oracle.sample_call(w1)
    assert ctr == {0: 1}
    assert rows[0]["top_ids"].size == 5
    w2 = synth.config2_window(3)
    assert (w2["B"], w2["V"]) == (5, 248320) and w2["counters"] == {0: 3}
    assert w2["row_pos"].tolist() == [115, 116, 117, 118, 119]
    w5 = synth.config5.__doc__
    assert "2048" in w5


# ---- verify-window acceptance ("#19 ...", "What changed"; "#559 ...", "Not done (yet)") --------
def test_accept_window_hand_cases():
    acc = oracle.accept_window
    # every draft matches: the whole window is kept, its last row's pick is the bonus token
    assert acc([0, 0, 0, 0, 0], [7, 8, 9, 10, 11], [7, 8, 9, 10, -1]) == {0: 5}
    # the first mismatch is kept (the target's own sample) and ends the window
    assert acc([0, 0, 0, 0, 0], [7, 8, 9, 10, 11], [7, 5, 9, 10, -1]) == {0: 2}
    assert acc([0, 0, 0, 0, 0], [7, 8, 9, 10, 11], [1, 8, 9, 10, -1]) == {0: 1}
    # a later match after a mismatch does not extend the window
    assert acc([0, 0, 0], [4, 5, 6], [4, 0, 6]) == {0: 2}
    # a lone row (no draft after it) keeps exactly one token
    assert acc([3], [42], [-1]) == {3: 1}
    # slots interleave; each slot's rows are its own window in row order
    assert acc([0, 1, 0, 1, 0, 1], [1, 2, 3, 4, 5, 6], [1, 2, 9, 4, -1, -1]) == {0: 2, 1: 3}
    # a pick of -1 (no candidate, out-of-range slot) never matches, even a -1 draft
    assert acc([0, 0], [-1, 3], [-1, -1]) == {0: 1}
    assert acc([0, 0], [-1, 3], [5, -1]) == {0: 1}


def test_accept_window_greedy_drafts_are_accepted():
    """Neutral greedy keys with drafts equal to each row's argmax (the textbook greedy pick): the
    whole window is accepted; one wrong draft at row j keeps j + 1 rows."""
    w = synth.config2_window(7)
    for s in w["slot_params"]:
        w["slot_params"][s] = synth.make_params(temperature=0.0, penalty_last_n=0)
    raw = [oracle.widen(w["logits"][b, :w["V"]], "f32") for b in range(w["B"])]
    argmax = [int(np.argmax(r)) for r in raw]
    drafts = argmax[:-1] + [-1]
    rows, ctr, keep = oracle.verify_call(w, drafts)
    assert [r["id"] for r in rows] == argmax
    assert keep == {0: w["B"]}
    assert ctr == w["counters"]                    # greedy slots draw nothing
    for j in range(w["B"] - 1):
        bad = list(drafts)
        bad[j] = (argmax[j] + 1) % w["V"]
        assert oracle.verify_call(w, bad)[2] == {0: j + 1}


def test_accept_window_sampled_counter_and_picks():
    """A sampled window keeps the target's own picks (the same rows as a plain call) and advances
    the slot's counter once."""
    w = synth.config2_window(2)
    rows_plain, ctr_plain = oracle.sample_call(w, with_allowed=False)
    picks = [r["id"] for r in rows_plain]
    rows, ctr, keep = oracle.verify_call(w, picks[:-1] + [-1])
    assert [r["id"] for r in rows] == picks
    assert ctr == ctr_plain == {0: w["counters"][0] + 1}
    assert keep == {0: w["B"]}


# ---- allowed_token_ids as a sampling mask ("#3200 ...", "Problem and result") ----------------
def _mask_params(**kw):
    return Params.from_dict(synth.make_params(**kw))


def test_mask_restricts_the_chain_to_the_named_ids():
    rng = np.random.default_rng(5)
    raw = (rng.standard_normal(500) * 3).astype(np.float32)
    top = int(np.argmax(raw))
    mask = [int(i) for i in rng.choice(np.delete(np.arange(500), top), 7, replace=False)]
    best_allowed = max(mask, key=lambda i: (raw[i], -i))
    g = oracle.sample_row(raw, _mask_params(temperature=0.0), None, 0, 0, mask)
    assert g["id"] == best_allowed                       # the greedy pick is the best named id
    s = oracle.sample_row(raw, _mask_params(temperature=1.3, top_k=64, top_p=1.0), None, 3, 0, mask)
    assert sorted(s["topk_ids"].tolist()) == sorted(mask)  # top_k larger than the mask: all of it
    assert s["topk_ids"][0] == best_allowed
    for c in range(200):
        r = oracle.sample_row(raw, _mask_params(temperature=2.0, top_k=64, top_p=1.0), None, 3, c, mask)
        assert r["id"] in mask
    one = oracle.sample_row(raw, _mask_params(temperature=0.9), None, 0, 0, [mask[3]])
    assert one["id"] == mask[3] and one["m1"] == one["m2"] == 1


def test_mask_edge_readings():
    rng = np.random.default_rng(6)
    raw = (rng.standard_normal(300) * 2).astype(np.float32)
    p = _mask_params(temperature=0.8, top_k=20, top_p=0.9, min_p=0.05, seed=11)
    plain = oracle.sample_row(raw, p, None, 7, 2)
    assert oracle.sample_row(raw, p, None, 7, 2, [])["id"] == plain["id"]          # empty: no mask
    assert oracle.sample_row(raw, p, None, 7, 2, None)["id"] == plain["id"]
    m = [5, 17, 17, -3, 300, 299, 5]                                               # dups, out of range
    a = oracle.sample_row(raw, p, None, 7, 2, m)
    b = oracle.sample_row(raw, p, None, 7, 2, [5, 17, 299])
    assert a["id"] == b["id"] and a["topk_ids"].tolist() == b["topk_ids"].tolist()
    none = oracle.sample_row(raw, p, None, 7, 2, [-1, 300, 1000])
    assert none["id"] == -1 and none.get("nocand")


def test_mask_keeps_the_penalties():
    """A named id in the history window is penalised inside the mask exactly as without it."""
    raw = np.array([1.0, 4.0, 3.9, -2.0, 0.5], np.float32)
    p = _mask_params(temperature=0.0, penalty_repeat=2.0, penalty_last_n=8)
    r = oracle.sample_row(raw, p, np.array([1], np.int32), 0, 0, [1, 2])
    assert r["id"] == 2                                  # 4.0 / 2 = 2.0 < 3.9
    assert oracle.sample_row(raw, p, None, 0, 0, [1, 2])["id"] == 1


# ---- per-slot histories kept between calls ("#19 ...", "min_p and the penalties") -------------
def _hw(rows, row_slot, params, pos=None):
    rows = np.asarray(rows, np.float32)
    pos = list(range(len(row_slot))) if pos is None else pos
    return synth._workload("ring_hand", "f32", rows.shape[1], rows, params, row_slot, pos, [], 0)


def _greedy_steps(raw, p, n):
    w = _hw([raw], [0], {0: p})
    state, ids = {}, []
    for _ in range(n):
        rows, _, state, keep = oracle.history_call(w, state)
        assert keep is None
        ids.append(rows[0]["id"])
    return ids, state


def test_history_hand_sequences():
    """Greedy decode of one fixed row, its picks fed back through the slot's history.

    repeat 2, freq 1 over a window of 8 (worked by hand): step 1 takes id 1 (4.0); step 2 sees
    id 1 at 4.0/2 - 1 = 1.0 and takes id 2 (3.9); step 3 sees 1.0 (id 1), 0.95 (id 2) and the
    untouched 1.0 of id 0, a tie that goes to the lower index, id 0; step 4: id 0 drops to
    1.0/2 - 1 = -0.5, id 1 is best at 1.0; step 5: id 1 counted twice, 2.0 - 2 = 0.0, id 2 at 0.95.
    A window of one id alternates the two best ids."""
    raw = [1.0, 4.0, 3.9, -2.0, 0.5]
    p = synth.make_params(temperature=0.0, penalty_repeat=2.0, penalty_freq=1.0, penalty_last_n=8)
    ids, state = _greedy_steps(raw, p, 5)
    assert ids == [1, 2, 0, 1, 2]
    assert state == {0: [1, 2, 0, 1, 2]}
    p1 = synth.make_params(temperature=0.0, penalty_repeat=2.0, penalty_freq=1.0, penalty_last_n=1)
    assert _greedy_steps(raw, p1, 6)[0] == [1, 2, 1, 2, 1, 2]
    p0 = synth.make_params(temperature=0.0, penalty_repeat=2.0, penalty_last_n=0)   # no penalty
    ids0, st0 = _greedy_steps(raw, p0, 3)
    assert ids0 == [1, 1, 1] and st0 == {0: [1, 1, 1]}                               # still recorded


def test_history_rows_of_one_call_share_the_window_and_append_in_row_order():
    a = [1.0, 4.0, 3.9, -2.0, 0.5]
    b = [0.0, 0.0, 0.0, 5.0, 0.0]
    p = synth.make_params(temperature=0.0, penalty_repeat=2.0, penalty_last_n=8)
    _, _, st, _ = oracle.history_call(_hw([a, b], [0, 0], {0: p}), {})
    assert st == {0: [1, 3]}
    _, _, st, _ = oracle.history_call(_hw([b, a], [0, 0], {0: p}), {})
    assert st == {0: [3, 1]}
    # both rows see the window from before the call: the second does not see the first's pick
    rows, _, st, _ = oracle.history_call(_hw([a, a], [0, 0], {0: p}), {})
    assert [r["id"] for r in rows] == [1, 1] and st == {0: [1, 1]}
    # the history given in the state is the window: id 1 penalised from the first call on
    rows, _, st, _ = oracle.history_call(_hw([a, a], [0, 0], {0: p}), {0: [9, 1]})
    assert [r["id"] for r in rows] == [2, 2] and st == {0: [9, 1, 2, 2]}
    # slots interleave; a slot without rows keeps its history untouched
    rows, _, st, _ = oracle.history_call(_hw([a, b, b], [1, 0, 1], {0: p, 1: p}), {0: [4], 2: [7]})
    assert st == {0: [4, 3], 1: [1, 3], 2: [7]}


def test_history_verify_appends_the_kept_rows_only():
    rows3 = [[0.0, 9.0, 0.0, 0.0], [0.0, 0.0, 9.0, 0.0], [0.0, 0.0, 0.0, 9.0]]   # argmax 1, 2, 3
    p = synth.make_params(temperature=0.0, penalty_last_n=0)
    w = _hw(rows3, [0, 0, 0], {0: p})
    _, _, st, keep = oracle.history_call(w, {0: [5]}, row_draft=[1, 2, -1])
    assert keep == {0: 3} and st == {0: [5, 1, 2, 3]}          # every draft matched: all + bonus
    _, _, st, keep = oracle.history_call(w, {0: [5]}, row_draft=[1, 0, -1])
    assert keep == {0: 2} and st == {0: [5, 1, 2]}             # the first miss is kept, then stop
    _, _, st, keep = oracle.history_call(w, {}, row_draft=[0, 2, -1])
    assert keep == {0: 1} and st == {0: [1]}


def test_history_no_pick_appends_nothing():
    raw = [1.0, 4.0, 3.9, -2.0, 0.5]
    p = synth.make_params(temperature=0.0, penalty_last_n=8)
    w = _hw([raw, raw], [0, 0], {0: p})
    w["allowed"], w["allowed_off"] = synth.csr([[-1, 99], [2]])
    rows, _, st, _ = oracle.history_call(w, {0: [3]}, mask_allowed=True)
    assert [r["id"] for r in rows] == [-1, 2] and st == {0: [3, 2]}


def test_history_matches_the_pages_upload_loop():
    """The pages' serve loop hands the sampler the request's last penalty_last_n tokens before
    every window; a kept history must give the same run (sampled rows, penalties, 40 steps)."""
    rng = np.random.default_rng(21)
    V = 64
    p = synth.make_params(temperature=0.9, top_k=12, top_p=0.95, min_p=0.02, penalty_repeat=1.4,
                          penalty_freq=0.3, penalty_present=0.2, penalty_last_n=6, seed=77)
    prompt = [int(x) for x in rng.integers(0, V, 9)]
    tokens = list(prompt)                 # the host's own record of the run
    state, ctr_a, ctr_b = {0: list(prompt)}, {0: 0}, {0: 0}
    for step in range(40):
        raw = (rng.standard_normal((1, V)) * 1.5).astype(np.float32)
        wa = synth._workload("loop", "f32", V, raw, {0: p}, [0], [step], [tokens[-6:]], 0)
        rows_a, ctr_a = oracle.sample_call(wa, counters=ctr_a)
        rows_b, ctr_b, state, _ = oracle.history_call(_hw(raw, [0], {0: p}, [step]), state, counters=ctr_b)
        assert rows_a[0]["id"] == rows_b[0]["id"]
        tokens.append(int(rows_a[0]["id"]))
    assert state[0] == tokens and ctr_a == ctr_b == {0: 40}
    assert len(set(tokens[len(prompt):])) > 5                    # the penalties moved the run around


def test_history_tail_capacity():
    st = {0: list(range(5000)), 1: [3, 4]}
    t, n = oracle.history_tail(st, 0)
    assert n == 5000 and t.tolist() == list(range(5000 - 4096, 5000))
    assert oracle.HISTORY_RING_CAP == 4096
    t, n = oracle.history_tail(st, 0, 10)
    assert t.tolist() == list(range(4990, 5000))
    t, n = oracle.history_tail(st, 0, 10 ** 6)                   # a ring of 4096 ids holds no more
    assert n == 5000 and t.tolist() == list(range(5000 - 4096, 5000))
    assert oracle.history_tail(st, 1)[0].tolist() == [3, 4]
    assert oracle.history_tail(st, 5)[0].size == 0 and oracle.history_tail(st, 5)[1] == 0
    assert oracle.history_tail(st, 1, 0)[0].size == 0


# ----------------------------------------------------------------------------- vocabulary shards
@pytest.mark.parametrize("seed", range(12))
def test_shard_records_merge_to_the_full_row(seed):
    """Splitting a row's vocabulary into slices, reporting each slice's record and merging them
    gives the full row's chain exactly: the same top_k list, cuts and pick, the same top_n
    alternatives and log-probabilities (to rounding of the log-sum-exp).  Ties straddle the cuts
    (values on a coarse grid) and history ids fall in every slice."""
    rng = np.random.default_rng(900 + seed)
    V = int(rng.integers(40, 400))
    raw = (np.round(rng.standard_normal(V) * 4) / 2).astype(f32)
    G = int(rng.integers(1, 5))
    cuts = np.sort(rng.choice(np.arange(1, V), size=G - 1, replace=False)).tolist()
    bounds = [0] + cuts + [V]
    hot = rng.integers(0, V, size=8)  # a few ids repeated, so counts above one matter
    hist = np.concatenate([rng.integers(0, V, size=int(rng.integers(0, 20))), rng.choice(hot, size=20)])
    p = Params(temperature=float(rng.choice([0.0, 0.7, 1.3])), top_k=int(rng.integers(0, 65)),
               top_p=float(rng.choice([1.0, 0.8])), min_p=float(rng.choice([0.0, 0.1])), penalty_repeat=1.5,
               penalty_freq=0.3, penalty_present=0.2, penalty_last_n=32, seed=int(rng.integers(0, 2**40)))
    k = 1 if p.greedy else p.k
    recs = [oracle.shard_record(raw[bounds[i]:bounds[i + 1]], bounds[i], p, hist, k, 7) for i in range(G)]
    m = oracle.merge_records(recs, p, 77, 5, 7)
    r = oracle.sample_row(raw, p, hist, 77, 5)
    lr = oracle.logprobs_row(raw, r["id"], 7)
    assert m["topk_ids"].tolist() == r["topk_ids"].tolist()
    assert m["m1"] == r["m1"] and m["m2"] == r["m2"] and m["id"] == r["id"]
    assert m["top_ids"].tolist() == lr["top_ids"].tolist()
    fin = np.isfinite(lr["top_lps"])
    assert np.max(np.abs(m["top_lps"][fin] - lr["top_lps"][fin]), initial=0.0) < 1e-12
    assert abs(m["chosen_lp"] - lr["chosen_lp"]) < 1e-12


def test_shard_record_hand_case():
    """Two slices of [3, 1, 4, 1 | 5, 9, 2, 6]: the second slice's best raw entries are 9 (id 5)
    and 6 (id 7); with repeat 2 over a history naming id 5 twice, its penalised 9 becomes 4.5, so
    the slice's best penalised entries are 6 (id 7) and 5 (id 4)."""
    raw = np.array([3, 1, 4, 1, 5, 9, 2, 6], dtype=f32)
    p = Params(temperature=1.0, top_k=2, penalty_repeat=2.0, penalty_last_n=8)
    r1 = oracle.shard_record(raw[4:], 4, p, [5, 5, 1], 2, 2)
    assert [(v, t) for v, t, _ in r1["pen"]] == [(6.0, 7), (5.0, 4)]
    assert r1["raw"] == [(9.0, 5), (6.0, 7)]
    assert abs(r1["lse"] - math.log(math.exp(5) + math.exp(9) + math.exp(2) + math.exp(6))) < 1e-12
