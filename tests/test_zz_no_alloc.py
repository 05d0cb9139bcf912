"""The allocation-free entry point gives the same results as the context-based call and the oracle.

strata_sample_rows_noalloc exists for callers that cannot call cudaMalloc (a framework whose
allocator owns all device memory, a server that must not grow its device footprint).  It keeps its
per-row key records, counter words and error word in a static device array instead of a context.
This test runs the same rows through both entry points, two calls in a row (the caller advances
the counters of sampled rows between calls, as the context does on the device), and requires equal
ids and log-probabilities within the tolerance of the other parity tests.  Both calls' rows are also
checked against the CPU oracle with the counters the test supplies (a greedy row, top_k 64 with
neutral cuts, top_k 0 meaning 20, a counter above 2^40).  It lives in a file of its own, collected
last.
"""
import numpy as np
import pytest

import oracle
import synth
from _harness import Stats, compare_sample

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LP_TOL = 1e-5


def _case():
    w = synth.config4(fused=True)
    # a mix of greedy and sampled rows, penalties on some, different top_k
    w["slot_params"][1] = dict(w["slot_params"][1], temperature=0.0)
    w["slot_params"][5] = dict(w["slot_params"][5], top_k=64, top_p=1.0, min_p=0.0, penalty_repeat=1.0,
                               penalty_freq=0.0, penalty_present=0.0)
    w["slot_params"][6] = dict(w["slot_params"][6], top_k=0, temperature=1.3)
    return w


def test_noalloc_matches_context_call_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import request_token_sampling_gb300 as S
    from request_token_sampling_gb300 import Sampler
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = _case()
    B, V = w["B"], w["V"]
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    logits, row_pos = T(w["logits"]), T(w["row_pos"])
    hist, hist_off = T(w["hist"]), T(w["hist_off"])
    params = [w["slot_params"][b] for b in range(B)]
    sampled = [p["temperature"] > 0 for p in params]
    start = [3, 0, 17, 2**40, 5, 9, 11, 0]

    with Sampler(device=0, max_slots=B, max_vocab=V, max_rows=B) as s:
        for b in range(B):
            s.restore_slot(b, params[b], start[b])
        ref = []
        for _ in range(2):
            o = s.sample(logits, T(w["row_slot"]), row_pos, hist=hist, hist_off=hist_off, top_n=20, chosen_lp=True)
            torch.cuda.synchronize()
            ref.append({k: v.cpu().numpy() for k, v in o.items()})
        assert s.errors() == 0

    counters = list(start)
    got = []
    free0 = None
    for call in range(2):
        out = {"ids": torch.full((B,), -7, dtype=torch.int32, device=dev),
               "chosen_lp": torch.empty(B, dtype=torch.float32, device=dev),
               "top_ids": torch.empty(B, 20, dtype=torch.int32, device=dev),
               "top_lps": torch.empty(B, 20, dtype=torch.float32, device=dev)}
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info(dev)[0]
        S.strata_sample_rows_noalloc(logits, params, counters, row_pos, out["ids"], hist=hist, hist_off=hist_off,
                                     top_n=20, chosen_lp=out["chosen_lp"], top_ids=out["top_ids"],
                                     top_lps=out["top_lps"])
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info(dev)[0] == free_before   # the call grew nothing
        got.append({k: v.cpu().numpy() for k, v in out.items()})
        counters = [c + 1 if sm else c for c, sm in zip(counters, sampled)]

    st = Stats()
    counters = {b: start[b] for b in range(B)}
    for call in range(2):
        rows, counters = oracle.sample_call(w, counters=counters)
        compare_sample(w, rows, got[call], top_n=20, stats=st, debug=False)
    assert st.rows == 2 * B
    for call in range(2):
        assert np.array_equal(got[call]["ids"], ref[call]["ids"]), call
        assert np.array_equal(got[call]["top_ids"], ref[call]["top_ids"]), call
        assert np.max(np.abs(got[call]["chosen_lp"] - ref[call]["chosen_lp"])) <= LP_TOL
        assert np.max(np.abs(got[call]["top_lps"] - ref[call]["top_lps"])) <= LP_TOL


def test_noalloc_rejects_too_many_rows():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import request_token_sampling_gb300 as S
    B = S.STRATA_NOALLOC_MAX_ROWS + 1
    x = torch.zeros((B, 64), dtype=torch.float32, device="cuda:0")
    with pytest.raises(S.StrataError) as ei:
        S.strata_sample_rows_noalloc(x, [synth.make_params()] * B, [0] * B,
                                     torch.zeros(B, dtype=torch.int64, device="cuda:0"),
                                     torch.zeros(B, dtype=torch.int32, device="cuda:0"))
    assert ei.value.code == S.STRATA_ERANGE
    assert "static scratch" in S.strata_last_error()
