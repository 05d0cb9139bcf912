"""Guard words around every output buffer (compute-sanitizer stands in for nothing here): each call
writes its outputs between sentinel words that must come back untouched, over ragged shapes, both
logit types, forced splits, pipelined flags and every entry point."""
import numpy as np
import pytest

import synth

from _harness import set_slots, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

G = 64                     # guard words on each side
SENT_I = 0x5A5A5A5A        # int32 sentinel
SENT_F = -1.2345e-33       # float32 sentinel (a value no output takes)


@pytest.fixture(scope="module")
def sampler():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from request_token_sampling_gb300 import Sampler
    s = Sampler(device=0, max_slots=16, max_vocab=synth.V_FULL, max_rows=64)
    yield s
    s.close()


class Guarded:
    """Output tensors, each a view into a larger buffer with G sentinel words on either side."""

    def __init__(self):
        self.bufs = {}

    def make(self, name, shape, dtype):
        n = int(np.prod(shape)) if shape else 1
        if dtype == torch.int32:
            buf = torch.full((n + 2 * G,), SENT_I, dtype=torch.int32, device="cuda:0")
        else:
            buf = torch.full((n + 2 * G,), SENT_F, dtype=torch.float32, device="cuda:0")
        self.bufs[name] = (buf, n)
        return buf[G:G + n].view(*shape) if shape else buf[G:G + n]

    def check(self):
        torch.cuda.synchronize()
        for name, (buf, n) in self.bufs.items():
            b = buf.cpu().numpy()
            lo, hi = b[:G], b[G + n:]
            if buf.dtype == torch.int32:
                assert (lo == SENT_I).all() and (hi == SENT_I).all(), f"{name}: guard words overwritten"
            else:
                assert (lo.view(np.uint32) == np.float32(SENT_F).view(np.uint32)).all(), f"{name}: low guard"
                assert (hi.view(np.uint32) == np.float32(SENT_F).view(np.uint32)).all(), f"{name}: high guard"


CASES = [
    dict(seed=1, B=5, V=4099, dtype="f32", split=0, flags=0),
    dict(seed=2, B=3, V=70001, dtype="bf16", split=3, flags=0),
    dict(seed=3, B=8, V=synth.V_FULL, dtype="f32", split=0, flags=3),
    dict(seed=4, B=2, V=17, dtype="f32", split=1, flags=0),
    dict(seed=5, B=6, V=20011, dtype="bf16", split=16, flags=1),
]


@pytest.mark.parametrize("case", CASES, ids=[f"V{c['V']}_{c['dtype']}_s{c['split']}_f{c['flags']}" for c in CASES])
def test_sample_outputs_stay_inside_their_buffers(sampler, case):
    from request_token_sampling_gb300 import STRATA_FLAG_SPLIT
    B, V = case["B"], case["V"]
    w = synth.random_case(case["seed"], B=B, V=V, dtype=case["dtype"], ld=V + (-V % 8) + 8, n_slots=3,
                          sampled_frac=0.7, hist_len=64, top_n=7, allowed_sizes=[0, 3, 40])
    set_slots(sampler, w)
    d = upload(w)
    g = Guarded()
    n_allowed = int(w["allowed_off"][-1])
    out = {"ids": g.make("ids", (B,), torch.int32), "chosen_lp": g.make("chosen_lp", (B,), torch.float32),
           "top_ids": g.make("top_ids", (B, 7), torch.int32), "top_lps": g.make("top_lps", (B, 7), torch.float32),
           "allowed_lps": g.make("allowed_lps", (max(1, n_allowed),), torch.float32),
           "topk_ids": g.make("topk_ids", (B, 64), torch.int32), "topk_vals": g.make("topk_vals", (B, 64), torch.float32),
           "kept": g.make("kept", (B, 2), torch.int32)}
    sampler.sample(d["logits"], d["row_slot"], d["row_pos"], V=V, hist=d["hist"], hist_off=d["hist_off"], top_n=7,
                   chosen_lp=True, allowed=d["allowed"], allowed_off=d["allowed_off"], debug=True,
                   flags=case["flags"] | STRATA_FLAG_SPLIT(case["split"]), out=out)
    g.check()
    ids = out["ids"].cpu().numpy()
    assert ((ids >= 0) & (ids < V)).all()


def test_verify_and_logprobs_outputs_stay_inside_their_buffers(sampler):
    w = synth.config2_window(3)
    set_slots(sampler, w)
    d = upload(w)
    g = Guarded()
    drafts = torch.tensor([1, 2, 3, 4, -1], dtype=torch.int32, device="cuda:0")
    out = {"ids": g.make("ids", (w["B"],), torch.int32), "keep": g.make("keep", (16,), torch.int32),
           "chosen_lp": g.make("chosen_lp", (w["B"],), torch.float32)}
    out["keep"].fill_(-1)
    sampler.verify(d["logits"], d["row_slot"], d["row_pos"], drafts, V=w["V"], hist=d["hist"], hist_off=d["hist_off"],
                   chosen_lp=True, out=out)
    g.check()
    w4 = synth.config4(fused=False)
    d4 = upload(w4)
    g4 = Guarded()
    n_allowed = int(w4["allowed_off"][-1])
    out4 = {"chosen_lp": g4.make("chosen_lp", (w4["B"],), torch.float32),
            "top_ids": g4.make("top_ids", (w4["B"], w4["top_n"]), torch.int32),
            "top_lps": g4.make("top_lps", (w4["B"], w4["top_n"]), torch.float32),
            "allowed_lps": g4.make("allowed_lps", (n_allowed,), torch.float32)}
    sampler.logprobs(d4["logits"], V=w4["V"], chosen=d4["chosen"], top_n=w4["top_n"], allowed=d4["allowed"],
                     allowed_off=d4["allowed_off"], out=out4)
    g4.check()
