"""The parity harness's rule for flagged rows, checked on the CPU with crafted oracle rows.

A row the oracle flags (a top_p or draw decision within 1e-6 of a boundary) may differ from the
oracle only across that boundary: the tests below build such rows by hand and require the harness
to accept the neighbouring pick and to reject any other id.
"""
import numpy as np
import pytest

from _harness import check_flagged_pick

f32 = np.float32


def _row(vals, m1, m2, u, flag_top_p=False, flag_draw=False, ids=(7, 3, 11, 5)):
    import oracle
    sel = np.asarray(vals, f32)
    j, _ = oracle.draw_index(sel, m2, 1.0, u)
    ids = np.asarray(ids[:sel.size], np.int64)
    return dict(topk_ids=ids, topk_vals=sel, m1=m1, m2=m2, u=u, j=j, id=int(ids[j]),
                flag_top_p=flag_top_p, flag_draw=flag_draw)


W = {"slot_params": {0: {"temperature": 1.0, "top_p": 1.0}}, "row_slot": np.zeros(1, np.int32)}


def test_draw_boundary_accepts_only_the_neighbour():
    vals = [2.0, 1.0, 0.0]
    w = np.exp(np.asarray(vals, np.float64) - 2.0)
    c0 = w[0] / w.sum()
    r = _row(vals, 3, 3, c0 + 5e-7, flag_draw=True)
    assert r["j"] == 1
    check_flagged_pick(W, 0, r, 3, 3)          # the oracle's own pick
    check_flagged_pick(W, 0, r, 7, 3)          # the survivor across the boundary
    with pytest.raises(AssertionError):
        check_flagged_pick(W, 0, r, 11, 3)     # two places away
    with pytest.raises(AssertionError):
        check_flagged_pick(W, 0, r, 99, 3)     # not a survivor at all


def test_top_p_boundary_allows_one_more_or_less_survivor():
    import oracle
    vals = [2.0, 1.0, 0.0, -1.0]
    q = np.exp(np.asarray(vals, np.float64) - 2.0)
    top_p = float(f32(q[:2].sum() / q.sum()))             # the cut sits on the second survivor's mass
    m2, flag = oracle.top_p_cut(np.asarray(vals, f32), 4, top_p)
    assert flag and m2 in (2, 3)
    w = {"slot_params": {0: {"temperature": 1.0, "top_p": top_p}}, "row_slot": np.zeros(1, np.int32)}
    r = _row(vals, 4, 2, 0.97, flag_top_p=True)
    # the GPU kept one survivor more: its pick must be the draw's decision over three survivors
    j3, _ = oracle.draw_index(np.asarray(vals, f32), 3, 1.0, 0.97)
    check_flagged_pick(w, 0, r, int(r["topk_ids"][j3]), 3)
    check_flagged_pick(w, 0, r, int(r["topk_ids"][j3]))         # without the debug count
    with pytest.raises(AssertionError):
        check_flagged_pick(w, 0, r, int(r["topk_ids"][3]), 3)    # outside the kept set
    with pytest.raises(AssertionError):
        check_flagged_pick(w, 0, r, int(r["topk_ids"][0]), 4)    # two more survivors than the cut allows


def test_unflagged_top_p_count_must_match():
    vals = [2.0, 1.0, 0.0]
    w = np.exp(np.asarray(vals, np.float64) - 2.0)
    r = _row(vals, 3, 2, w[0] / w[:2].sum() + 5e-7, flag_draw=True)
    with pytest.raises(AssertionError):
        check_flagged_pick(W, 0, r, r["id"], 3)
