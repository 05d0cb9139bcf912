"""Planted mistakes in a copy of the oracle must each fail the pin suite (CPU only).

Every mutation below is a plausible slip in writing the chain down (a swapped branch, a dropped
or extra term, a flipped sign or comparison, a wrong index or word, the cuts in the wrong order).
The test copies ``oracle/``, ``synth/`` and ``tests/`` to a temporary folder, plants one mistake,
runs ``test_oracle_pins.py`` there and requires it to fail.  Nothing here touches a GPU.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("sampling.py", "x * r32, x / r32", "x / r32, x * r32"),
    ("sampling.py", "np.where(c > 0, p32, np.float32(0))", "c.astype(np.float32) * p32"),
    ("sampling.py", "(x - sub)", "(x + sub)"),
    ("sampling.py", "window = hist_ids[hist_ids.size - h:]", "window = hist_ids[:h]"),
    ("sampling.py", "np.lexsort((idx, -v))", "np.lexsort((-idx, -v))"),
    ("sampling.py", "sel.astype(np.float32) >= np.float32(thr)", "sel.astype(np.float32) > np.float32(thr)"),
    ("sampling.py", "thr = np.float32(sel[0]) + c_logf", "thr = np.float32(sel[0]) - c_logf"),
    ("sampling.py", "q = np.exp(v - v[0])", "q = np.exp((v - v[0]) / 0.7)"),
    ("sampling.py", "cum = np.cumsum(q) / np.sum(q)", "cum = np.cumsum(q[::-1])[::-1] / np.sum(q)"),
    ("sampling.py", "hit = np.nonzero(cum > u * W)[0]", "hit = np.nonzero(cum >= u * W)[0]"),
    ("sampling.py", "w = np.exp((v - v[0]) / float(np.float32(temperature)))",
     "w = np.exp((v - v[0]) * float(np.float32(temperature)))"),
    ("sampling.py", "lse = m + np.log(np.sum(np.exp(l - m)))", "lse = np.log(np.sum(np.exp(l - m)))"),
    ("sampling.py", "uniq = np.unique(a[ok])", "uniq = a[ok]"),
    ("sampling.py", "m1 = min_p_cut(sel, p.min_p)\n    m2, f_tp = top_p_cut(sel, m1, p.top_p)",
     "m2, f_tp = top_p_cut(sel, k, p.top_p)\n    m1 = min(m2, min_p_cut(sel, p.min_p)); m2 = m1"),
    ("sampling.py", "counters[s] = counters.get(s, 0) + 1", "counters[s] = counters.get(s, 0) + 2"),
    ("sampling.py", "return DEFAULT_SAMPLED_TOP_K if self.top_k == 0 else int(self.top_k)",
     "return int(self.top_k) or 1"),
    ("philox.py", "c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & MASK32, lo1, (hi0 ^ c3 ^ k1) & MASK32, lo0",
     "c0, c1, c2, c3 = (hi0 ^ c1 ^ k0) & MASK32, lo1, (hi1 ^ c3 ^ k1) & MASK32, lo0"),
    ("philox.py", "(position & MASK32, position >> 32, counter & MASK32, counter >> 32)",
     "(counter & MASK32, counter >> 32, position & MASK32, position >> 32)"),
    ("philox.py", "return (out[0] >> 8) * (2.0 ** -24)", "return (out[1] >> 8) * (2.0 ** -24)"),
    ("philox.py", "    for _ in range(10):", "    for _ in range(9):"),
    ("philox.py", "(seed & MASK32, seed >> 32))", "(seed >> 32, seed & MASK32))"),
    ("philox.py", "        k1 = (k1 + PHILOX_W32_1) & MASK32", "        k1 = (k1 + PHILOX_W32_0) & MASK32"),
    ("philox.py", "return (out[0] >> 8) * (2.0 ** -24)", "return (out[0] & 0xFFFFFF) * (2.0 ** -24)"),
    ("sampling.py", "        if not open_[s]:\n            continue\n", ""),
    ("sampling.py", "        keep[s] += 1\n        if d < 0 or t < 0 or t != d:\n            open_[s] = False",
     "        if d < 0 or t < 0 or t != d:\n            open_[s] = False\n        else:\n            keep[s] += 1"),
    ("sampling.py", "        order = keep[rank_order(pen[keep])]", "        order = rank_order(pen)[:keep.size]"),
    ("sampling.py", "        keep = np.unique(a[(a >= 0) & (a < V)])", "        keep = np.unique(np.clip(a, 0, V - 1))"),
    ("sampling.py", "        if keep is not None and taken[s] > keep.get(s, 0):\n            continue\n", ""),
    ("sampling.py", "if keep is not None and taken[s] > keep.get(s, 0):", "if keep is not None and taken[s] >= keep.get(s, 0):"),
    ("sampling.py", "        if t >= 0:\n            new.setdefault(s, []).append(t)", "        new.setdefault(s, []).append(t)"),
    ("sampling.py", "new.setdefault(s, []).append(t)", "new.setdefault(s, []).insert(len(state.get(s, [])), t)"),
    ("sampling.py", "np.asarray(h[len(h) - m:], dtype=np.int32)", "np.asarray(h[:m], dtype=np.int32)"),
    ("sampling.py", "astype(np.uint32) << 16).view(np.float32)", "astype(np.uint32) << 15).view(np.float32)"),
    ("sampling.py", "(np.asarray(row, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)",
     "np.asarray(row, dtype=np.uint16).view(np.float16).astype(np.float32)"),
    ("sampling.py", "if not (0 <= p.top_k <= MAX_TOP_K):", "if not (1 <= p.top_k <= MAX_TOP_K):"),
    ("sampling.py", "if not (np.float32(p.penalty_repeat) > 0):", "if not (np.float32(p.penalty_repeat) >= 0):"),
    ("sampling.py", "    if np.float32(p.min_p) < 0:\n        return False\n", ""),
    ("sampling.py", "lse = float(mx + np.log(np.sum(np.exp(lses - mx))))", "lse = float(mx)"),
    ("sampling.py", "pen = sorted((e for r in records for e in r[\"pen\"]), key=lambda e: (-e[0], e[1]))",
     "pen = sorted((e for r in records for e in r[\"pen\"]), key=lambda e: (-e[0], -e[1]))"),
    ("sampling.py", "            if t >= v0:\n                counts[t - v0] = c", "            if t >= v0:\n                counts[t - v0] = 1"),
    ("sampling.py", "res.update(id=int(order[0]), topk_ids=order[:1].copy()",
     "res.update(id=int(rank_order(raw32)[0]), topk_ids=order[:1].copy()"),
    ("sampling.py", "    if tp <= 0.0:\n        return 1, False", "    if tp <= 0.0:\n        return m1, False"),
    ("sampling.py", "lse_a = m + np.log(np.sum(np.exp(l[uniq] - m)))", "lse_a = m + np.log(np.sum(np.exp(l - m)))"),
    ("sampling.py", "        if 0 <= t < V:\n            counts[t]", "        if t < V:\n            counts[t]"),
    ("sampling.py", "np.float32(p.penalty_repeat) == 1 and np.float32(p.penalty_freq) == 0",
     "np.float32(p.penalty_repeat) == 1 or np.float32(p.penalty_freq) == 0"),
    ("sampling.py", "return dict(pen=[(float(pen[i]), v0 + int(i), float(raw[i])) for i in op],",
     "return dict(pen=[(float(pen[i]), int(i), float(raw[i])) for i in op],"),
    ("sampling.py", "    orr = rank_order(raw)[:top_n]", "    orr = rank_order(pen)[:top_n]"),
    ("sampling.py", "    order = rank_order(raw32)[:n]", "    order = rank_order(raw32)[1:n + 1]"),
    ("sampling.py", "    k = min(p.k, order.size)", "    k = min(p.k, order.size) - 1"),
    ("sampling.py", "lse = float(m + np.log(np.sum(np.exp(l - m)))) if n and",
     "lse = float(np.log(np.sum(np.exp(l - m)))) if n and"),
    ("sampling.py", "raw = sorted((e for r in records for e in r[\"raw\"]), key=lambda e: (-e[0], e[1]))",
     "raw = sorted((e for r in records for e in r[\"raw\"]), key=lambda e: (e[0], e[1]))"),
    ("sampling.py", "k = 1 if p.greedy else min(p.k, len(pen))", "k = min(p.k, len(pen))"),
    ("sampling.py", "        if not p.greedy:\n            sampled_slots.add(s)", "        sampled_slots.add(s)"),
    ("sampling.py", "int(w[\"row_pos\"][b]), counters.get(s, 0), mask)", "int(w[\"row_pos\"][b]), counters.get(s, 0) + b, mask)"),
    ("sampling.py", "        if d < 0 or t < 0 or t != d:", "        if t != d:"),
    ("sampling.py", "float(lp[chosen]) if 0 <= chosen < V else", "float(lp[chosen]) if chosen < V else"),
    ("sampling.py", "m = min(len(h), HISTORY_RING_CAP, max(0, int(max_n)))", "m = min(len(h), max(0, int(max_n)))"),
    ("sampling.py", "    m = np.max(l)\n    lse = m + np.log(np.sum(np.exp(l - m)))\n    return l - lse",
     "    m = np.max(l)\n    lse = m + np.log(np.sum(np.exp(l - m)))\n    return l - m"),
]


def _run_mutant(base, i):
    """Plant mutation i in a fresh copy and run the pin suite there: (anchor found, exit code)."""
    fn, old, new = MUTATIONS[i]
    d = base / f"m{i}"
    for sub in ("oracle", "synth", "tests"):
        shutil.copytree(os.path.join(ROOT, sub), d / sub, ignore=shutil.ignore_patterns("__pycache__", "*.pyc"))
    target = d / "oracle" / fn
    src = target.read_text()
    if old not in src:
        return False, None
    target.write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        str(d / "tests" / "test_oracle_pins.py")],
                       cwd=d, capture_output=True, text=True, timeout=600)
    return True, r.returncode


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every mutant's outcome, the pin suites run a few at a time (each is its own process)."""
    base = tmp_path_factory.mktemp("mutants")
    workers = max(1, min(8, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(lambda i: _run_mutant(base, i), range(len(MUTATIONS))))


@pytest.mark.parametrize("i", range(len(MUTATIONS)), ids=[f"{m[0]}:{i}" for i, m in enumerate(MUTATIONS)])
def test_planted_mistake_is_caught(outcomes, i):
    found, rc = outcomes[i]
    assert found, "mutation anchor vanished from the oracle"
    assert rc != 0, f"planted mistake survived: {MUTATIONS[i][2]!r}"
