"""The C-ABI library builds, loads and exports every function include/strata_sample.h declares,
and its host-only logic (key validation, defaults, struct layout) behaves as documented.  No GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "strata_sample.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(strata_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def S():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_strata_build", os.path.join(ROOT, "request_token_sampling_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build_library()
    import request_token_sampling_gb300 as S
    return S


def test_every_declared_symbol_is_exported(S):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(S.lib, n), n
    assert set(names) == set(S._binding.EXPORTED)
    # and the binding exposes each under the same name
    for n in names:
        assert callable(getattr(S, n)), n


def test_struct_layout_matches_header(S):
    p = S.strata_sampling_params
    assert ctypes.sizeof(p) == 48
    assert p.seed.offset == 40 and p.penalty_last_n.offset == 32 and p.temperature.offset == 4


def test_defaults(S):
    d = S.strata_default_params()
    assert d == dict(temperature=0.0, top_k=0, top_p=1.0, min_p=0.0, penalty_repeat=1.0, penalty_freq=0.0,
                     penalty_present=0.0, penalty_last_n=64, seed=0)
    assert S.strata_validate_params(d) == 0


@pytest.mark.parametrize("over,ok", [
    (dict(top_k=64), True), (dict(top_k=65), False), (dict(top_k=-1), False), (dict(top_k=0), True),
    (dict(temperature=float("nan")), False), (dict(temperature=-3.0), True),
    (dict(top_p=float("inf")), False), (dict(min_p=-0.1), False), (dict(min_p=2.0), True),
    (dict(penalty_repeat=0.0), False), (dict(penalty_repeat=-1.0), False), (dict(penalty_repeat=1e-3), True),
    (dict(penalty_freq=-2.0), True), (dict(penalty_last_n=4096), True), (dict(penalty_last_n=4097), False),
    (dict(penalty_last_n=-1), False), (dict(seed=2**64 - 1), True),
])
def test_validation_rules(S, over, ok):
    p = dict(S.strata_default_params(), **over)
    rc = S.strata_validate_params(p)
    assert (rc == 0) == ok, (over, S.lib.strata_last_error())
    if not ok:
        assert rc == S.STRATA_EINVAL and S.lib.strata_last_error()


def test_struct_size_rules(S):
    c = S.strata_sampling_params()
    S.lib.strata_default_params(ctypes.byref(c))
    c.struct_size = 40
    assert S.lib.strata_validate_params(ctypes.byref(c)) == S.STRATA_EINVAL
    c.struct_size = 64                                 # a newer caller's larger struct is accepted
    assert S.lib.strata_validate_params(ctypes.byref(c)) == 0
    c.struct_size = 48
    c.reserved = 1
    assert S.lib.strata_validate_params(ctypes.byref(c)) == S.STRATA_EINVAL


def test_create_without_gpu_fails_cleanly(S):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(S.StrataError) as ei:
        S.strata_create(0, 4, 1000, 4)
    assert ei.value.code == S.STRATA_ECUDA


def test_null_arguments_rejected_without_cuda(S):
    assert S.lib.strata_sample_rows(None, None, 0, 1, 10, 10, None, None, None, None, 0, None, 0, None, None, None,
                                    None, None, None, None, None, None, 0, None) == S.STRATA_EINVAL
    assert S.lib.strata_read_errors(None, None, None) == S.STRATA_EINVAL
    assert S.lib.strata_history_enable(None) == S.STRATA_EINVAL
    assert S.lib.strata_history_set(None, 0, None, 0, None) == S.STRATA_EINVAL
    assert S.lib.strata_history_get(None, 0, None, 0, None, None, None) == S.STRATA_EINVAL
    assert S.lib.strata_shard_rows(None, None, 0, 1, 10, 10, 0, None, None, None, 0, 0, None, 0, None) == S.STRATA_EINVAL
    assert S.lib.strata_merge_shards(None, None, 1, 1, None, None, None, 0, None, None, None, None, None, None, 0,
                                     None) == S.STRATA_EINVAL
    S.lib.strata_destroy(None)


def test_record_layout_constants(S):
    """A slice record holds the header, 64 penalised entries of 16 bytes and 20 raw keys of 8."""
    from request_token_sampling_gb300 import sharded
    assert sharded.REC_RAW + 8 * S.STRATA_MAX_TOP_N <= S.STRATA_SHARD_RECORD_BYTES
    assert sharded.REC_PEN == 16 and sharded.REC_RAW == 16 + 16 * S.STRATA_MAX_TOP_K
    assert S.STRATA_SHARD_RECORD_BYTES % 16 == 0


def test_history_capacity_constants(S):
    import oracle
    text = open(HEADER).read()
    cap = int(re.search(r"#define STRATA_HISTORY_CAP\s+(\d+)", text).group(1))
    assert cap == S.STRATA_HISTORY_CAP == oracle.HISTORY_RING_CAP
    assert cap & (cap - 1) == 0                         # a power of two: ring positions are masked
    assert cap >= S.STRATA_MAX_PENALTY_LAST_N           # every penalty window fits


def test_header_constants_match_the_binding(S):
    """Every integer constant the header defines has the same value under the same name in Python."""
    text = open(HEADER).read()
    found = 0
    for name, expr in re.findall(r"^#define (STRATA_[A-Z0-9_]+)[ \t]+([^/\n]+)", text, flags=re.M):
        expr = expr.strip()
        if name == "STRATA_SAMPLE_H" or "(n)" in name or not expr:
            continue
        value = eval(re.sub(r"(0x[0-9A-Fa-f]+|\d+)u\b", r"\1", expr))  # integer literals and shifts only
        assert getattr(S, name) == value, name
        found += 1
    assert found >= 30
    assert S.STRATA_FLAG_SPLIT(5) == 5 << 8
