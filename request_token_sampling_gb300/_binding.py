"""ctypes binding of the strata_sample C ABI (include/strata_sample.h).

Argument marshalling only: every step of sampling runs in the library's CUDA kernel.  PyTorch is
used for device memory and streams: tensors are passed by ``data_ptr()`` and the stream by its
``cuda_stream`` handle.  The functions keep the C names.  There is no fallback: if the shared
library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .build import LIB_PATH

STRATA_OK = 0
STRATA_EINVAL = -1
STRATA_EALIGN = -2
STRATA_ERANGE = -3
STRATA_ECUDA = -4
STRATA_ENOMEM = -5

STRATA_DTYPE_F32 = 0
STRATA_DTYPE_BF16 = 1

STRATA_MAX_TOP_K = 64
STRATA_DEFAULT_TOP_K = 20
STRATA_DEFAULT_LAST_N = 64
STRATA_MAX_TOP_N = 20
STRATA_MAX_PENALTY_LAST_N = 4096
STRATA_MAX_VOCAB = 524288
STRATA_NOALLOC_MAX_ROWS = 1024
STRATA_HISTORY_CAP = 4096
STRATA_MAX_SHARDS = 16
STRATA_SHARD_RECORD_BYTES = 1280

STRATA_FLAG_PDL = 0x1
STRATA_FLAG_EARLY_LOAD = 0x2
STRATA_FLAG_ALLOWED_MASK = 0x4
STRATA_FLAG_HISTORY_RING = 0x8
STRATA_FLAG_CONCURRENT = 0x10
STRATA_FLAG_OWN_OUTPUTS = 0x20
STRATA_FLAG_RESIDENT = 0x40
STRATA_CONCURRENT_ROW_BYTES = 1 << 19
STRATA_FLAG_TEST_STALL = 0x10000


def STRATA_FLAG_SPLIT(n: int) -> int:
    return (int(n) & 0x1F) << 8


STRATA_DEVERR_SLOT = 0x01
STRATA_DEVERR_ALLOWED = 0x02
STRATA_DEVERR_CHOSEN = 0x04
STRATA_DEVERR_TIMEOUT = 0x08
STRATA_DEVERR_NOCAND = 0x10
STRATA_DEVERR_HISTORY = 0x20
STRATA_DEVERR_SHAPE = 0x40

EXPORTED = (
    "strata_version", "strata_last_error", "strata_default_params", "strata_validate_params",
    "strata_create", "strata_destroy", "strata_set_slot_params", "strata_get_slot_state",
    "strata_set_slot_state", "strata_sample_rows", "strata_logprobs_rows", "strata_read_errors",
    "strata_launch_shape", "strata_sample_rows_noalloc", "strata_sample_verify", "strata_history_enable",
    "strata_history_set", "strata_history_get", "strata_shard_rows", "strata_merge_shards",
)


class strata_sampling_params(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("temperature", ctypes.c_float),
        ("top_k", ctypes.c_int32),
        ("top_p", ctypes.c_float),
        ("min_p", ctypes.c_float),
        ("penalty_repeat", ctypes.c_float),
        ("penalty_freq", ctypes.c_float),
        ("penalty_present", ctypes.c_float),
        ("penalty_last_n", ctypes.c_int32),
        ("reserved", ctypes.c_uint32),
        ("seed", ctypes.c_uint64),
    ]


PARAM_KEYS = ("temperature", "top_k", "top_p", "min_p", "penalty_repeat", "penalty_freq",
              "penalty_present", "penalty_last_n", "seed")


class StrataError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"strata error {code}: {message}")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"the CUDA sampler library is not built ({LIB_PATH}); "
                          "run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, u32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_int64
    P = ctypes.POINTER(strata_sampling_params)
    sig = {
        "strata_version": ([], i32),
        "strata_last_error": ([], ctypes.c_char_p),
        "strata_default_params": ([P], None),
        "strata_validate_params": ([P], i32),
        "strata_create": ([ctypes.POINTER(vp), i32, i32, i32, i32], i32),
        "strata_destroy": ([vp], None),
        "strata_set_slot_params": ([vp, i32, P, i32, vp], i32),
        "strata_get_slot_state": ([vp, i32, P, ctypes.POINTER(ctypes.c_uint64), vp], i32),
        "strata_set_slot_state": ([vp, i32, P, ctypes.c_uint64, vp], i32),
        "strata_sample_rows": ([vp, vp, i32, i32, i32, i64, vp, vp, vp, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp,
                                vp, vp, vp, u32, vp], i32),
        "strata_logprobs_rows": ([vp, vp, i32, i32, i32, i64, vp, vp, i32, vp, vp, vp, vp, vp, u32, vp], i32),
        "strata_sample_verify": ([vp, vp, i32, i32, i32, i64, vp, vp, vp, vp, vp, i32, vp, vp, i32, vp, vp, vp, u32,
                                  vp], i32),
        "strata_read_errors": ([vp, ctypes.POINTER(ctypes.c_uint32), vp], i32),
        "strata_launch_shape": ([vp, i32, i32, i32, i32, i32, u32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                 ctypes.POINTER(i32), ctypes.POINTER(i32)], i32),
        "strata_sample_rows_noalloc": ([vp, i32, i32, i32, i64, P, ctypes.POINTER(ctypes.c_uint64), vp, vp, vp, vp,
                                        i32, vp, vp, vp, vp], i32),
        "strata_history_enable": ([vp], i32),
        "strata_history_set": ([vp, i32, vp, i64, vp], i32),
        "strata_history_get": ([vp, i32, vp, i32, ctypes.POINTER(i32), ctypes.POINTER(i64), vp], i32),
        "strata_shard_rows": ([vp, vp, i32, i32, i32, i64, i32, vp, vp, vp, i32, i32, vp, u32, vp], i32),
        "strata_merge_shards": ([vp, vp, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, u32, vp], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def _check(rc: int) -> None:
    if rc != STRATA_OK:
        raise StrataError(rc, lib.strata_last_error().decode(errors="replace"))


def _ptr(t) -> Optional[int]:
    """Device address of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _typed(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return _ptr(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def to_c_params(p) -> strata_sampling_params:
    c = strata_sampling_params()
    lib.strata_default_params(ctypes.byref(c))
    if isinstance(p, strata_sampling_params):
        return p
    for k in PARAM_KEYS:
        if k in p:
            setattr(c, k, p[k])
    return c


def from_c_params(c: strata_sampling_params) -> dict:
    return {k: getattr(c, k) for k in PARAM_KEYS}


# ------------------------------------------------------------------------------ C-named calls
def strata_version() -> int:
    return lib.strata_version()


def strata_last_error() -> str:
    return lib.strata_last_error().decode(errors="replace")


def strata_default_params() -> dict:
    c = strata_sampling_params()
    lib.strata_default_params(ctypes.byref(c))
    return from_c_params(c)


def strata_validate_params(p) -> int:
    c = to_c_params(p)
    return lib.strata_validate_params(ctypes.byref(c))


def strata_create(device: int = 0, max_slots: int = 64, max_vocab: int = 262144, max_rows: int = 1024):
    h = ctypes.c_void_p()
    _check(lib.strata_create(ctypes.byref(h), device, max_slots, max_vocab, max_rows))
    return h


def strata_destroy(ctx) -> None:
    lib.strata_destroy(ctx)


def strata_set_slot_params(ctx, slot: int, params, reset_counter: bool = False, stream=None) -> None:
    c = to_c_params(params)
    _check(lib.strata_set_slot_params(ctx, slot, ctypes.byref(c), int(bool(reset_counter)), _stream(stream)))


def strata_get_slot_state(ctx, slot: int, stream=None):
    c = strata_sampling_params()
    ctr = ctypes.c_uint64()
    _check(lib.strata_get_slot_state(ctx, slot, ctypes.byref(c), ctypes.byref(ctr), _stream(stream)))
    return from_c_params(c), int(ctr.value)


def strata_set_slot_state(ctx, slot: int, params, counter: int, stream=None) -> None:
    c = to_c_params(params)
    _check(lib.strata_set_slot_state(ctx, slot, ctypes.byref(c), ctypes.c_uint64(counter), _stream(stream)))


def _logits_args(logits, V):
    import torch
    if logits.dim() != 2:
        raise ValueError("logits must be [B, ld]")
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    if logits.dtype == torch.float32:
        dt = STRATA_DTYPE_F32
    elif logits.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        dt = STRATA_DTYPE_BF16
    else:
        raise TypeError(f"unsupported logits dtype {logits.dtype}")
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    V = logits.shape[1] if V is None else int(V)
    return logits.data_ptr(), dt, int(logits.shape[0]), V, int(logits.stride(0))


def strata_sample_rows(ctx, logits, row_slot, row_pos, out_ids, V=None, hist=None, hist_off=None,
                       top_n: int = 0, chosen_lp=None, top_ids=None, top_lps=None, allowed=None,
                       allowed_off=None, allowed_lps=None, topk_ids=None, topk_vals=None, kept=None,
                       flags: int = 0, stream=None) -> None:
    import torch
    ptr, dt, B, V, ld = _logits_args(logits, V)
    n_hist = 0 if hist_off is None else int(hist_off.numel()) - 1
    _check(lib.strata_sample_rows(
        ctx, ptr, dt, B, V, ld,
        _typed(row_slot, torch.int32, "row_slot"), _typed(row_pos, torch.int64, "row_pos"),
        _typed(hist, torch.int32, "hist"), _typed(hist_off, torch.int32, "hist_off"), n_hist,
        _typed(out_ids, torch.int32, "out_ids"),
        int(top_n), _typed(chosen_lp, torch.float32, "chosen_lp"), _typed(top_ids, torch.int32, "top_ids"),
        _typed(top_lps, torch.float32, "top_lps"),
        _typed(allowed, torch.int32, "allowed"), _typed(allowed_off, torch.int32, "allowed_off"),
        _typed(allowed_lps, torch.float32, "allowed_lps"),
        _typed(topk_ids, torch.int32, "topk_ids"), _typed(topk_vals, torch.float32, "topk_vals"),
        _typed(kept, torch.int32, "kept"), int(flags), _stream(stream)))


def strata_sample_verify(ctx, logits, row_slot, row_pos, row_draft, out_ids, slot_keep, V=None, hist=None,
                         hist_off=None, top_n: int = 0, chosen_lp=None, top_ids=None, top_lps=None, flags: int = 0,
                         stream=None) -> None:
    import torch
    ptr, dt, B, V, ld = _logits_args(logits, V)
    n_hist = 0 if hist_off is None else int(hist_off.numel()) - 1
    _check(lib.strata_sample_verify(
        ctx, ptr, dt, B, V, ld,
        _typed(row_slot, torch.int32, "row_slot"), _typed(row_pos, torch.int64, "row_pos"),
        _typed(row_draft, torch.int32, "row_draft"),
        _typed(hist, torch.int32, "hist"), _typed(hist_off, torch.int32, "hist_off"), n_hist,
        _typed(out_ids, torch.int32, "out_ids"), _typed(slot_keep, torch.int32, "slot_keep"),
        int(top_n), _typed(chosen_lp, torch.float32, "chosen_lp"), _typed(top_ids, torch.int32, "top_ids"),
        _typed(top_lps, torch.float32, "top_lps"), int(flags), _stream(stream)))


def strata_logprobs_rows(ctx, logits, V=None, chosen=None, chosen_lp=None, top_n: int = 0, top_ids=None,
                         top_lps=None, allowed=None, allowed_off=None, allowed_lps=None, flags: int = 0,
                         stream=None) -> None:
    import torch
    ptr, dt, B, V, ld = _logits_args(logits, V)
    _check(lib.strata_logprobs_rows(
        ctx, ptr, dt, B, V, ld,
        _typed(chosen, torch.int32, "chosen"), _typed(chosen_lp, torch.float32, "chosen_lp"),
        int(top_n), _typed(top_ids, torch.int32, "top_ids"), _typed(top_lps, torch.float32, "top_lps"),
        _typed(allowed, torch.int32, "allowed"), _typed(allowed_off, torch.int32, "allowed_off"),
        _typed(allowed_lps, torch.float32, "allowed_lps"), int(flags), _stream(stream)))


def strata_shard_rows(ctx, logits, row_slot, records, id_offset: int, V=None, hist=None, hist_off=None,
                      top_n: int = 0, flags: int = 0, stream=None) -> None:
    """One vocabulary slice of B rows (columns = ids id_offset ..) -> records [B][1280] uint8."""
    import torch
    ptr, dt, B, V, ld = _logits_args(logits, V)
    n_hist = 0 if hist_off is None else int(hist_off.numel()) - 1
    _check(lib.strata_shard_rows(
        ctx, ptr, dt, B, V, ld, int(id_offset), _typed(row_slot, torch.int32, "row_slot"),
        _typed(hist, torch.int32, "hist"), _typed(hist_off, torch.int32, "hist_off"), n_hist,
        int(top_n), _typed(records, torch.uint8, "records"), int(flags), _stream(stream)))


def strata_merge_shards(ctx, records, row_slot, row_pos, out_ids, top_n: int = 0, chosen_lp=None, top_ids=None,
                        top_lps=None, topk_ids=None, topk_vals=None, kept=None, flags: int = 0,
                        stream=None) -> None:
    """Merge records [n_shards][B][1280] uint8 into the rows' samples and logprobs."""
    import torch
    if records.dim() != 3 or records.shape[2] != STRATA_SHARD_RECORD_BYTES:
        raise ValueError("records must be [n_shards, B, STRATA_SHARD_RECORD_BYTES]")
    _check(lib.strata_merge_shards(
        ctx, _typed(records, torch.uint8, "records"), int(records.shape[0]), int(records.shape[1]),
        _typed(row_slot, torch.int32, "row_slot"), _typed(row_pos, torch.int64, "row_pos"),
        _typed(out_ids, torch.int32, "out_ids"), int(top_n), _typed(chosen_lp, torch.float32, "chosen_lp"),
        _typed(top_ids, torch.int32, "top_ids"), _typed(top_lps, torch.float32, "top_lps"),
        _typed(topk_ids, torch.int32, "topk_ids"), _typed(topk_vals, torch.float32, "topk_vals"),
        _typed(kept, torch.int32, "kept"), int(flags), _stream(stream)))


def strata_read_errors(ctx, stream=None) -> int:
    bits = ctypes.c_uint32()
    _check(lib.strata_read_errors(ctx, ctypes.byref(bits), _stream(stream)))
    return int(bits.value)


def strata_launch_shape(ctx, mode: int, dtype: int, B: int, V: int, top_n: int = 0, flags: int = 0) -> dict:
    s, c, m, g = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib.strata_launch_shape(ctx, mode, dtype, B, V, top_n, flags, ctypes.byref(s), ctypes.byref(c),
                                   ctypes.byref(m), ctypes.byref(g)))
    return dict(split=s.value, chunk=c.value, smem=m.value, grid=g.value)


def strata_sample_rows_noalloc(logits, row_params, row_counters, row_pos, out_ids, V=None, hist=None,
                               hist_off=None, top_n: int = 0, chosen_lp=None, top_ids=None, top_lps=None,
                               stream=None) -> None:
    """Allocation-free sampling: row b is its own slot with keys row_params[b] (dicts) and draw
    counter row_counters[b]; the caller advances the counters.  See the C header for the rules."""
    import torch
    ptr, dt, B, V, ld = _logits_args(logits, V)
    if len(row_params) != B or len(row_counters) != B:
        raise ValueError("one key set and one counter per row")
    params = (strata_sampling_params * max(B, 1))()
    for b, p in enumerate(row_params):
        params[b] = to_c_params(p)
    ctrs = (ctypes.c_uint64 * max(B, 1))(*[int(c) for c in row_counters])
    _check(lib.strata_sample_rows_noalloc(
        ptr, dt, B, V, ld, params, ctrs, _typed(row_pos, torch.int64, "row_pos"), _typed(hist, torch.int32, "hist"),
        _typed(hist_off, torch.int32, "hist_off"), _typed(out_ids, torch.int32, "out_ids"), int(top_n),
        _typed(chosen_lp, torch.float32, "chosen_lp"), _typed(top_ids, torch.int32, "top_ids"),
        _typed(top_lps, torch.float32, "top_lps"), _stream(stream)))


def strata_history_enable(ctx) -> None:
    _check(lib.strata_history_enable(ctx))


def strata_history_set(ctx, slot: int, ids, stream=None) -> None:
    """Replace a slot's kept history by `ids` (any integer sequence, host side)."""
    import numpy as np
    a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).reshape(-1))
    _check(lib.strata_history_set(ctx, slot, a.ctypes.data if a.size else None, int(a.size), _stream(stream)))


def strata_history_get(ctx, slot: int, max_n: int = STRATA_HISTORY_CAP, stream=None):
    """(newest min(length, capacity, max_n) ids of the slot, oldest first, as int32 numpy; length)."""
    import numpy as np
    out = np.zeros(max(int(max_n), 1), dtype=np.int32)
    n, length = ctypes.c_int(), ctypes.c_int64()
    _check(lib.strata_history_get(ctx, slot, out.ctypes.data, int(max_n), ctypes.byref(n), ctypes.byref(length),
                                  _stream(stream)))
    return out[:n.value].copy(), int(length.value)
