"""Vocabulary-sliced sampling across processes: each rank holds one slice of every row's logits.

A rank reduces its slice to records (``Sampler.shard``: strata_shard_rows), the ranks exchange the
records with one all-gather over a ``torch.distributed`` group, and every rank merges all of them
(``Sampler.merge``: strata_merge_shards).  Every rank then holds the same samples and log-probs as
a whole-row call, and its slots' counters advance the same way, so the ranks stay in step.  The
exchange moves STRATA_SHARD_RECORD_BYTES per row per rank; no logits leave their GPU.

``unpack_record`` reads one record back on the host (the layout include/strata_sample.h
documents), for inspection and tests.
"""
from __future__ import annotations

import struct

from . import _binding as B

REC_PEN = 16                 # byte offset of the penalised entries
REC_RAW = REC_PEN + 16 * 64  # byte offset of the raw keys


def gather_records(records, group=None):
    """All-gather a rank's records ([B, STRATA_SHARD_RECORD_BYTES] uint8) into
    [world, B, STRATA_SHARD_RECORD_BYTES], slice r from rank r."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(records) for _ in range(world)]
    dist.all_gather(parts, records.contiguous(), group=group)
    return torch.stack(parts, 0)


def sample_sliced(sampler, logits, id_offset: int, row_slot, row_pos, hist=None, hist_off=None, top_n: int = 0,
                  chosen_lp: bool = False, group=None, flags: int = 0, stream=None) -> dict:
    """One sampling step over rows whose vocabulary is split across the group's ranks: this rank's
    columns hold ids id_offset .. id_offset + logits.shape[1] - 1.  Returns the merged outputs
    (identical on every rank).  `stream` (a torch CUDA stream or a raw cudaStream_t handle; None:
    the current stream) orders the slice launch, the all-gather and the merge one after another."""
    rec = sampler.shard(logits, row_slot, id_offset, hist=hist, hist_off=hist_off, top_n=top_n, flags=flags,
                        stream=stream)
    if stream is None:
        allrec = gather_records(rec, group)
    else:
        import torch
        ts = torch.cuda.ExternalStream(stream) if isinstance(stream, int) else stream
        with torch.cuda.stream(ts):     # the collective waits for the slice launch on this stream
            allrec = gather_records(rec, group)
    return sampler.merge(allrec, row_slot, row_pos, top_n=top_n, chosen_lp=chosen_lp, stream=stream)


def _key_value(hi: int) -> float:
    bits = (hi & 0x7FFFFFFF) if hi & 0x80000000 else (~hi & 0xFFFFFFFF)
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def unpack_record(buf) -> dict:
    """One record (STRATA_SHARD_RECORD_BYTES bytes) as
    {"pen": [(penalised value, id, raw logit)], "raw": [(raw value, id)], "lse": float}."""
    b = bytes(buf)
    if len(b) != B.STRATA_SHARD_RECORD_BYTES:
        raise ValueError(f"a record is {B.STRATA_SHARD_RECORD_BYTES} bytes, got {len(b)}")
    n_pen, n_raw, lse_bits, _ = struct.unpack_from("<4I", b, 0)
    lse = struct.unpack("<f", struct.pack("<I", lse_bits))[0]
    pen = []
    for j in range(min(n_pen, 64)):
        lo, hi, raw_bits, _ = struct.unpack_from("<4I", b, REC_PEN + 16 * j)
        raw = struct.unpack("<f", struct.pack("<I", raw_bits))[0]
        pen.append((_key_value(hi), 0xFFFFFFFF - lo, raw))
    raw_list = []
    for j in range(min(n_raw, B.STRATA_MAX_TOP_N)):
        lo, hi = struct.unpack_from("<2I", b, REC_RAW + 8 * j)
        raw_list.append((_key_value(hi), 0xFFFFFFFF - lo))
    return dict(pen=pen, raw=raw_list, lse=lse)
