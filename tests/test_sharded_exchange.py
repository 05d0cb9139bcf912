"""The exchange of vocabulary-slice records between ranks, on CPU with the gloo backend (world size
2): each rank reduces its half of every row to the oracle's record, packs it in the layout
include/strata_sample.h documents, and the package's ``gather_records`` all-gathers the records;
every rank reads them back with ``unpack_record`` and merges them with the oracle.  Both ranks must
reach the same result, equal to the oracle on the whole rows.  No GPU: the records stand in for
what strata_shard_rows writes on each rank's GPU."""
import os
import socket
import struct
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_strata_build", os.path.join(ROOT, "request_token_sampling_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build_library()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ord(v: float) -> int:
    """Order-preserving uint32 of a float32 (the record key's high word)."""
    bits = struct.unpack("<I", struct.pack("<f", v))[0]
    if bits == 0x80000000:
        bits = 0
    return (~bits & 0xFFFFFFFF) if bits & 0x80000000 else (bits | 0x80000000)


def pack_record(rec: dict, nbytes: int) -> bytes:
    """An oracle record in the library's byte layout."""
    buf = bytearray(nbytes)
    lse = struct.unpack("<I", struct.pack("<f", rec["lse"]))[0]
    struct.pack_into("<4I", buf, 0, len(rec["pen"]), len(rec["raw"]), lse, 0)
    for j, (v, t, raw) in enumerate(rec["pen"]):
        struct.pack_into("<2If I", buf, 16 + 16 * j, 0xFFFFFFFF - t, _ord(v), raw, 0)
    for j, (v, t) in enumerate(rec["raw"]):
        struct.pack_into("<2I", buf, 16 + 16 * 64 + 8 * j, 0xFFFFFFFF - t, _ord(v))
    return bytes(buf)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist
    import oracle
    import synth
    from request_token_sampling_gb300 import STRATA_SHARD_RECORD_BYTES
    from request_token_sampling_gb300.sharded import gather_records, unpack_record
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.config4(fused=True)
        V, top_n = w["V"], w["top_n"]
        bounds = [0, 124160, V]
        lo, hi = bounds[rank], bounds[rank + 1]
        mine = np.zeros((w["B"], STRATA_SHARD_RECORD_BYTES), np.uint8)
        params = []
        for b in range(w["B"]):
            s = int(w["row_slot"][b])
            p = oracle.Params.from_dict(w["slot_params"][s])
            params.append((s, p))
            raw = oracle.widen(w["logits"][b, :V], w["dtype"])
            rec = oracle.shard_record(raw[lo:hi], lo, p, oracle.sampling._slot_history(w, s),
                                      1 if p.greedy else p.k, top_n)
            mine[b] = np.frombuffer(pack_record(rec, STRATA_SHARD_RECORD_BYTES), np.uint8)
        allrec = gather_records(torch.from_numpy(mine)).numpy()
        out = []
        for b, (s, p) in enumerate(params):
            recs = [unpack_record(allrec[g, b].tobytes()) for g in range(world)]
            m = oracle.merge_records(recs, p, int(w["row_pos"][b]), int(w["counters"].get(s, 0)), top_n)
            out.append((m["id"], m["topk_ids"].tolist(), m["top_ids"].tolist(), m["top_lps"].tolist(),
                        m["chosen_lp"]))
        q.put((rank, allrec.shape, out))
    finally:
        dist.destroy_process_group()


def test_record_exchange_gloo_world2():
    _build()
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, shape0, out0), (_, shape1, out1) = res
    assert shape0 == shape1 == (2, 8, 1280)
    assert out0 == out1, "the ranks merged to different results"
    w = synth.config4(fused=True)
    rows, _ = oracle.sample_call(w, with_allowed=False)
    for b, r in enumerate(rows):
        gid, topk, top_ids, top_lps, chosen_lp = out0[b]
        assert gid == r["id"] and topk == r["topk_ids"].tolist() and top_ids == r["top_ids"].tolist()
        assert np.max(np.abs(np.asarray(top_lps) - r["top_lps"])) <= 1e-5    # fp32 log-sum-exp per slice
        assert abs(chosen_lp - r["chosen_lp"]) <= 1e-5


class _OracleSlices:
    """A stand-in for a rank's Sampler on CPU: `shard` packs the oracle's records of the rank's slice
    in the library's layout, `merge` reads the gathered records back and merges them with the
    oracle, so `sample_sliced` runs its real exchange between the two."""

    def __init__(self, w):
        self.w = w

    def shard(self, logits, row_slot, id_offset, hist=None, hist_off=None, top_n=0, flags=0, stream=None):
        import oracle
        import torch
        from request_token_sampling_gb300 import STRATA_SHARD_RECORD_BYTES
        w = self.w
        out = np.zeros((w["B"], STRATA_SHARD_RECORD_BYTES), np.uint8)
        for b in range(w["B"]):
            s = int(w["row_slot"][b])
            p = oracle.Params.from_dict(w["slot_params"][s])
            raw = np.asarray(logits[b].numpy(), np.float32)
            rec = oracle.shard_record(raw, id_offset, p, oracle.sampling._slot_history(w, s),
                                      1 if p.greedy else p.k, top_n)
            out[b] = np.frombuffer(pack_record(rec, STRATA_SHARD_RECORD_BYTES), np.uint8)
        return torch.from_numpy(out)

    def merge(self, allrec, row_slot, row_pos, top_n=0, chosen_lp=False, stream=None):
        import oracle
        from request_token_sampling_gb300.sharded import unpack_record
        w, a = self.w, allrec.numpy()
        ids = []
        for b in range(w["B"]):
            s = int(w["row_slot"][b])
            p = oracle.Params.from_dict(w["slot_params"][s])
            recs = [unpack_record(a[g, b].tobytes()) for g in range(a.shape[0])]
            ids.append(oracle.merge_records(recs, p, int(w["row_pos"][b]), int(w["counters"].get(s, 0)), top_n)["id"])
        return {"ids": ids}


def _sliced_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import synth
    from request_token_sampling_gb300.sharded import sample_sliced
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.config3()                       # bf16 batch slots, greedy and sampled
        import oracle
        raw = np.stack([oracle.widen(w["logits"][b, :w["V"]], w["dtype"]) for b in range(w["B"])])
        cut = [0, 100000, w["V"]]
        part = torch.from_numpy(np.ascontiguousarray(raw[:, cut[rank]:cut[rank + 1]]))
        out = sample_sliced(_OracleSlices(w), part, cut[rank], None, None, top_n=w["top_n"])
        q.put((rank, [int(x) for x in out["ids"]]))
    finally:
        dist.destroy_process_group()


def test_sample_sliced_over_gloo_world2():
    """`sample_sliced` on two gloo ranks, each holding part of config 3's rows: both ranks return
    the whole-row oracle's picks."""
    _build()
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sliced_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    rows, _ = oracle.sample_call(synth.config3(), with_allowed=False)
    assert res[0][1] == res[1][1] == [r["id"] for r in rows]


def test_pack_unpack_round_trip():
    """The package's reader inverts the documented layout, -0.0 read as +0.0, for every sign."""
    _build()
    sys.path.insert(0, ROOT)
    from request_token_sampling_gb300 import STRATA_SHARD_RECORD_BYTES
    from request_token_sampling_gb300.sharded import unpack_record
    rec = dict(pen=[(3.5, 7, 4.0), (0.0, 2, 0.0), (-1.25, 100000, -1.0), (float("-inf"), 5, float("-inf"))],
               raw=[(4.0, 7), (-0.5, 9)], lse=12.25)
    got = unpack_record(pack_record(rec, STRATA_SHARD_RECORD_BYTES))
    assert got == rec
    neg0 = dict(pen=[(-0.0, 3, -0.0)], raw=[], lse=0.0)
    got = unpack_record(pack_record(neg0, STRATA_SHARD_RECORD_BYTES))
    assert got["pen"][0][0] == 0.0 and not np.signbit(got["pen"][0][0]) and got["pen"][0][1] == 3
    with pytest.raises(ValueError):
        unpack_record(b"\0" * 16)
