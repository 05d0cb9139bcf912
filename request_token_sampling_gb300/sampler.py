"""A small object wrapper over the C-named calls: owns a context and allocates output tensors."""
from __future__ import annotations

from . import _binding as B


class Sampler:
    """One context on one device; every method is one C-ABI call (plus torch output allocation)."""

    def __init__(self, device: int = 0, max_slots: int = 64, max_vocab: int = 262144, max_rows: int = 1024):
        self.device = device
        self.max_slots = max_slots
        self.ctx = B.strata_create(device, max_slots, max_vocab, max_rows)

    def close(self) -> None:
        if self.ctx is not None:
            B.strata_destroy(self.ctx)
            self.ctx = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def set_slot(self, slot: int, params, reset_counter: bool = False, stream=None) -> None:
        B.strata_set_slot_params(self.ctx, slot, params, reset_counter, stream)

    def slot_state(self, slot: int, stream=None):
        return B.strata_get_slot_state(self.ctx, slot, stream)

    def restore_slot(self, slot: int, params, counter: int, stream=None) -> None:
        B.strata_set_slot_state(self.ctx, slot, params, counter, stream)

    def history_enable(self) -> None:
        B.strata_history_enable(self.ctx)

    def history_set(self, slot: int, ids, stream=None) -> None:
        B.strata_history_set(self.ctx, slot, ids, stream)

    def history_get(self, slot: int, max_n: int = B.STRATA_HISTORY_CAP, stream=None):
        return B.strata_history_get(self.ctx, slot, max_n, stream)

    def errors(self, stream=None) -> int:
        return B.strata_read_errors(self.ctx, stream)

    def shape(self, mode: int, dtype: int, rows: int, V: int, top_n: int = 0, flags: int = 0) -> dict:
        return B.strata_launch_shape(self.ctx, mode, dtype, rows, V, top_n, flags)

    def sample(self, logits, row_slot, row_pos, V=None, hist=None, hist_off=None, top_n: int = 0,
               chosen_lp: bool = False, allowed=None, allowed_off=None, debug: bool = False, flags: int = 0,
               stream=None, out=None) -> dict:
        import torch
        rows = logits.shape[0]
        dev = logits.device
        o = out if out is not None else {}
        if "ids" not in o:
            o["ids"] = torch.empty(rows, dtype=torch.int32, device=dev)
        if chosen_lp and "chosen_lp" not in o:
            o["chosen_lp"] = torch.empty(rows, dtype=torch.float32, device=dev)
        if top_n > 0 and "top_ids" not in o:
            o["top_ids"] = torch.empty(rows, top_n, dtype=torch.int32, device=dev)
            o["top_lps"] = torch.empty(rows, top_n, dtype=torch.float32, device=dev)
        if allowed_off is not None and "allowed_lps" not in o:
            # at least one element: a zero-size tensor has no device address
            o["allowed_lps"] = torch.empty(max(1, int(allowed.numel())), dtype=torch.float32, device=dev)
        if debug and "topk_ids" not in o:
            o["topk_ids"] = torch.empty(rows, 64, dtype=torch.int32, device=dev)
            o["topk_vals"] = torch.empty(rows, 64, dtype=torch.float32, device=dev)
            o["kept"] = torch.empty(rows, 2, dtype=torch.int32, device=dev)
        B.strata_sample_rows(self.ctx, logits, row_slot, row_pos, o["ids"], V=V, hist=hist, hist_off=hist_off,
                             top_n=top_n, chosen_lp=o.get("chosen_lp"), top_ids=o.get("top_ids"),
                             top_lps=o.get("top_lps"), allowed=allowed, allowed_off=allowed_off,
                             allowed_lps=o.get("allowed_lps"), topk_ids=o.get("topk_ids"),
                             topk_vals=o.get("topk_vals"), kept=o.get("kept"), flags=flags, stream=stream)
        return o

    def verify(self, logits, row_slot, row_pos, row_draft, V=None, hist=None, hist_off=None, top_n: int = 0,
               chosen_lp: bool = False, flags: int = 0, stream=None, out=None) -> dict:
        """Sample verify windows: the picks plus, per slot, the number of rows to keep."""
        import torch
        rows = logits.shape[0]
        dev = logits.device
        o = out if out is not None else {}
        if "ids" not in o:
            o["ids"] = torch.empty(rows, dtype=torch.int32, device=dev)
        if "keep" not in o:
            o["keep"] = torch.full((self.max_slots,), -1, dtype=torch.int32, device=dev)
        if chosen_lp and "chosen_lp" not in o:
            o["chosen_lp"] = torch.empty(rows, dtype=torch.float32, device=dev)
        if top_n > 0 and "top_ids" not in o:
            o["top_ids"] = torch.empty(rows, top_n, dtype=torch.int32, device=dev)
            o["top_lps"] = torch.empty(rows, top_n, dtype=torch.float32, device=dev)
        B.strata_sample_verify(self.ctx, logits, row_slot, row_pos, row_draft, o["ids"], o["keep"], V=V, hist=hist,
                               hist_off=hist_off, top_n=top_n, chosen_lp=o.get("chosen_lp"),
                               top_ids=o.get("top_ids"), top_lps=o.get("top_lps"), flags=flags, stream=stream)
        return o

    def logprobs(self, logits, V=None, chosen=None, top_n: int = 0, allowed=None, allowed_off=None,
                 flags: int = 0, stream=None, out=None) -> dict:
        import torch
        rows = logits.shape[0]
        dev = logits.device
        o = out if out is not None else {}
        if chosen is not None and "chosen_lp" not in o:
            o["chosen_lp"] = torch.empty(rows, dtype=torch.float32, device=dev)
        if top_n > 0 and "top_ids" not in o:
            o["top_ids"] = torch.empty(rows, top_n, dtype=torch.int32, device=dev)
            o["top_lps"] = torch.empty(rows, top_n, dtype=torch.float32, device=dev)
        if allowed_off is not None and "allowed_lps" not in o:
            o["allowed_lps"] = torch.empty(max(1, int(allowed.numel())), dtype=torch.float32, device=dev)
        B.strata_logprobs_rows(self.ctx, logits, V=V, chosen=chosen, chosen_lp=o.get("chosen_lp"), top_n=top_n,
                               top_ids=o.get("top_ids"), top_lps=o.get("top_lps"), allowed=allowed,
                               allowed_off=allowed_off, allowed_lps=o.get("allowed_lps"), flags=flags,
                               stream=stream)
        return o

    def shard(self, logits, row_slot, id_offset: int, V=None, hist=None, hist_off=None, top_n: int = 0,
              flags: int = 0, stream=None, out=None):
        """One vocabulary slice of the rows (its columns hold ids id_offset ..): the rows' records,
        a [B, STRATA_SHARD_RECORD_BYTES] uint8 tensor."""
        import torch
        rows = logits.shape[0]
        rec = out if out is not None else torch.empty(rows, B.STRATA_SHARD_RECORD_BYTES, dtype=torch.uint8,
                                                      device=logits.device)
        B.strata_shard_rows(self.ctx, logits, row_slot, rec, id_offset, V=V, hist=hist, hist_off=hist_off,
                            top_n=top_n, flags=flags, stream=stream)
        return rec

    def merge(self, records, row_slot, row_pos, top_n: int = 0, chosen_lp: bool = False, debug: bool = False,
              stream=None, out=None) -> dict:
        """Merge every slice's records ([n_shards, B, STRATA_SHARD_RECORD_BYTES] uint8): the same
        outputs as `sample` on the whole rows."""
        import torch
        rows = records.shape[1]
        dev = records.device
        o = out if out is not None else {}
        if "ids" not in o:
            o["ids"] = torch.empty(rows, dtype=torch.int32, device=dev)
        if chosen_lp and "chosen_lp" not in o:
            o["chosen_lp"] = torch.empty(rows, dtype=torch.float32, device=dev)
        if top_n > 0 and "top_ids" not in o:
            o["top_ids"] = torch.empty(rows, top_n, dtype=torch.int32, device=dev)
            o["top_lps"] = torch.empty(rows, top_n, dtype=torch.float32, device=dev)
        if debug and "topk_ids" not in o:
            o["topk_ids"] = torch.empty(rows, 64, dtype=torch.int32, device=dev)
            o["topk_vals"] = torch.empty(rows, 64, dtype=torch.float32, device=dev)
            o["kept"] = torch.empty(rows, 2, dtype=torch.int32, device=dev)
        B.strata_merge_shards(self.ctx, records, row_slot, row_pos, o["ids"], top_n=top_n,
                              chosen_lp=o.get("chosen_lp"), top_ids=o.get("top_ids"), top_lps=o.get("top_lps"),
                              topk_ids=o.get("topk_ids"), topk_vals=o.get("topk_vals"), kept=o.get("kept"),
                              stream=stream)
        return o
