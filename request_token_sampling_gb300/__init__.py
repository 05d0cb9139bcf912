"""GB300-native decode-time token sampler.

A C-ABI shared library (``include/strata_sample.h``) over one fused sm_103a CUDA kernel that, per
head-logit row, applies the request's repeat/frequency/presence penalties over its history window,
selects top_k with ties to the lowest index, cuts min_p and top_p, applies temperature and draws one
token from Philox(seed, position) with a per-slot counter that persists across calls; greedy rows
take the penalised argmax.  The same launch can return raw-logit log-probabilities (the chosen
token's, the top 0..20 alternatives, and allowed_token_ids renormalisation).

This package is the thin Python binding (ctypes; PyTorch tensors for device memory and streams).
Importing it fails loudly when the CUDA library has not been built.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import StrataError, lib, strata_sampling_params  # noqa: F401
from .sampler import Sampler  # noqa: F401
