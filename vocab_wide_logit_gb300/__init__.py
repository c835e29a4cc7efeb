"""libdsample: the GB300 vocab-wide sampling pass (CFG combine, max/logsumexp/argmax,
exact top-ratio filter, Gumbel-max) and the large-vocab greedy max/LSE/argmax pass.

The compute lives in the CUDA library (csrc/, built by build.py); the Python
side only marshals arguments through the C ABI declared in include/dsample.h.
"""
from ._lib import (DS_DEV_ERR_LAYOUT, DS_DEV_ERR_NO_UNCOND, DS_DEV_ERR_PARAM, DS_MAX_VOCAB, DsError,
                   ds_greedy_lse, ds_sample, load, status_string, top_k)
from .api import greedy_lse, sample, sample_host

__all__ = ["ds_sample", "ds_greedy_lse", "sample", "sample_host", "greedy_lse", "load", "top_k",
           "status_string", "DsError", "DS_MAX_VOCAB", "DS_DEV_ERR_LAYOUT", "DS_DEV_ERR_NO_UNCOND",
           "DS_DEV_ERR_PARAM"]
