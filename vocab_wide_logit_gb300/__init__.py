"""libdsample: the GB300 vocab-wide sampling pass (CFG combine, max/logsumexp/argmax,
exact top-ratio filter, Gumbel-max) and the large-vocab greedy max/LSE/argmax pass.

The compute lives in the CUDA library (csrc/, built by build.py); the Python
side only marshals arguments through the C ABI declared in include/dsample.h.
"""
from ._lib import (DS_DEV_ERR_LAYOUT, DS_DEV_ERR_NO_UNCOND, DS_DEV_ERR_PARAM, DS_DTYPE_BF16, DS_DTYPE_F32,
                   DS_FLAG_KEEP_TIES, DS_FLAG_SKIP_EXACT_PASS, DS_MARKED, DS_MAX_VOCAB, DsError, ds_greedy_lse, ds_log_softmax, ds_merge_triples, ds_reveal, ds_sample, load,
                   launch_count, status_string, top_k)
from .api import greedy_lse, log_softmax, merge_triples, reveal, sample, sample_host

__all__ = ["ds_sample", "ds_greedy_lse", "ds_merge_triples", "ds_log_softmax", "ds_reveal", "sample",
           "sample_host", "greedy_lse", "merge_triples", "log_softmax", "reveal", "load", "top_k", "launch_count", "DS_DTYPE_F32", "DS_DTYPE_BF16",
           "status_string", "DsError", "DS_MAX_VOCAB", "DS_DEV_ERR_LAYOUT", "DS_DEV_ERR_NO_UNCOND",
           "DS_DEV_ERR_PARAM", "DS_FLAG_KEEP_TIES", "DS_FLAG_SKIP_EXACT_PASS", "DS_MARKED"]
