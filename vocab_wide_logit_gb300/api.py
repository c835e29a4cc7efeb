"""Tensor-level wrappers over the C ABI (allocation of outputs and host<->device copies only)."""
import torch

from . import _lib


def sample(request_ids, c_logits, u_logits, seq_lens, guidance, temperature, top_ratio, seed, iteration,
           out_tokens=None, out_logprobs=None, d_status=None, stream=None, top_ratios=None, iterations=None,
           keep_ties=False):
    """Sample every cell of c_logits [C, P, V] (bf16, cuda). Returns (tokens int32 [C, P],
    logprobs float32 [C, P]). top_ratios / iterations: optional per-request device arrays [B]."""
    C, P, V = c_logits.shape
    dev = c_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((C, P), dtype=torch.int32, device=dev)
    if out_logprobs is None:
        out_logprobs = torch.empty((C, P), dtype=torch.float32, device=dev)
    _lib.ds_sample(request_ids, c_logits, u_logits, seq_lens, guidance, temperature, top_ratio, seed,
                   iteration, out_tokens, out_logprobs, d_status=d_status, stream=stream, top_ratios=top_ratios,
                   iterations=iterations, keep_ties=keep_ties)
    return out_tokens, out_logprobs


class HostSampler:
    """End-to-end use from host memory: per call, copy the step's logits from pinned host
    buffers to device buffers owned by this object, run ds_sample, copy (tokens, logprobs)
    back to pinned host buffers. Metadata (ids, lengths, guidance, temperature) is uploaded once."""

    def __init__(self, request_ids, seq_lens, guidance, temperature, C, P, P_u, V, device="cuda"):
        self.C, self.P, self.P_u, self.V = int(C), int(P), int(P_u), int(V)
        self.request_ids = request_ids.to(device)
        self.seq_lens = seq_lens.to(device)
        self.guidance = guidance.to(device)
        self.temperature = temperature.to(device)
        self.c_dev = torch.empty((self.C, self.P, self.V), dtype=torch.bfloat16, device=device)
        self.u_dev = (torch.empty((self.C, self.P_u, self.V), dtype=torch.bfloat16, device=device)
                      if self.P_u > 0 else None)
        self.tok_dev = torch.empty((self.C, self.P), dtype=torch.int32, device=device)
        self.lp_dev = torch.empty((self.C, self.P), dtype=torch.float32, device=device)
        self.tok_host = torch.empty((self.C, self.P), dtype=torch.int32).pin_memory()
        self.lp_host = torch.empty((self.C, self.P), dtype=torch.float32).pin_memory()

    def h2d_bytes(self):
        return self.c_dev.numel() * 2 + (self.u_dev.numel() * 2 if self.u_dev is not None else 0)

    def d2h_bytes(self):
        return self.tok_host.numel() * 4 + self.lp_host.numel() * 4

    def __call__(self, c_host, u_host, top_ratio, seed, iteration, stream=None):
        self.c_dev.copy_(c_host, non_blocking=True)
        if self.u_dev is not None:
            self.u_dev.copy_(u_host, non_blocking=True)
        _lib.ds_sample(self.request_ids, self.c_dev, self.u_dev, self.seq_lens, self.guidance,
                       self.temperature, top_ratio, seed, iteration, self.tok_dev, self.lp_dev, stream=stream)
        self.tok_host.copy_(self.tok_dev, non_blocking=True)
        self.lp_host.copy_(self.lp_dev, non_blocking=True)
        return self.tok_host, self.lp_host


def sample_host(*args, **kwargs):
    """Construct a HostSampler (see its docstring)."""
    return HostSampler(*args, **kwargs)


def greedy_lse(logits, out_max=None, out_lse=None, out_argmax=None, stream=None):
    """Per-row (max, lse, argmax) of bf16 logits [n, V] on the GPU."""
    n, V = logits.shape
    dev = logits.device
    if out_max is None:
        out_max = torch.empty(n, dtype=torch.float32, device=dev)
    if out_lse is None:
        out_lse = torch.empty(n, dtype=torch.float32, device=dev)
    if out_argmax is None:
        out_argmax = torch.empty(n, dtype=torch.int32, device=dev)
    _lib.ds_greedy_lse(logits, out_max, out_lse, out_argmax, stream=stream)
    return out_max, out_lse, out_argmax


def merge_triples(triples, stream=None):
    """Merge per-shard triples float32 [n, shards, 3] -> (max, lse, argmax) per token on the GPU."""
    n = triples.shape[0]
    dev = triples.device
    out_max = torch.empty(n, dtype=torch.float32, device=dev)
    out_lse = torch.empty(n, dtype=torch.float32, device=dev)
    out_argmax = torch.empty(n, dtype=torch.int32, device=dev)
    _lib.ds_merge_triples(triples, out_max, out_lse, out_argmax, stream=stream)
    return out_max, out_lse, out_argmax


def log_softmax(logits, dtype=torch.float32, stream=None):
    """Dense log-softmax of bf16 logits [n, V] (fp32 or bf16 out) and the per-row (max, lse, argmax)."""
    n, V = logits.shape
    dev = logits.device
    out = torch.empty((n, V), dtype=dtype, device=dev)
    out_max = torch.empty(n, dtype=torch.float32, device=dev)
    out_lse = torch.empty(n, dtype=torch.float32, device=dev)
    out_argmax = torch.empty(n, dtype=torch.int32, device=dev)
    _lib.ds_log_softmax(logits, out, out_max, out_lse, out_argmax, stream=stream)
    return out, out_max, out_lse, out_argmax


def reveal(scores, tokens, seq_lens, reveal_counts, canvas, stream=None):
    """Commit the top reveal_counts[r] cells of each request (score desc, flattened index asc) into
    canvas (in place); returns the uint8 [C, P] flags of the committed cells."""
    revealed = torch.empty(scores.shape, dtype=torch.uint8, device=scores.device)
    _lib.ds_reveal(scores, tokens, seq_lens, reveal_counts, canvas, revealed, stream=stream)
    return revealed
