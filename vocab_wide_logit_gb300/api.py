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
    """End-to-end use from host memory. Each step copies its logits from pinned host buffers to
    device buffers owned by this object, runs ds_sample, and copies (tokens, logprobs) back to
    pinned host buffers. Metadata (ids, lengths, guidance, temperature) is uploaded once.

    Steps are pipelined over `depth` buffer sets: submit() queues a step's host-to-device copy on
    a copy stream, the sampling on a compute stream once that copy is done, and the copy back on a
    third stream once the sampling is done, then returns at once; so step i + 1's copy (the
    link-bound part) runs while step i samples. result(slot) waits for a step and returns its
    pinned host outputs, which stay valid until the slot is submitted again (depth steps later).
    A call (sampler(...)) is submit() followed by result()."""

    def __init__(self, request_ids, seq_lens, guidance, temperature, C, P, P_u, V, device="cuda", depth=2):
        self.C, self.P, self.P_u, self.V = int(C), int(P), int(P_u), int(V)
        self.depth = int(depth)
        self.request_ids = request_ids.to(device)
        self.seq_lens = seq_lens.to(device)
        self.guidance = guidance.to(device)
        self.temperature = temperature.to(device)
        d = self.depth
        self.c_dev = [torch.empty((self.C, self.P, self.V), dtype=torch.bfloat16, device=device) for _ in range(d)]
        self.u_dev = [(torch.empty((self.C, self.P_u, self.V), dtype=torch.bfloat16, device=device)
                       if self.P_u > 0 else None) for _ in range(d)]
        self.tok_dev = [torch.empty((self.C, self.P), dtype=torch.int32, device=device) for _ in range(d)]
        self.lp_dev = [torch.empty((self.C, self.P), dtype=torch.float32, device=device) for _ in range(d)]
        self.tok_host = [torch.empty((self.C, self.P), dtype=torch.int32).pin_memory() for _ in range(d)]
        self.lp_host = [torch.empty((self.C, self.P), dtype=torch.float32).pin_memory() for _ in range(d)]
        self.h2d = torch.cuda.Stream(device=device)
        self.compute = torch.cuda.Stream(device=device)
        self.d2h = torch.cuda.Stream(device=device)
        self.copied = [torch.cuda.Event() for _ in range(d)]
        self.sampled = [torch.cuda.Event() for _ in range(d)]
        self.returned = [torch.cuda.Event() for _ in range(d)]
        self.n = 0

    def h2d_bytes(self):
        return self.c_dev[0].numel() * 2 + (self.u_dev[0].numel() * 2 if self.u_dev[0] is not None else 0)

    def d2h_bytes(self):
        return self.tok_host[0].numel() * 4 + self.lp_host[0].numel() * 4

    def submit(self, c_host, u_host, top_ratio, seed, iteration):
        s = self.n % self.depth
        self.n += 1
        # the slot's device buffers are free once its previous sampling is done, and its host
        # outputs once their copy has been waited for (result() of that step)
        self.returned[s].synchronize()
        self.h2d.wait_event(self.sampled[s])
        with torch.cuda.stream(self.h2d):
            self.c_dev[s].copy_(c_host, non_blocking=True)
            if self.u_dev[s] is not None:
                self.u_dev[s].copy_(u_host, non_blocking=True)
            self.copied[s].record(self.h2d)
        self.compute.wait_event(self.copied[s])
        _lib.ds_sample(self.request_ids, self.c_dev[s], self.u_dev[s], self.seq_lens, self.guidance,
                       self.temperature, top_ratio, seed, iteration, self.tok_dev[s], self.lp_dev[s],
                       stream=self.compute)
        self.sampled[s].record(self.compute)
        self.d2h.wait_event(self.sampled[s])
        with torch.cuda.stream(self.d2h):
            self.tok_host[s].copy_(self.tok_dev[s], non_blocking=True)
            self.lp_host[s].copy_(self.lp_dev[s], non_blocking=True)
            self.returned[s].record(self.d2h)
        return s

    def result(self, slot):
        self.returned[slot].synchronize()
        return self.tok_host[slot], self.lp_host[slot]

    def __call__(self, c_host, u_host, top_ratio, seed, iteration):
        return self.result(self.submit(c_host, u_host, top_ratio, seed, iteration))


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
