"""CPU oracle of the vocab-wide sampling pass -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this package. It wraps the plain C++ oracle (dsoracle.cpp) with numpy
marshalling; it shares no code with the CUDA library and does not import it.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, u32, u64, f32 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                   ctypes.c_uint64, ctypes.c_float)
        L.dso_philox4x32_10.argtypes = [P, P, P]
        L.dso_philox4x32_10.restype = None
        L.dso_uniform.argtypes = [u32]
        L.dso_uniform.restype = ctypes.c_double
        L.dso_gumbel.argtypes = [u32]
        L.dso_gumbel.restype = ctypes.c_double
        L.dso_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.dso_bf16_to_float.restype = f32
        L.dso_cfg.argtypes = [f32, f32, f32]
        L.dso_cfg.restype = f32
        L.dso_top_k.argtypes = [f32, i32]
        L.dso_top_k.restype = i32
        L.dso_sample_cells.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, f32, u64, u32,
                                       P, i64, P, P, P, P, P, P, P, P]
        L.dso_sample_cells.restype = ctypes.c_int
        L.dso_sample_cells_ex.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, P, f32, u64, P, u32, u32,
                                          P, i64, P, P, P, P, P, P, P, P]
        L.dso_sample_cells_ex.restype = ctypes.c_int
        L.dso_greedy_rows.argtypes = [P, i32, i32, P, i64, P, P, P]
        L.dso_greedy_rows.restype = ctypes.c_int
        L.dso_merge_triples.argtypes = [P, P, P, P, i32, P, P, P]
        L.dso_merge_triples.restype = None
        L.dso_reveal.argtypes = [P, P, P, P, i32, i32, i32, P, P]
        L.dso_reveal.restype = ctypes.c_int
        _LIB = L
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def philox4x32_10(ctr, key):
    ctr = np.asarray(ctr, dtype=np.uint32).reshape(4)
    key = np.asarray(key, dtype=np.uint32).reshape(2)
    out = np.zeros(4, dtype=np.uint32)
    lib().dso_philox4x32_10(_ptr(ctr), _ptr(key), _ptr(out))
    return out


def uniform(x):
    return lib().dso_uniform(int(x) & 0xFFFFFFFF)


def gumbel(x):
    return lib().dso_gumbel(int(x) & 0xFFFFFFFF)


def bf16_to_float(h):
    return lib().dso_bf16_to_float(int(h) & 0xFFFF)


def cfg(c, u, g):
    return lib().dso_cfg(float(c), float(u), float(g))


def top_k(top_ratio, V):
    return int(lib().dso_top_k(float(top_ratio), int(V)))


class OracleError(RuntimeError):
    pass


def sample_cells(request_ids, c_bits, u_bits, seq_lens, C, P, V, guidance, temperature,
                 top_ratio, seed, iteration, cells=None, top_ratios=None, iterations=None, keep_ties=False):
    """Run the sampling oracle on the listed cells (all cells when None).

    c_bits / u_bits are the raw bf16 bit patterns (uint16) of c_logits [C][P][V] and
    u_logits [C][P_u][V]. top_ratios / iterations (length B) replace the scalars per
    request when given. Returns a dict of numpy arrays indexed like `cells`.
    """
    top_ratios = _c(top_ratios, np.float32) if top_ratios is not None else None
    iterations = _c(iterations, np.uint32) if iterations is not None else None
    request_ids = _c(request_ids, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    guidance = _c(guidance, np.float32)
    temperature = _c(temperature, np.float32)
    c_bits = _c(c_bits, np.uint16)
    u_bits = _c(u_bits, np.uint16) if u_bits is not None else None
    B = int(seq_lens.shape[0])
    if cells is None:
        cells = np.arange(int(C) * int(P), dtype=np.int64)
    cells = _c(cells, np.int64)
    n = int(cells.shape[0])
    out = {
        "tokens": np.zeros(n, np.int32), "logprobs": np.zeros(n, np.float64),
        "lse": np.zeros(n, np.float64), "max": np.zeros(n, np.float32),
        "argmax": np.zeros(n, np.int32), "top1": np.zeros(n, np.float64),
        "top2": np.zeros(n, np.float64), "thresh_ties": np.zeros(n, np.int32),
    }
    rc = lib().dso_sample_cells_ex(
        _ptr(request_ids), _ptr(c_bits), _ptr(u_bits), _ptr(seq_lens), B, int(C), int(P), int(V),
        _ptr(guidance), _ptr(temperature), _ptr(top_ratios), float(top_ratio), int(seed) & (2**64 - 1),
        _ptr(iterations), int(iteration), 1 if keep_ties else 0, _ptr(cells), n, _ptr(out["tokens"]),
        _ptr(out["logprobs"]),
        _ptr(out["lse"]), _ptr(out["max"]), _ptr(out["argmax"]), _ptr(out["top1"]),
        _ptr(out["top2"]), _ptr(out["thresh_ties"]))
    if rc != 0:
        raise OracleError("dso_sample_cells_ex returned %d" % rc)
    return out


def greedy_rows(bits, n, V, rows=None):
    """Greedy oracle: per listed row of bf16 logits [n][V], (max, lse, argmax)."""
    bits = _c(bits, np.uint16)
    if rows is None:
        rows = np.arange(int(n), dtype=np.int64)
    rows = _c(rows, np.int64)
    k = int(rows.shape[0])
    mx = np.zeros(k, np.float32)
    lse = np.zeros(k, np.float64)
    am = np.zeros(k, np.int32)
    rc = lib().dso_greedy_rows(_ptr(bits), int(n), int(V), _ptr(rows), k, _ptr(mx), _ptr(lse),
                               _ptr(am))
    if rc != 0:
        raise OracleError("dso_greedy_rows returned %d" % rc)
    return {"max": mx, "lse": lse, "argmax": am}


def merge_triples(maxes, lses, local_argmax, shard_base):
    maxes = _c(maxes, np.float32)
    lses = _c(lses, np.float64)
    local_argmax = _c(local_argmax, np.int32)
    shard_base = _c(shard_base, np.int32)
    om = np.zeros(1, np.float32)
    ol = np.zeros(1, np.float64)
    oa = np.zeros(1, np.int32)
    lib().dso_merge_triples(_ptr(maxes), _ptr(lses), _ptr(local_argmax), _ptr(shard_base),
                            int(maxes.shape[0]), _ptr(om), _ptr(ol), _ptr(oa))
    return float(om[0]), float(ol[0]), int(oa[0])


def reveal(scores, tokens, seq_lens, reveal_counts, canvas):
    """Confidence ranking and reveal (see dso_reveal): returns (new canvas, revealed flags)."""
    scores = _c(scores, np.float32)
    C, P = scores.shape
    tokens = _c(tokens, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    reveal_counts = _c(reveal_counts, np.int32)
    out = np.array(canvas, dtype=np.int32, copy=True, order="C")
    rev = np.zeros((C, P), np.uint8)
    rc = lib().dso_reveal(_ptr(scores), _ptr(tokens), _ptr(seq_lens), _ptr(reveal_counts),
                          int(seq_lens.shape[0]), int(C), int(P), _ptr(out), _ptr(rev))
    if rc != 0:
        raise OracleError("dso_reveal returned %d" % rc)
    return out, rev
