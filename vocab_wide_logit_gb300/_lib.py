"""ctypes binding of libdsample (argument marshalling only).

Every step of the sampling and greedy passes runs in the CUDA library; this
module only turns torch tensors into device pointers and the current CUDA
stream into a handle. There is no fallback: if the library is missing the
import of a call raises.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libdsample.so")

DS_OK = 0
DS_ERR_INVALID_ARG = 1
DS_ERR_UNSUPPORTED = 2
DS_ERR_CUDA = 3
DS_DEV_ERR_LAYOUT = 1
DS_DEV_ERR_NO_UNCOND = 2
DS_DEV_ERR_PARAM = 4
DS_MAX_VOCAB = 524281

EXPORTED = ("ds_sample", "ds_greedy_lse", "ds_status_string", "ds_top_k", "ds_merge_triples", "ds_log_softmax",
            "ds_reveal", "ds_sample_ex", "ds_launch_count")
DS_FLAG_KEEP_TIES = 1
DS_FLAG_SKIP_EXACT_PASS = 2
DS_MARKED = -2
DS_DTYPE_F32 = 0
DS_DTYPE_BF16 = 1

_lib = None


class DsError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (fn, status_string(code), code))


def load(path: str = LIB_PATH):
    """Load libdsample.so (raises OSError when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError("libdsample.so not built at %s: run __graft_entry__.build() or "
                      "python vocab_wide_logit_gb300/build.py" % path)
    L = ctypes.CDLL(path)
    vp, i32, u32, u64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float
    L.ds_sample.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, f32, u64, u32, vp, vp, vp, vp]
    L.ds_sample.restype = ctypes.c_int
    L.ds_greedy_lse.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    L.ds_greedy_lse.restype = ctypes.c_int
    L.ds_status_string.argtypes = [ctypes.c_int]
    L.ds_status_string.restype = ctypes.c_char_p
    L.ds_top_k.argtypes = [f32, i32]
    L.ds_top_k.restype = i32
    L.ds_launch_count.argtypes = []
    L.ds_launch_count.restype = ctypes.c_uint64
    L.ds_merge_triples.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    L.ds_merge_triples.restype = ctypes.c_int
    L.ds_log_softmax.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp]
    L.ds_log_softmax.restype = ctypes.c_int
    L.ds_reveal.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp]
    L.ds_reveal.restype = ctypes.c_int
    L.ds_sample_ex.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, f32, u64, vp, u32, u32, vp, vp, vp,
                               vp]
    L.ds_sample_ex.restype = ctypes.c_int
    _lib = L
    return L


def status_string(code: int) -> str:
    return load().ds_status_string(int(code)).decode()


def top_k(top_ratio: float, V: int) -> int:
    return int(load().ds_top_k(float(top_ratio), int(V)))


def launch_count() -> int:
    """Kernels the library has launched in this process so far (ds_launch_count)."""
    return int(load().ds_launch_count())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def ds_sample(request_ids, c_logits, u_logits, seq_lens, guidance, temperature, top_ratio, seed,
              iteration, out_tokens, out_logprobs, d_status=None, B=None, C=None, P=None, V=None,
              stream=None, check=True, top_ratios=None, iterations=None, keep_ties=False, flags=0):
    """Call ds_sample (ds_sample_ex when per-request top_ratios / iterations are given) on device
    tensors. Shapes: c_logits [C, P, V] bf16, u_logits [C, P_u, V] bf16 or None,
    request_ids/seq_lens int32 [B], guidance/temperature float32 [B], top_ratios float32 [B] or
    None, iterations int32/uint32 [B] or None, out_tokens int32 [C, P], out_logprobs float32
    [C, P], d_status uint32/int32 [1] or None. flags: extra DS_FLAG_* bits (keep_ties sets
    DS_FLAG_KEEP_TIES)."""
    if C is None:
        C, P, V = c_logits.shape
    if B is None:
        B = seq_lens.shape[0]
    flags = int(flags) | (DS_FLAG_KEEP_TIES if keep_ties else 0)
    if top_ratios is None and iterations is None and flags == 0:
        rc = load().ds_sample(_ptr(request_ids), _ptr(c_logits), _ptr(u_logits), _ptr(seq_lens), int(B),
                              int(C), int(P), int(V), _ptr(guidance), _ptr(temperature), float(top_ratio),
                              int(seed) & (2 ** 64 - 1), int(iteration), _ptr(out_tokens), _ptr(out_logprobs),
                              _ptr(d_status), _stream(stream))
        name = "ds_sample"
    else:
        rc = load().ds_sample_ex(_ptr(request_ids), _ptr(c_logits), _ptr(u_logits), _ptr(seq_lens), int(B),
                                 int(C), int(P), int(V), _ptr(guidance), _ptr(temperature), _ptr(top_ratios),
                                 float(top_ratio), int(seed) & (2 ** 64 - 1), _ptr(iterations), int(iteration),
                                 flags, _ptr(out_tokens), _ptr(out_logprobs),
                                 _ptr(d_status), _stream(stream))
        name = "ds_sample_ex"
    if check and rc != DS_OK:
        raise DsError(name, rc)
    return rc


def ds_greedy_lse(logits, out_max, out_lse, out_argmax, n=None, V=None, stream=None, check=True):
    """Call ds_greedy_lse on device tensors: logits [n, V] bf16, outputs [n] float32/float32/int32."""
    if n is None:
        n, V = logits.shape
    rc = load().ds_greedy_lse(_ptr(logits), int(n), int(V), _ptr(out_max), _ptr(out_lse), _ptr(out_argmax),
                              _stream(stream))
    if check and rc != DS_OK:
        raise DsError("ds_greedy_lse", rc)
    return rc


def ds_merge_triples(triples, out_max, out_lse, out_argmax, n=None, shards=None, stream=None, check=True):
    """Call ds_merge_triples: triples float32 [n, shards, 3] (max, lse, global argmax bits)."""
    if n is None:
        n, shards = triples.shape[0], triples.shape[1]
    rc = load().ds_merge_triples(_ptr(triples), int(n), int(shards), _ptr(out_max), _ptr(out_lse),
                                 _ptr(out_argmax), _stream(stream))
    if check and rc != DS_OK:
        raise DsError("ds_merge_triples", rc)
    return rc


def ds_log_softmax(logits, out, out_max, out_lse, out_argmax, out_dtype=None, n=None, V=None, stream=None,
                   check=True):
    """Call ds_log_softmax: logits [n, V] bf16; out [n, V] float32 or bfloat16."""
    import torch
    if n is None:
        n, V = logits.shape
    if out_dtype is None:
        out_dtype = DS_DTYPE_BF16 if out.dtype == torch.bfloat16 else DS_DTYPE_F32
    rc = load().ds_log_softmax(_ptr(logits), int(n), int(V), _ptr(out), int(out_dtype), _ptr(out_max),
                               _ptr(out_lse), _ptr(out_argmax), _stream(stream))
    if check and rc != DS_OK:
        raise DsError("ds_log_softmax", rc)
    return rc


def ds_reveal(scores, tokens, seq_lens, reveal_counts, canvas, revealed=None, d_status=None, B=None, C=None,
              P=None, stream=None, check=True):
    """Call ds_reveal: scores float32 [C, P], tokens/canvas int32 [C, P], seq_lens/reveal_counts int32 [B],
    revealed uint8 [C, P] or None."""
    if C is None:
        C, P = scores.shape
    if B is None:
        B = seq_lens.shape[0]
    rc = load().ds_reveal(_ptr(scores), _ptr(tokens), _ptr(seq_lens), _ptr(reveal_counts), int(B), int(C),
                          int(P), _ptr(canvas), _ptr(revealed), _ptr(d_status), _stream(stream))
    if check and rc != DS_OK:
        raise DsError("ds_reveal", rc)
    return rc
