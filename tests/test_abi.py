"""CPU checks of the C ABI: the library loads without a GPU, exports every symbol the public
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import oracle
import vocab_wide_logit_gb300 as pkg
from vocab_wide_logit_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from vocab_wide_logit_gb300 import build
    build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(ds_[a-z_0-9]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"ds_sample", "ds_greedy_lse", "ds_status_string", "ds_top_k"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(_lib.EXPORTED) == names


def test_status_strings(lib):
    for code in range(4):
        assert pkg.status_string(code)
    assert pkg.status_string(99) == "unknown status"


def test_top_k_matches_oracle_definition(lib):
    for V in (1, 2, 7, 100, 1025, 4097, 248320, 262137, 262144, 524281):
        for ratio in (1e-7, 0.001, 0.05, 0.1, 0.25, 1 / 3, 0.5, 0.9, 0.999, 1.0):
            assert pkg.top_k(ratio, V) == oracle.top_k(ratio, V), (ratio, V)
    assert pkg.top_k(0.0, 10) == 0 and pkg.top_k(1.5, 10) == 0 and pkg.top_k(0.5, 0) == 0


FAKE = ctypes.c_void_p(0x100000)  # never dereferenced: every call below fails validation first


def _sample(lib, B=1, C=1, P=1, V=8, ratio=0.1, it=0, ptr=FAKE, c=FAKE):
    return lib.ds_sample(ptr, c, None, ptr, B, C, P, V, ptr, ptr, ratio, 0, it, ptr, ptr, None, None)


def test_host_side_argument_errors(lib):
    assert _sample(lib, V=0) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, ratio=0.0) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, ratio=1.01) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, ratio=float("nan")) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, C=257) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, B=-1) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, it=1 << 24) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, B=0, P=3) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, ptr=None) == _lib.DS_ERR_INVALID_ARG
    assert _sample(lib, c=ctypes.c_void_p(0x100001)) == _lib.DS_ERR_INVALID_ARG  # bf16 needs 2-byte alignment
    assert _sample(lib, V=_lib.DS_MAX_VOCAB + 1) == _lib.DS_ERR_UNSUPPORTED
    # empty calls are valid no-ops
    assert _sample(lib, C=0) == _lib.DS_OK
    assert _sample(lib, P=0) == _lib.DS_OK
    assert lib.ds_greedy_lse(FAKE, 0, 10, FAKE, FAKE, FAKE, None) == _lib.DS_OK
    assert lib.ds_greedy_lse(FAKE, 3, 0, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_greedy_lse(None, 3, 10, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG


def test_merge_and_log_softmax_argument_errors(lib):
    # ds_merge_triples
    assert lib.ds_merge_triples(FAKE, 0, 4, FAKE, FAKE, FAKE, None) == _lib.DS_OK
    assert lib.ds_merge_triples(FAKE, 5, 0, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_merge_triples(FAKE, -1, 4, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_merge_triples(None, 5, 4, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_merge_triples(ctypes.c_void_p(0x100002), 5, 4, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG
    # ds_log_softmax
    f32, bf16 = _lib.DS_DTYPE_F32, _lib.DS_DTYPE_BF16
    assert lib.ds_log_softmax(FAKE, 0, 10, FAKE, f32, FAKE, FAKE, FAKE, None) == _lib.DS_OK
    assert lib.ds_log_softmax(FAKE, 2, 0, FAKE, f32, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_log_softmax(FAKE, 2, 10, FAKE, 7, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_log_softmax(FAKE, 2, 10, None, f32, FAKE, FAKE, FAKE, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_log_softmax(FAKE, 2, 10, ctypes.c_void_p(0x100002), f32, FAKE, FAKE, FAKE,
                              None) == _lib.DS_ERR_INVALID_ARG  # fp32 output needs 4-byte alignment
    assert lib.ds_log_softmax(FAKE, 2, 10, ctypes.c_void_p(0x100001), bf16, FAKE, FAKE, FAKE,
                              None) == _lib.DS_ERR_INVALID_ARG


def test_python_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(OSError):
        saved = _lib._lib
        _lib._lib = None
        try:
            _lib.load(str(tmp_path / "missing.so"))
        finally:
            _lib._lib = saved


def test_reveal_argument_errors(lib):
    f = FAKE
    assert lib.ds_reveal(f, f, f, f, 2, 0, 10, f, None, None, None) == _lib.DS_OK
    assert lib.ds_reveal(f, f, f, f, 0, 3, 0, f, None, None, None) == _lib.DS_OK
    assert lib.ds_reveal(f, f, f, f, 0, 3, 5, f, None, None, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_reveal(f, f, f, f, -1, 3, 5, f, None, None, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_reveal(None, f, f, f, 2, 3, 5, f, None, None, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_reveal(f, f, f, f, 2, 3, 5, None, None, None, None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_reveal(ctypes.c_void_p(0x100002), f, f, f, 2, 3, 5, f, None, None,
                         None) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_reveal(f, f, f, f, 2, 256, 1 << 24, f, None, None, None) == _lib.DS_ERR_UNSUPPORTED


def test_sample_ex_argument_errors(lib):
    f = FAKE

    def ex(ratios=None, ratio=0.1, iters=None, it=0, V=8, flags=0):
        return lib.ds_sample_ex(f, f, None, f, 1, 1, 1, V, f, f, ratios, ratio, 0, iters, it, flags, f, f, None, None)

    # the scalars are checked only when no per-request array replaces them
    assert ex(ratio=0.0) == _lib.DS_ERR_INVALID_ARG
    assert ex(it=1 << 24) == _lib.DS_ERR_INVALID_ARG
    assert ex(ratios=ctypes.c_void_p(0x100002), ratio=0.0) == _lib.DS_ERR_INVALID_ARG  # misaligned array
    assert ex(iters=ctypes.c_void_p(0x100001), it=1 << 24) == _lib.DS_ERR_INVALID_ARG
    assert ex(V=_lib.DS_MAX_VOCAB + 1) == _lib.DS_ERR_UNSUPPORTED
    assert ex(flags=4) == _lib.DS_ERR_INVALID_ARG
    assert lib.ds_sample_ex(f, f, None, f, 1, 0, 1, 8, f, f, None, 0.1, 0, None, 0, 1, f, f, None, None) == _lib.DS_OK
