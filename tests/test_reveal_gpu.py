"""Parity of ds_reveal (confidence ranking and reveal, "Sampler support for
discrete diffusion", Hert4's first comment) with the oracle: the committed
canvas and the committed-cell flags are compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import vocab_wide_logit_gb300 as pkg
from vocab_wide_logit_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _dev():
    assert torch.cuda.is_available(), "needs a GPU"
    return torch.device("cuda", 0)


def _run(scores, tokens, seq_lens, counts, canvas):
    dev = _dev()
    s = torch.from_numpy(np.ascontiguousarray(scores, np.float32)).to(dev)
    t = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).to(dev)
    sl = torch.from_numpy(np.asarray(seq_lens, np.int32)).to(dev)
    rc = torch.from_numpy(np.asarray(counts, np.int32)).to(dev)
    cv = torch.from_numpy(np.ascontiguousarray(canvas, np.int32)).to(dev)
    rev = pkg.reveal(s, t, sl, rc, cv)
    torch.cuda.synchronize()
    return cv.cpu().numpy(), rev.cpu().numpy()


def test_reveal_after_sampling_config3():
    dev = _dev()
    inp = wl.config3()
    c = inp.c_logits.to(dev)
    u = inp.u_logits.to(dev)
    tok, lp = pkg.sample(torch.from_numpy(inp.request_ids).to(dev), c, u,
                         torch.from_numpy(inp.seq_lens).to(dev), torch.from_numpy(inp.guidance).to(dev),
                         torch.from_numpy(inp.temperature).to(dev), inp.top_ratio, inp.seed, 0)
    tokens = tok.cpu().numpy()
    scores = lp.cpu().numpy()
    rng = np.random.Generator(np.random.PCG64(12))
    counts = (inp.C * inp.seq_lens * rng.uniform(0.0, 0.3, size=inp.B)).astype(np.int32)
    counts[0], counts[1], counts[2] = 0, -3, inp.C * int(inp.seq_lens[2]) + 5
    canvas = np.full((inp.C, inp.P), 1024, np.int32)
    got = _run(scores, tokens, inp.seq_lens, counts, canvas)
    want = oracle.reveal(scores, tokens, inp.seq_lens, counts, canvas)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1], want[1])


@pytest.mark.parametrize("levels", [2, 5, 40, 300, 0])
def test_reveal_with_ties_and_signed_zeros(levels):
    """Requests of up to 4 x 2049 cells are ranked in shared memory; the 4 x 4500 one (18000 cells,
    above the staging budget) by the 64-bit select over global memory."""
    rng = np.random.Generator(np.random.PCG64(levels + 40))
    C, seq_lens = 4, np.array([0, 1, 17, 300, 2049, 64, 4500], np.int32)
    P = int(seq_lens.sum())
    if levels:
        scores = (rng.integers(0, levels, size=(C, P)) - levels // 2).astype(np.float32)
        scores[rng.random((C, P)) < 0.3] = -0.0  # -0 and +0 tie
    else:
        scores = rng.standard_normal((C, P)).astype(np.float32)
        scores[0, :50] = -np.inf
    tokens = rng.integers(0, 100000, size=(C, P)).astype(np.int32)
    counts = np.array([3, 1, 20, 600, 1, C * 64, 7001], np.int32)
    canvas = rng.integers(-5, 0, size=(C, P)).astype(np.int32)
    got = _run(scores, tokens, seq_lens, counts, canvas)
    want = oracle.reveal(scores, tokens, seq_lens, counts, canvas)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1], want[1])


def test_reveal_reports_a_bad_layout_and_writes_nothing():
    dev = _dev()
    C, P = 2, 10
    s = torch.zeros((C, P), dtype=torch.float32, device=dev)
    t = torch.ones((C, P), dtype=torch.int32, device=dev)
    cv = torch.full((C, P), 7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sl = torch.tensor([4, 5], dtype=torch.int32, device=dev)  # sums to 9, not 10
    rc = torch.tensor([3, 3], dtype=torch.int32, device=dev)
    pkg.ds_reveal(s, t, sl, rc, cv, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) & pkg.DS_DEV_ERR_LAYOUT
    assert (cv == 7).all()
