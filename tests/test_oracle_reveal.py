"""Pins of the oracle's confidence ranking and reveal ("Sampler support for
discrete diffusion", Hert4's first comment: rank the flattened canvas by score
and commit the top reveal_count), checked against a numpy lexsort, against the
invariants of a top-k selection and on hand-worked cases."""
import numpy as np
import pytest

import oracle


def _numpy_reveal(scores, tokens, seq_lens, counts, canvas):
    C, P = scores.shape
    out = canvas.copy()
    rev = np.zeros((C, P), np.uint8)
    off = 0
    for T, k in zip(seq_lens, counts):
        T = int(T)
        block = scores[:, off:off + T].reshape(-1)          # flattened f = c * T + t
        f = np.arange(block.shape[0])
        order = np.lexsort((f, -block.astype(np.float64)))  # score desc, then f asc
        k = int(min(max(int(k), 0), block.shape[0]))
        for fi in order[:k]:
            c, t = divmod(int(fi), T)
            out[c, off + t] = tokens[c, off + t]
            rev[c, off + t] = 1
        off += T
    return out, rev


def _case(rng, C, seq_lens, n_levels=None):
    P = int(np.sum(seq_lens))
    if n_levels:  # few distinct values: many exact ties
        scores = rng.integers(0, n_levels, size=(C, P)).astype(np.float32) * np.float32(0.25) - np.float32(1.0)
    else:
        scores = rng.standard_normal((C, P)).astype(np.float32)
    tokens = rng.integers(0, 1025, size=(C, P)).astype(np.int32)
    canvas = np.full((C, P), 1024, np.int32)  # every cell masked
    return scores, tokens, canvas


@pytest.mark.parametrize("n_levels", [None, 3, 1])
def test_matches_numpy_lexsort(n_levels):
    rng = np.random.Generator(np.random.PCG64(7 + (n_levels or 0)))
    for trial in range(25):
        C = int(rng.integers(1, 5))
        B = int(rng.integers(1, 6))
        seq_lens = rng.integers(0, 9, size=B).astype(np.int32)
        counts = rng.integers(-2, 40, size=B).astype(np.int32)
        scores, tokens, canvas = _case(rng, C, seq_lens, n_levels)
        got = oracle.reveal(scores, tokens, seq_lens, counts, canvas)
        want = _numpy_reveal(scores, tokens, seq_lens, counts, canvas)
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]), trial


def test_topk_invariants():
    rng = np.random.Generator(np.random.PCG64(3))
    C, seq_lens = 8, np.array([100, 37, 1, 250], np.int32)
    counts = np.array([10, 37 * 8, 5, 0], np.int32)
    scores, tokens, canvas = _case(rng, C, seq_lens, n_levels=7)
    out, rev = oracle.reveal(scores, tokens, seq_lens, counts, canvas)
    off = 0
    for T, k in zip(seq_lens, counts):
        blk = scores[:, off:off + T]
        r = rev[:, off:off + T].astype(bool)
        assert r.sum() == min(k, C * T)
        if r.any() and (~r).any():
            assert blk[r].min() >= blk[~r].max()
            # at a tied cut, the revealed cells have the smaller flattened indices
            cut = blk[r].min()
            f = np.arange(C * T).reshape(C, T)
            tied_in = f[r & (blk == cut)]
            tied_out = f[~r & (blk == cut)]
            if tied_in.size and tied_out.size:
                assert tied_in.max() < tied_out.min()
        assert np.array_equal(out[:, off:off + T][r], tokens[:, off:off + T][r])
        assert np.all(out[:, off:off + T][~r] == 1024)
        off += T


def test_worked_example():
    # one request, C = 2, T = 3: flattened scores 0.5, 0.1, 0.9 | 0.9, 0.2, 0.3
    scores = np.array([[0.5, 0.1, 0.9], [0.9, 0.2, 0.3]], np.float32)
    tokens = np.array([[10, 11, 12], [13, 14, 15]], np.int32)
    canvas = np.full((2, 3), -1, np.int32)
    out, rev = oracle.reveal(scores, tokens, [3], [3], canvas)
    # 0.9 at f = 2 before 0.9 at f = 3, then 0.5 at f = 0
    assert out.tolist() == [[10, -1, 12], [13, -1, -1]]
    assert rev.tolist() == [[1, 0, 1], [1, 0, 0]]
    out, rev = oracle.reveal(scores, tokens, [3], [0], canvas)
    assert (out == -1).all() and (rev == 0).all()
    out, rev = oracle.reveal(scores, tokens, [3], [99], canvas)
    assert np.array_equal(out, tokens) and (rev == 1).all()
