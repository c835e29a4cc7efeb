"""Pins of the GPU side's Gumbel bound table (gen_gumbel_bounds.py), checked against the mathematics.

Every pruning decision of the sampling kernels trusts lo <= G(x) <= hi for the bucket of the
Philox word x, with G = -log(-log U) and U = ((x >> 8) + 1/2) 2^-24. A bucket whose bounds were
too tight would drop a token that can win the race, and only a rare token mismatch would show
it, so the table is checked here for every one of the 2^24 values of j = x >> 8:

- in double, vectorised: lo <= G(j) <= hi for all j, with 1 - U formed exactly near U = 1;
- at the bucket edges (G increases with j), in 50-digit arithmetic;
- the bounds are also tight enough to be useful (a loose bound only costs time, but a table
  that was, say, shifted by one bucket would be loose at one end and wrong at the other).
"""
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GEN = os.path.join(ROOT, "vocab_wide_logit_gb300", "csrc", "gen_gumbel_bounds.py")


def _table():
    with tempfile.TemporaryDirectory() as td:
        out = os.path.join(td, "t.inc")
        subprocess.run([sys.executable, GEN, out], check=True)
        with open(out) as f:
            text = f.read()
    shift = None
    rows = []
    for line in text.splitlines():
        line = line.strip()
        if line.startswith("#define DS_GUMBEL_BUCKET_SHIFT"):
            shift = int(line.split()[-1])
        elif line.startswith("{") and line.endswith("},"):
            a, b = line[1:-2].split(",")
            rows.append((float.fromhex(a.strip().rstrip("f")), float.fromhex(b.strip().rstrip("f"))))
    t = np.array(rows, dtype=np.float64)
    return shift, t[:, 0], t[:, 1]


def _gumbel_all_j():
    """G(j) for every 24-bit j, in double."""
    j = np.arange(1 << 24, dtype=np.float64)
    g = np.empty_like(j)
    half = 1 << 23
    u = (j[:half] + 0.5) * 2.0 ** -24
    g[:half] = -np.log(-np.log(u))
    w = ((1 << 24) - j[half:] - 0.5) * 2.0 ** -24  # 1 - U, exact
    g[half:] = -np.log(-np.log1p(-w))
    return g


def test_table_shape_and_values_are_fp32():
    shift, lo, hi = _table()
    assert shift == 21 and lo.size == 2048 and hi.size == 2048
    assert np.array_equal(lo.astype(np.float32).astype(np.float64), lo)
    assert np.array_equal(hi.astype(np.float32).astype(np.float64), hi)
    assert np.all(lo < hi)
    # buckets are ordered: G increases with the word
    assert np.all(np.diff(lo) > 0) and np.all(np.diff(hi) > 0)


def test_bounds_hold_for_every_24_bit_word():
    shift, lo, hi = _table()
    g = _gumbel_all_j()
    b = np.arange(1 << 24) >> (shift - 8)  # bucket of j = x >> 8
    assert np.all(lo[b] <= g), "a lower bound exceeds G at j = %d" % int(np.argmax(lo[b] > g))
    assert np.all(g <= hi[b]), "an upper bound is below G at j = %d" % int(np.argmax(g > hi[b]))
    # tight: each bound sits within 1e-6 (relative) of G at its end of the bucket
    per = 1 << (shift - 8)
    first = g[::per]
    last = g[per - 1::per]
    assert np.all(first - lo <= 1e-6 * np.maximum(1.0, np.abs(first)))
    assert np.all(hi - last <= 1e-6 * np.maximum(1.0, np.abs(last)))


def test_bucket_edges_in_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    shift, lo, hi = _table()
    per = 1 << (shift - 8)
    two24 = mpmath.mpf(2) ** 24

    def G(j):
        u = (mpmath.mpf(j) + mpmath.mpf(1) / 2) / two24
        return -mpmath.log(-mpmath.log(u))

    for b in list(range(0, 2048, 7)) + [1, 1023, 1024, 2046, 2047]:
        assert mpmath.mpf(lo[b]) <= G(b * per), b
        assert G((b + 1) * per - 1) <= mpmath.mpf(hi[b]), b
    # the whole range the kernels assume: G in [lo[0], hi[2047]] for every word
    assert mpmath.mpf(lo[0]) <= G(0) and G((1 << 24) - 1) <= mpmath.mpf(hi[-1])
    assert -2.9 < lo[0] < -2.8 and 17.3 < hi[-1] < 17.4
