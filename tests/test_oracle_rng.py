"""Pins of the oracle's random-number path: Philox4x32-10, the uniform map and the Gumbel map.

Philox is pinned two ways that do not go through the oracle's own code: the
known-answer vectors distributed with the algorithm's reference library
(tests/golden/philox4x32_10_kat.txt) and PyTorch's independent header-only
Philox engine, compiled here as a separate program.
"""
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _kat_rows():
    rows = []
    with open(os.path.join(HERE, "golden", "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v = [int(x, 16) for x in line.split()]
            rows.append((v[0:4], v[4:6], v[6:10]))
    return rows


def test_philox_known_answers():
    rows = _kat_rows()
    assert len(rows) == 3
    for ctr, key, expect in rows:
        got = oracle.philox4x32_10(ctr, key)
        assert [int(x) for x in got] == expect


def _torch_include():
    import torch
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    if not os.path.exists(os.path.join(inc, "ATen", "core", "PhiloxRNGEngine.h")):
        return None
    return inc


def test_philox_matches_torch_header_engine():
    """PyTorch's at::philox_engine(seed, subsequence, offset) draws Philox4x32-10 at counter
    (offset lo, offset hi, subsequence lo, subsequence hi) with key (seed lo, seed hi)."""
    inc = _torch_include()
    if inc is None or shutil.which("g++") is None:
        pytest.skip("torch Philox header or g++ not available")
    src = r'''
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
#include <cstdint>
int main() {
  unsigned long long s, sub, off;
  while (std::scanf("%llu %llu %llu", &s, &sub, &off) == 3) {
    at::philox_engine e(s, sub, off);
    uint32_t a = e(), b = e(), c = e(), d = e();
    std::printf("%u %u %u %u\n", a, b, c, d);
  }
  return 0;
}
'''
    rng = np.random.Generator(np.random.PCG64(7))
    cases = [(int(rng.integers(0, 2**63)), int(rng.integers(0, 2**63)), int(rng.integers(0, 2**63)))
             for _ in range(200)]
    cases += [(0, 0, 0), (2**64 - 1, 2**64 - 1, 2**64 - 1), (3, (5 << 32) | 1000, (7 << 32) | 11)]
    with tempfile.TemporaryDirectory() as td:
        cpp = os.path.join(td, "p.cpp")
        exe = os.path.join(td, "p")
        with open(cpp, "w") as f:
            f.write(src)
        r = subprocess.run(["g++", "-std=c++17", "-O1", "-I", inc, cpp, "-o", exe],
                           capture_output=True, text=True)
        if r.returncode != 0:
            pytest.skip("could not compile against torch's Philox header: " + r.stderr[-300:])
        inp = "".join("%d %d %d\n" % c for c in cases)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
    lines = out.strip().split("\n")
    assert len(lines) == len(cases)
    for (seed, sub, off), line in zip(cases, lines):
        ctr = [off & 0xFFFFFFFF, off >> 32, sub & 0xFFFFFFFF, sub >> 32]
        key = [seed & 0xFFFFFFFF, seed >> 32]
        assert [int(x) for x in oracle.philox4x32_10(ctr, key)] == [int(x) for x in line.split()]


def test_uniform_map_closed_form():
    # U = ((x >> 8) + 1/2) / 2^24: lattice midpoints, never 0 or 1.
    assert oracle.uniform(0) == 0.5 / 2**24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 0.5 / 2**24
    assert oracle.uniform(0x80000000) == 0.5 + 0.5 / 2**24
    assert oracle.uniform(0x000000FF) == oracle.uniform(0)  # low 8 bits unused
    assert oracle.uniform(0x00000100) == 1.5 / 2**24


def test_gumbel_map_against_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    for x in [0, 1 << 8, 0x12345678, 0x7FFFFF00, 0x80000000, 0xFFFFFE00, 0xFFFFFF00, 0xFFFFFFFF]:
        u = mpmath.mpf((x >> 8)) + mpmath.mpf(1) / 2
        u = u / mpmath.mpf(2) ** 24
        want = -mpmath.log(-mpmath.log(u))
        got = oracle.gumbel(x)
        assert abs(got - float(want)) <= 1e-12 * max(1.0, abs(float(want)))
    # extremes: G ranges over about [-2.85, 17.33]
    assert -2.9 < oracle.gumbel(0) < -2.8
    assert 17.3 < oracle.gumbel(0xFFFFFFFF) < 17.4


def test_philox_stream_is_uniform():
    """Kolmogorov-Smirnov on U over a block of Philox outputs, and the Gumbel mean (Euler's gamma)."""
    from scipy import stats
    xs = []
    for i in range(4000):
        xs.extend(int(v) for v in oracle.philox4x32_10([i, 17, 1000, 5 << 8], [3, 0]))
    u = np.array([oracle.uniform(x) for x in xs])
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    g = np.array([oracle.gumbel(x) for x in xs])
    euler_gamma = 0.5772156649015329
    assert abs(g.mean() - euler_gamma) < 5 * (math.pi / math.sqrt(6)) / math.sqrt(len(g))
    assert abs(g.var() - math.pi ** 2 / 6) < 0.1
