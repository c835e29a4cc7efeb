"""Pin of the noise counter layout, by a brute-force race at nonzero position, row and iteration.

The sampler keys each vocabulary id's Gumbel draw on Philox4x32-10 with
counter = (id >> 2, t, request_id, iteration << 8 | row) and key = (seed low, seed high), and
takes word (id & 3) of the output block ("Sampler support for discrete diffusion", Hert4's first
comment, asks for Gumbel sampling and leaves the keying open; this layout is the library's
stated reading). The race here is written out from the pinned primitives (oracle.philox4x32_10,
checked against the Random123 known answers and torch's engine; oracle.gumbel, checked in
50-digit arithmetic), with the kept set from a full numpy sort, and must give the oracle's token
at every cell. Rows, positions and iterations are all nonzero and distinct, so a layout with t and
the row swapped, a wrong shift of the iteration, a global instead of request-local position, the
request index in place of its id, or swapped key words, each changes some token, which the test
also checks, so the pin has the power to see those mistakes.
"""
import numpy as np

import oracle
from vocab_wide_logit_gb300 import workloads as wl

V = 37
RATIO = 0.5           # k = ceil(18.5) = 19 kept of 37
TAU = 1.7             # hot enough that the noise decides most cells
SEED = (0x9E3779B97F4A7C15 ^ 0x1234) & (2 ** 64 - 1)
ITERATION = 0xA5A5A5  # < 2^24, bits on both sides of any plausible shift
SEQ = np.array([3, 5, 4], np.int32)
RIDS = np.array([1000 + 7919 * r for r in range(3)], np.int32)
C = 3


def _inputs():
    rng = np.random.Generator(np.random.PCG64(404))
    P = int(SEQ.sum())
    z = (rng.standard_normal((C, P, V)) * 1.5).astype(np.float32)
    c = wl.to_bf16(z)
    return c, c.float().numpy()  # z = c exactly (guidance 0)


def _race(z_row, k, ctr_fn, key):
    order = np.lexsort((np.arange(V), -z_row.astype(np.float64)))  # z desc, id asc
    kept = order[:k]
    best, best_s = None, -np.inf
    for i in sorted(int(v) for v in kept):
        words = oracle.philox4x32_10(ctr_fn(i), key)
        s = float(z_row[i]) + TAU * oracle.gumbel(int(words[i & 3]))
        if s > best_s:
            best, best_s = i, s
    return best


def _layouts():
    key = [SEED & 0xFFFFFFFF, SEED >> 32]
    swapped_key = [SEED >> 32, SEED & 0xFFFFFFFF]
    return {
        "stated": (lambda i, t, p, r, rid, row: [i >> 2, t, rid, (ITERATION << 8) | row], key),
        "t and row swapped": (lambda i, t, p, r, rid, row: [i >> 2, row, rid, (ITERATION << 8) | t], key),
        "iteration shifted by 16": (lambda i, t, p, r, rid, row: [i >> 2, t, rid,
                                                                  ((ITERATION << 16) | row) & 0xFFFFFFFF], key),
        "global position": (lambda i, t, p, r, rid, row: [i >> 2, p, rid, (ITERATION << 8) | row], key),
        "request index for id": (lambda i, t, p, r, rid, row: [i >> 2, t, r, (ITERATION << 8) | row], key),
        "key words swapped": (lambda i, t, p, r, rid, row: [i >> 2, t, rid, (ITERATION << 8) | row], swapped_key),
    }


def test_noise_layout_brute_force_at_nonzero_position_row_and_iteration():
    c, z = _inputs()
    P = int(SEQ.sum())
    k = oracle.top_k(RATIO, V)
    assert k == 19
    bits = wl.bf16_bits(c)
    zeros = np.zeros(len(SEQ), np.float32)
    tau = np.full(len(SEQ), TAU, np.float32)
    ref = oracle.sample_cells(RIDS, bits, None, SEQ, C, P, V, zeros, tau, RATIO, SEED, ITERATION)
    tokens = ref["tokens"].reshape(C, P)
    offs = np.concatenate([[0], np.cumsum(SEQ)[:-1]])
    diffs = {name: 0 for name in _layouts()}
    for row in range(C):
        for p in range(P):
            r = int(np.searchsorted(offs, p, side="right") - 1)
            t = p - int(offs[r])
            for name, (ctr, key) in _layouts().items():
                tok = _race(z[row, p], k, lambda i: [v & 0xFFFFFFFF for v in ctr(i, t, p, r, int(RIDS[r]), row)],
                            key)
                if name == "stated":
                    assert tok == int(tokens[row, p]), (row, p)
                elif tok != int(tokens[row, p]):
                    diffs[name] += 1
    # every plausible mistake in the layout moves some token
    for name, n in diffs.items():
        if name != "stated":
            assert n > 0, name
