"""Pins of the sampling oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than its own code: exact
rational arithmetic, high-precision logsumexp, a full sort, numpy/torch library
routines, closed-form distributions (chi-square), invariants and the printed
rules of the pages (ceil(0.1 * V); smallest-ID ties; p = exp(z - lse)).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from vocab_wide_logit_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
PAGES = json.load(open(os.path.join(HERE, "golden", "pages_constants.json")))


# ---------------------------------------------------------------------------- helpers
def round_to_f32(q: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) fp32 value of an exact rational."""
    f = np.float32(float(q))
    best = None
    for cand in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        err = abs(Fraction(float(cand)) - q)
        if best is None or err < best[0] or (err == best[0] and (int(cand.view(np.uint32)) & 1) == 0):
            best = (err, cand)
    return np.float32(best[1])


def single_request(z_rows_bits, V, g=0.0, tau=1.0, ratio=1.0, seed=0, iteration=0, rid=1000, u_bits=None):
    """Run the oracle on one request whose rows are given as bf16 bit patterns [P, V] (C = 1)."""
    P = z_rows_bits.shape[0]
    return oracle.sample_cells([rid], z_rows_bits.reshape(-1), None if u_bits is None else u_bits.reshape(-1),
                               [P], 1, P, V, [g], [tau], ratio, seed, iteration)


def bits_of(values):
    return wl.bf16_bits(wl.to_bf16(np.asarray(values, np.float32)))


# ---------------------------------------------------------------------------- decode and combine
def test_bf16_decode_matches_torch_for_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_to_float(int(h)) for h in pats], dtype=np.float32)
    finite = ~np.isnan(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))


def test_cfg_combine_is_exactly_rounded():
    """z = c + g (c - u): fp32 difference, then a single rounding of g*d + c (exact rationals)."""
    rng = np.random.Generator(np.random.PCG64(11))
    c = wl.to_bf16(rng.standard_normal(3000).astype(np.float32) * 4).float().numpy()
    u = wl.to_bf16(c + rng.standard_normal(3000).astype(np.float32) * 2).float().numpy()
    gs = np.array([0.5, 1.5, 2.0, 3.7, 7.25, 0.1], np.float32)
    for i in range(3000):
        g = gs[i % len(gs)]
        d = round_to_f32(Fraction(float(c[i])) - Fraction(float(u[i])))
        want = round_to_f32(Fraction(float(g)) * Fraction(float(d)) + Fraction(float(c[i])))
        got = np.float32(oracle.cfg(c[i], u[i], g))
        assert got.view(np.uint32) == want.view(np.uint32), (c[i], u[i], g)
    # guidance 0: the unconditional logits are not used at all
    for i in range(50):
        assert np.float32(oracle.cfg(c[i], np.float32(np.nan), 0.0)) == c[i]


# ---------------------------------------------------------------------------- kept count
def test_top_k_pins_from_the_pages():
    rule = PAGES["top_ratio_rule"]
    for V, k in rule["cases"]:
        assert oracle.top_k(rule["ratio"], V) == k
        assert k == math.ceil(rule["ratio"] * V - 1e-9)  # the pages' ceil(0.1 * V)
    # The product is taken in fp32: in double, 0.1f * 248320 = 24832.00037 would round up.
    assert math.ceil(float(np.float32(0.1)) * 248320) == 24833
    assert oracle.top_k(0.1, 248320) == 24832
    assert oracle.top_k(1.0, 1025) == 1025
    assert oracle.top_k(1e-9, 1025) == 1
    assert oracle.top_k(0.5, 1) == 1


# ---------------------------------------------------------------------------- lse, argmax, invariants
def test_lse_against_high_precision_and_invariants():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.Generator(np.random.PCG64(5))
    for V in (1, 2, 7, 16, 33, 200):
        for sigma in (0.5, 4.0, 30.0):
            bits = bits_of(rng.standard_normal((3, V)).astype(np.float32) * sigma).reshape(3, V)
            r = single_request(bits, V, tau=0.0)
            z = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy().reshape(3, V)
            for j in range(3):
                want = mpmath.log(mpmath.fsum(mpmath.exp(mpmath.mpf(float(v))) for v in z[j]))
                assert abs(r["lse"][j] - float(want)) <= 1e-12 * max(1.0, abs(float(want)))
                assert r["max"][j] == z[j].max()
                assert r["argmax"][j] == int(np.argmax(z[j]))  # first occurrence
                assert r["logprobs"][j] <= 0.0
                total = math.fsum(math.exp(float(v) - r["lse"][j]) for v in z[j])
                assert abs(total - 1.0) <= 1e-6
                # temperature 0: the token is the argmax and its logprob is the max log-prob
                assert r["tokens"][j] == r["argmax"][j]
                assert abs(r["logprobs"][j] - (float(z[j].max()) - r["lse"][j])) <= 1e-12


def test_lse_matches_torch_logsumexp_float64():
    rng = np.random.Generator(np.random.PCG64(6))
    V = 4097
    bits = bits_of(rng.standard_normal((4, V)).astype(np.float32) * 6).reshape(4, V)
    r = single_request(bits, V, tau=0.0)
    z = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double()
    want = torch.logsumexp(z.reshape(4, V), dim=1).numpy()
    assert np.allclose(r["lse"], want, rtol=0, atol=1e-12)


def test_smallest_id_wins_ties():
    """Ties at the maximum go to the smallest token id (greedy and temperature 0)."""
    V = 64
    row = np.linspace(-3, 1, V).astype(np.float32)
    row[[9, 40, 41]] = 2.0
    bits = bits_of(row[None, :]).reshape(1, V)
    r = single_request(bits, V, tau=0.0)
    assert r["argmax"][0] == 9 and r["tokens"][0] == 9
    gr = oracle.greedy_rows(bits.reshape(-1), 1, V)
    assert gr["argmax"][0] == 9
    assert gr["max"][0] == 2.0


def test_all_neg_inf_row():
    V = 10
    bits = bits_of(np.full((1, V), -np.inf, np.float32)).reshape(1, V)
    for tau in (0.0, 0.9):
        r = single_request(bits, V, tau=tau, ratio=0.3)
        assert r["tokens"][0] == 0
        assert r["lse"][0] == -np.inf
        assert np.isnan(r["logprobs"][0])


# ---------------------------------------------------------------------------- top-ratio set and Gumbel
def _replicated_rows(z_row, P):
    return np.tile(bits_of(z_row[None, :]).reshape(1, -1), (P, 1))


def _kept_by_full_sort(z, k):
    order = sorted(range(len(z)), key=lambda i: (-float(z[i]), i))
    return set(order[:k])


def test_kept_set_matches_full_sort_and_frequencies_match_softmax():
    """Over many independent cells with identical logits, sampled tokens stay inside the
    k largest (full sort, smallest-id ties) and follow softmax(z/tau) restricted to them."""
    from scipy import stats
    V, P, tau, ratio = 24, 30000, 1.3, 0.25
    rng = np.random.Generator(np.random.PCG64(21))
    z_row = wl.to_bf16(rng.standard_normal(V).astype(np.float32) * 1.5).float().numpy()
    z_row[5] = z_row[11] = np.sort(z_row)[-6]  # a tie inside the kept range
    k = oracle.top_k(ratio, V)
    assert k == 6
    r = single_request(_replicated_rows(z_row, P), V, tau=tau, ratio=ratio, seed=99)
    zf = wl.to_bf16(z_row).float().numpy()
    kept = _kept_by_full_sort(zf, k)
    toks = r["tokens"]
    assert set(np.unique(toks).tolist()) <= kept
    assert set(np.unique(toks).tolist()) == kept  # every kept token is reachable
    ids = sorted(kept)
    w = np.array([math.exp(float(zf[i]) / tau) for i in ids])
    counts = np.array([(toks == i).sum() for i in ids])
    chi = stats.chisquare(counts, w / w.sum() * counts.sum())
    assert chi.pvalue > 1e-3, chi
    # logprob is the unfiltered, untempered log-softmax of the sampled token
    lse = math.log(math.fsum(math.exp(float(v)) for v in zf))
    for j in range(0, P, 997):
        assert abs(r["logprobs"][j] - (float(zf[toks[j]]) - lse)) <= 1e-12


def test_threshold_ties_keep_smallest_ids():
    """Exactly k tokens are kept: at a tie straddling the cut, the smallest ids stay."""
    V, P = 12, 6000
    z_row = np.array([5, 4, 3, 3, 3, 3, 1, 0, -1, -2, -3, -4], np.float32)
    ratio = 4.0 / 12.0  # k = 4: {0, 1} and two of the four 3s
    assert oracle.top_k(ratio, V) == 4
    r = single_request(_replicated_rows(z_row, P), V, tau=5.0, ratio=ratio, seed=3)
    assert set(np.unique(r["tokens"]).tolist()) == {0, 1, 2, 3}
    assert (r["thresh_ties"] == 2).all()


def test_temperature_zero_and_k_one_reduce_to_argmax():
    rng = np.random.Generator(np.random.PCG64(8))
    V, P = 50, 300
    bits = bits_of(rng.standard_normal((P, V)).astype(np.float32) * 2).reshape(P, V)
    z = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    argmax = np.argmax(z, axis=1)
    r0 = single_request(bits, V, tau=0.0, ratio=0.5, seed=4)
    assert np.array_equal(r0["tokens"], argmax)
    for seed in (0, 1, 12345):
        r1 = single_request(bits, V, tau=3.0, ratio=1.0 / V, seed=seed)  # k = 1
        assert np.array_equal(r1["tokens"], argmax)


def test_ratio_one_is_unfiltered_gumbel_softmax():
    from scipy import stats
    V, P, tau = 8, 40000, 0.8
    z_row = np.array([0.5, 1.0, -1.0, 0.0, 2.0, 1.5, -0.5, 0.25], np.float32)
    r = single_request(_replicated_rows(z_row, P), V, tau=tau, ratio=1.0, seed=17, iteration=3)
    w = np.exp(z_row.astype(np.float64) / tau)
    counts = np.bincount(r["tokens"], minlength=V)
    assert stats.chisquare(counts, w / w.sum() * counts.sum()).pvalue > 1e-3


def test_noise_is_keyed_on_seed_iteration_and_position():
    V, P = 40, 400
    z_row = np.zeros(V, np.float32)  # uniform logits: the token is decided by the noise alone
    bits = _replicated_rows(z_row, P)
    a = single_request(bits, V, tau=1.0, ratio=1.0, seed=1, iteration=0)["tokens"]
    b = single_request(bits, V, tau=1.0, ratio=1.0, seed=1, iteration=0)["tokens"]
    c = single_request(bits, V, tau=1.0, ratio=1.0, seed=2, iteration=0)["tokens"]
    d = single_request(bits, V, tau=1.0, ratio=1.0, seed=1, iteration=1)["tokens"]
    e = single_request(bits, V, tau=1.0, ratio=1.0, seed=1, iteration=0, rid=7)["tokens"]
    assert np.array_equal(a, b)
    for other in (c, d, e):
        assert (a != other).mean() > 0.8
    # positions draw independently: roughly uniform over V
    assert len(np.unique(a)) > V * 0.9


# ---------------------------------------------------------------------------- packing
def test_mixed_batch_equals_requests_run_alone():
    """A request's cells give the same result in a mixed batch (guidance 0 requests pass no u,
    u packed over guided requests only) as when sampled alone: the noise is keyed on the request
    id and the request-local position, not on the packing."""
    inp = wl.make_sample_inputs("mix", C=3, seq_lens=[5, 3, 7, 2], V=37,
                                guidance=[2.0, 0.0, 1.5, 0.0], temperature=[0.9, 0.0, 0.7, 1.1],
                                sigma_c=2.0, sigma_u=1.0, top_ratio=0.2, seed=9)
    c_bits = wl.bf16_bits(inp.c_logits)
    u_bits = wl.bf16_bits(inp.u_logits)
    full = oracle.sample_cells(inp.request_ids, c_bits, u_bits, inp.seq_lens, inp.C, inp.P, inp.V,
                               inp.guidance, inp.temperature, inp.top_ratio, 77, 5)
    offs = np.concatenate([[0], np.cumsum(inp.seq_lens)])
    uoff = 0
    c3 = inp.c_logits
    for r in range(inp.B):
        T = int(inp.seq_lens[r])
        cr = wl.bf16_bits(c3[:, offs[r]:offs[r] + T])
        ur = None
        if inp.guidance[r] != 0:
            ur = wl.bf16_bits(inp.u_logits[:, uoff:uoff + T])
            uoff += T
        alone = oracle.sample_cells([inp.request_ids[r]], cr, ur, [T], inp.C, T, inp.V, [inp.guidance[r]],
                                    [inp.temperature[r]], inp.top_ratio, 77, 5)
        for c in range(inp.C):
            for t in range(T):
                j_full = c * inp.P + offs[r] + t
                j_alone = c * T + t
                assert full["tokens"][j_full] == alone["tokens"][j_alone]
                assert full["logprobs"][j_full] == alone["logprobs"][j_alone]


def test_layout_errors_are_reported():
    bits = bits_of(np.zeros((2, 4), np.float32)).reshape(-1)
    with pytest.raises(oracle.OracleError):  # seq_lens do not sum to P
        oracle.sample_cells([1], bits, None, [3], 1, 2, 4, [0.0], [0.0], 0.5, 0, 0)
    with pytest.raises(oracle.OracleError):  # guidance != 0 but no u
        oracle.sample_cells([1], bits, None, [2], 1, 2, 4, [1.0], [0.0], 0.5, 0, 0)


# ---------------------------------------------------------------------------- greedy and shard merge
def test_greedy_rows_against_library_routines():
    g = wl.make_greedy_inputs("t", n=24, V=3001, sigma=4.0, seed=12)
    bits = wl.bf16_bits(g.logits)
    r = oracle.greedy_rows(bits, g.n, g.V)
    x = g.logits.double()
    assert np.allclose(r["lse"], torch.logsumexp(x, dim=1).numpy(), rtol=0, atol=1e-12)
    assert np.array_equal(r["max"], g.logits.float().max(dim=1).values.numpy())
    assert np.array_equal(r["argmax"], np.argmax(g.logits.float().numpy(), axis=1))
    for row, ids in zip(g.planted_rows, g.planted_ids):
        assert r["argmax"][row] == ids.min()
    # page 3: exact selected-token probability without dense logits
    p = np.exp(r["max"].astype(np.float64) - r["lse"])
    dense = torch.softmax(x, dim=1).max(dim=1).values.numpy()
    assert np.allclose(p, dense, rtol=1e-12, atol=0)


def test_shard_merge_equals_unsharded():
    """Merging per-shard (max, lse, argmax) triples reproduces the unsharded row, with the
    smallest global id on ties across shards."""
    V, n_shards = 1000, 4
    row = np.random.Generator(np.random.PCG64(2)).standard_normal(V).astype(np.float32)
    row[[130, 620, 999]] = 9.0  # tie across shards 0, 2 and 3
    bits = bits_of(row[None, :]).reshape(-1)
    whole = oracle.greedy_rows(bits, 1, V)
    bounds = [0, 250, 500, 750, 1000]
    mx, ls, am = [], [], []
    for s in range(n_shards):
        part = bits[bounds[s]:bounds[s + 1]]
        gr = oracle.greedy_rows(part, 1, bounds[s + 1] - bounds[s])
        mx.append(gr["max"][0]); ls.append(gr["lse"][0]); am.append(gr["argmax"][0])
    m, l, a = oracle.merge_triples(mx, ls, am, bounds[:-1])
    assert m == whole["max"][0] and a == whole["argmax"][0] == 130
    assert abs(l - whole["lse"][0]) < 1e-12


# ---------------------------------------------------------------------------- per-request ratio / iteration
def test_per_request_ratio_and_iteration_equal_separate_scalar_calls():
    """A batch whose requests carry their own top ratio and iteration gives each request the
    tokens that a batch of that request alone gives with the scalars (the noise is keyed on the
    request id and the request-local position, so packing does not matter)."""
    from vocab_wide_logit_gb300 import workloads as wl
    C, V = 3, 257
    seq = np.array([5, 7, 4], np.int32)
    inp = wl.make_sample_inputs("pr", C, seq, V, [2.0, 0.0, 1.5], [0.9, 1.3, 0.5], 3.0, 1.5, 0.1, seed=9)
    ratios = np.array([0.02, 0.5, 1.0], np.float32)
    iters = np.array([0, 17, 123456], np.uint32)
    c_bits = wl.bf16_bits(inp.c_logits).reshape(C, inp.P, V)
    u_all = wl.bf16_bits(inp.u_logits).reshape(C, inp.P_u, V)
    both = oracle.sample_cells(inp.request_ids, c_bits, u_all, seq, C, inp.P, V, inp.guidance,
                               inp.temperature, 0.1, inp.seed, 0, top_ratios=ratios, iterations=iters)
    tok = both["tokens"].reshape(C, inp.P)
    lp = both["logprobs"].reshape(C, inp.P)
    off, off_u = 0, 0
    for r in range(3):
        T = int(seq[r])
        cs = np.ascontiguousarray(c_bits[:, off:off + T])
        us = np.ascontiguousarray(u_all[:, off_u:off_u + T]) if inp.guidance[r] != 0 else None
        one = oracle.sample_cells(inp.request_ids[r:r + 1], cs, us, seq[r:r + 1], C, T, V,
                                  inp.guidance[r:r + 1], inp.temperature[r:r + 1], float(ratios[r]), inp.seed,
                                  int(iters[r]))
        assert np.array_equal(one["tokens"].reshape(C, T), tok[:, off:off + T])
        assert np.array_equal(one["logprobs"].reshape(C, T), lp[:, off:off + T])
        off += T
        if inp.guidance[r] != 0:
            off_u += T
    # the iteration and the ratio do change the draw somewhere
    base = oracle.sample_cells(inp.request_ids, c_bits, u_all, seq, C, inp.P, V, inp.guidance,
                               inp.temperature, 0.1, inp.seed, 0)
    assert not np.array_equal(base["tokens"], both["tokens"])
    with pytest.raises(oracle.OracleError):
        oracle.sample_cells(inp.request_ids, c_bits, u_all, seq, C, inp.P, V, inp.guidance, inp.temperature,
                            0.1, inp.seed, 0, top_ratios=np.array([0.1, 0.0, 0.1], np.float32))
    with pytest.raises(oracle.OracleError):
        oracle.sample_cells(inp.request_ids, c_bits, u_all, seq, C, inp.P, V, inp.guidance, inp.temperature,
                            0.1, inp.seed, 0, iterations=np.array([0, 1 << 24, 0], np.uint32))


# ---------------------------------------------------------------------------- keep-ties filter mode
def _bf16_bits_of(values):
    import torch
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_keep_ties_brute_force_on_a_tiny_vocabulary():
    """Keep-ties mode against a brute-force race built from the pinned Philox and Gumbel
    primitives: the kept set is every id whose z reaches the k-th largest z."""
    V, k_ratio = 16, 0.25  # k = 4
    rng = np.random.Generator(np.random.PCG64(5))
    key = (123456789, 987)
    seed = key[0] | (key[1] << 32)
    for trial in range(40):
        # few distinct values: the cut often falls inside a run of equal z
        z = rng.integers(0, 4, size=V).astype(np.float32)
        bits = _bf16_bits_of(z).reshape(1, 1, V)
        tau = 0.8
        rid = 1000 + trial
        out = oracle.sample_cells([rid], bits, None, [1], 1, 1, V, [0.0], [tau], k_ratio, seed, 3,
                                  keep_ties=True)
        zk = np.sort(z)[::-1][oracle.top_k(k_ratio, V) - 1]
        kept = np.nonzero(z >= zk)[0]
        best, best_s = None, -np.inf
        for i in kept:
            words = oracle.philox4x32_10([i >> 2, 0, rid, (3 << 8) | 0], key)
            s = float(z[i]) + tau * oracle.gumbel(int(words[i & 3]))
            if s > best_s:
                best, best_s = int(i), s
        assert int(out["tokens"][0]) == best, trial
        assert int(out["thresh_ties"][0]) == 0


def test_keep_ties_equals_exact_k_when_the_cut_is_clean():
    from vocab_wide_logit_gb300 import workloads as wl
    inp = wl.config1()
    c_bits = wl.bf16_bits(inp.c_logits)
    u_bits = wl.bf16_bits(inp.u_logits)
    a = oracle.sample_cells(inp.request_ids, c_bits, u_bits, inp.seq_lens, inp.C, inp.P, inp.V, inp.guidance,
                            inp.temperature, inp.top_ratio, inp.seed, 0)
    b = oracle.sample_cells(inp.request_ids, c_bits, u_bits, inp.seq_lens, inp.C, inp.P, inp.V, inp.guidance,
                            inp.temperature, inp.top_ratio, inp.seed, 0, keep_ties=True)
    clean = a["thresh_ties"] == 0
    assert clean.mean() > 0.5
    assert np.array_equal(a["tokens"][clean], b["tokens"][clean])
    # where ties straddle the cut the kept set only grows: the exact-k winner's score cannot beat b's
    assert np.all(b["top1"][~clean] >= a["top1"][~clean])
