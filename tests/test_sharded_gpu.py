"""Parity of the vocabulary-sharded greedy path and of the dense log-softmax
write-out against the oracle ("perf: avoid full-vocab all-gather for draft
greedy sampling", Design and invariants).

Sharded: the vocabulary of each row is split into S shards ("ranks", emulated
in one process); each shard runs ds_greedy_lse on its own contiguous buffer,
its triple is packed as three FP32 words with the global argmax's bits in the
third, and ds_merge_triples merges them. The result must equal the unsharded
pass: max and argmax bit for bit, lse within fp32 rounding.
"""
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


def _shard_triples(x, bounds):
    n = x.shape[0]
    S = len(bounds) - 1
    tr = torch.empty((n, S, 3), dtype=torch.float32, device=x.device)
    for s in range(S):
        b0, b1 = int(bounds[s]), int(bounds[s + 1])
        m, l, a = pkg.greedy_lse(x[:, b0:b1].contiguous())
        tr[:, s, 0] = m
        tr[:, s, 1] = l
        tr[:, s, 2] = (a + b0).to(torch.int32).view(torch.float32)
    return tr


@pytest.mark.parametrize("S", [1, 2, 3, 4, 8])
def test_sharded_greedy_merges_to_the_unsharded_pass(S):
    dev = _dev()
    g = wl.make_greedy_inputs("shard", n=48, V=248320, sigma=4.0, seed=11 + S, tie_fraction=0.25)
    x = g.logits.to(dev)
    fm, fl, fa = pkg.greedy_lse(x)
    rng = np.random.Generator(np.random.PCG64(S))
    cuts = np.sort(rng.choice(np.arange(1, g.V), size=S - 1, replace=False)) if S > 1 else np.zeros(0, np.int64)
    bounds = np.concatenate([[0], cuts, [g.V]])
    mm, ml, ma = pkg.merge_triples(_shard_triples(x, bounds))
    torch.cuda.synchronize()
    assert torch.equal(mm, fm)
    assert torch.equal(ma, fa)
    assert torch.allclose(ml, fl, rtol=0, atol=5e-5)
    ref = oracle.greedy_rows(wl.bf16_bits(g.logits), g.n, g.V)
    assert np.array_equal(ma.cpu().numpy(), ref["argmax"])
    assert np.abs(ml.cpu().numpy().astype(np.float64) - ref["lse"]).max() <= 1e-4
    # planted ties: the smallest planted id wins even when the tied ids sit in different shards
    for r, ids in zip(g.planted_rows, g.planted_ids):
        assert int(ma[r]) == int(ids.min())


def test_merge_against_the_oracle_merge_with_empty_shards():
    dev = _dev()
    V = 4097
    g = wl.make_greedy_inputs("shard_inf", n=16, V=V, sigma=3.0, seed=5, tie_fraction=0.0)
    bits = wl.bf16_bits(g.logits).reshape(g.n, V).copy()
    bounds = np.array([0, 1000, 1001, 2500, V])
    ninf = np.uint16(0xFF80)
    bits[3, 1000:2500] = ninf            # two shards of row 3 are all -inf
    bits[5, :] = ninf                    # row 5 is all -inf
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    tr = _shard_triples(x, bounds)
    mm, ml, ma = pkg.merge_triples(tr)
    trh = tr.cpu().numpy()
    for r in range(g.n):
        base = bounds[:-1].astype(np.int32)
        local = trh[r, :, 2].view(np.int32) - base
        om, ol, oa = oracle.merge_triples(trh[r, :, 0], trh[r, :, 1].astype(np.float64), local, base)
        assert float(mm[r]) == om or (np.isinf(om) and float(mm[r]) == om)
        assert int(ma[r]) == oa
        if np.isfinite(ol):
            assert abs(float(ml[r]) - ol) <= 1e-5 * max(1.0, abs(ol))
        else:
            assert float(ml[r]) == ol
    assert float(mm[5]) == -np.inf and float(ml[5]) == -np.inf


@pytest.mark.parametrize("V", [1, 7, 1025, 4097, 248320, 300000])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("offset", [0, 1])
def test_dense_log_softmax_matches_the_oracle(V, dtype, offset):
    """Rows up to about 262k logits are held on chip by a cluster (one read); V = 300000 takes the
    two-pass form (the triple pass, then the write pass)."""
    dev = _dev()
    n = 6 if V > 5000 else 9
    g = wl.make_greedy_inputs("lsm", n=n, V=V, sigma=3.0, seed=V % 97, tie_fraction=0.0)
    # offset 1: the rows start one element past a 16-byte boundary (element-wise path)
    buf = torch.empty(n * V + offset, dtype=torch.bfloat16)
    buf[offset:] = g.logits.reshape(-1)
    x = buf.to(dev)[offset:].view(n, V)
    out, mx, lse, am = pkg.log_softmax(x, dtype=dtype)
    gm, gl, ga = pkg.greedy_lse(x)
    torch.cuda.synchronize()
    # max and argmax are exact; lse is summed in another order than the greedy pass, so
    # the two agree to fp32 rounding (each is held to the oracle's double lse below)
    assert torch.equal(mx, gm) and torch.equal(am, ga)
    assert torch.allclose(lse, gl, rtol=1e-6, atol=1e-6)
    ref = oracle.greedy_rows(wl.bf16_bits(g.logits), n, V)
    xs = g.logits.float().numpy().astype(np.float64)
    want = xs - ref["lse"][:, None]
    got = out.float().cpu().numpy().astype(np.float64)
    if dtype == torch.float32:
        assert np.abs(got - want).max() <= 2e-4
    else:
        # bf16 output: within the lse tolerance plus one bf16 rounding
        assert (np.abs(got - want) <= 2e-4 + np.abs(want) * 2.0 ** -8).all()
    # probabilities sum to one
    p = np.exp(got).sum(axis=1)
    assert np.abs(p - 1.0).max() <= (1e-3 if dtype == torch.float32 else 3e-2)
