"""Seeded synthetic inputs for the sampling pass and the greedy pass.

This module only draws random inputs (torch CPU generators for the large normal
draws, numpy PCG64 for small choices; values rounded to bf16 by torch): it
holds none of the method's arithmetic. The tests feed the same
inputs to the CUDA library and to the CPU oracle, and the benchmark times the
library on them.

Shapes follow the pages' workloads: a diffusion canvas of C = 8 codebook rows,
about 100 positions per request and V = 1025 (1024 codes plus a mask token),
packed across requests along positions ("Add a sampler resource for discrete
diffusion", Contract; "Sampler support for discrete diffusion", Hert4's batch
table with target_len 100), and the V = 248320 vocabulary of the large-vocab
greedy case ("perf: avoid full-vocab all-gather for draft greedy sampling",
Design and invariants).
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch


def request_id_of(r: int) -> int:
    """Request ids are distinct and differ from the request index."""
    return 1000 + 7919 * r


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """Round fp32 values to bf16 (round to nearest even) as a CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a CPU bf16 tensor (flattened)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)


@dataclass
class SampleInputs:
    name: str
    C: int
    V: int
    seq_lens: np.ndarray          # int32 [B]
    request_ids: np.ndarray       # int32 [B]
    guidance: np.ndarray          # float32 [B]
    temperature: np.ndarray       # float32 [B]
    top_ratio: float
    seed: int
    c_logits: torch.Tensor        # bf16 CPU [C, P, V]
    u_logits: Optional[torch.Tensor]  # bf16 CPU [C, P_u, V] or None
    iterations: List[int] = field(default_factory=lambda: [0])

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def P(self) -> int:
        return int(self.seq_lens.sum())

    @property
    def P_u(self) -> int:
        return int(self.seq_lens[self.guidance != 0].sum())

    @property
    def cells(self) -> int:
        return self.C * self.P

    def algorithmic_bytes(self) -> int:
        """Bytes one call must move: c, u for guided requests, 8 B of output per cell."""
        return 2 * self.V * self.C * self.P + 2 * self.V * self.C * self.P_u + 8 * self.C * self.P


def make_sample_inputs(name, C, seq_lens, V, guidance, temperature, sigma_c, sigma_u,
                       top_ratio, seed, iterations=(0,), gen_seed=None) -> SampleInputs:
    """c ~ N(0, sigma_c^2) rounded to bf16; u = bf16(float(c) + N(0, sigma_u^2)) for the
    requests with guidance != 0, packed in request order."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    guidance = np.asarray(guidance, dtype=np.float32)
    temperature = np.asarray(temperature, dtype=np.float32)
    B = int(seq_lens.shape[0])
    P = int(seq_lens.sum())
    gen = torch.Generator().manual_seed(int(seed if gen_seed is None else gen_seed))
    c32 = torch.randn((C, P, V), generator=gen, dtype=torch.float32)
    c32 *= float(np.float32(sigma_c))
    c = c32.to(torch.bfloat16)
    del c32
    guided = guidance != 0
    u = None
    if guided.any():
        if guided.all():
            cu = c.float()
        else:
            # Positions of guided requests, in request order.
            offs = np.concatenate([[0], np.cumsum(seq_lens)]).astype(np.int64)
            pos = np.concatenate([np.arange(offs[r], offs[r + 1]) for r in range(B) if guided[r]])
            cu = c[:, torch.from_numpy(pos)].float()
        noise = torch.randn(cu.shape, generator=gen, dtype=torch.float32)
        noise *= float(np.float32(sigma_u))
        cu += noise
        del noise
        u = cu.to(torch.bfloat16)
        del cu
    rids = np.array([request_id_of(r) for r in range(B)], dtype=np.int32)
    return SampleInputs(name=name, C=C, V=V, seq_lens=seq_lens, request_ids=rids,
                        guidance=guidance, temperature=temperature, top_ratio=float(top_ratio),
                        seed=int(seed), c_logits=c, u_logits=u, iterations=list(iterations))


def config1() -> SampleInputs:
    """Single request, C=8 rows x T=100 positions x V=1025; g=2, tau=0.9, ratio 0.1, seed 0."""
    return make_sample_inputs("cfg1: B=1 C=8 T=100 V=1025 g=2 tau=0.9", 8, [100], 1025,
                              [2.0], [0.9], 2.0, 1.0, 0.1, seed=0)


def config2() -> SampleInputs:
    """8 requests, C=8, ragged T ~ U{50..200}, V=1025, guidance from {0, 2} and temperature
    from {0, 0.9} per request (both kinds of each always present), ratio 0.1, seed 1."""
    rng = np.random.Generator(np.random.PCG64(1001))
    B = 8
    T = rng.integers(50, 201, size=B)
    g = rng.choice(np.array([0.0, 2.0], np.float32), size=B)
    tau = rng.choice(np.array([0.0, 0.9], np.float32), size=B)
    # Force a mix: at least one request of each guidance and each temperature.
    if (g == 0).all() or (g != 0).all():
        g[0], g[1] = 0.0, 2.0
    if (tau == 0).all() or (tau != 0).all():
        tau[2], tau[3] = 0.0, 0.9
    return make_sample_inputs("cfg2: B=8 C=8 T~U{50..200} V=1025 g in {0,2} tau in {0,0.9}", 8, T,
                              1025, g, tau, 2.0, 1.0, 0.1, seed=1)


def config3() -> SampleInputs:
    """64 requests, C=8, ragged T ~ U{100..400}, V=1025, sigma_c=3, sigma_u=1.5, g=2, tau=0.9,
    ratio 0.1, seed 2, iterations 0..31 on the same buffers."""
    rng = np.random.Generator(np.random.PCG64(1002))
    B = 64
    T = rng.integers(100, 401, size=B)
    return make_sample_inputs("cfg3: B=64 C=8 T~U{100..400} V=1025 g=2 tau=0.9", 8, T, 1025,
                              np.full(B, 2.0, np.float32), np.full(B, 0.9, np.float32), 3.0, 1.5,
                              0.1, seed=2, iterations=range(32))


def config5() -> SampleInputs:
    """64 requests x 16 positions (1024 cells, C=1), V=248320, sigma_c=4, sigma_u=2, g=1.5,
    tau=0.7, ratio 0.1 (k=24832), seed 3."""
    B = 64
    return make_sample_inputs("cfg5: B=64 T=16 C=1 V=248320 g=1.5 tau=0.7", 1, np.full(B, 16), 248320,
                              np.full(B, 1.5, np.float32), np.full(B, 0.7, np.float32), 4.0, 2.0,
                              0.1, seed=3)


@dataclass
class GreedyInputs:
    name: str
    n: int
    V: int
    logits: torch.Tensor            # bf16 CPU [n, V]
    planted_rows: np.ndarray        # rows whose maximum was planted at several ids
    planted_ids: List[np.ndarray]   # the planted ids of each planted row

    def algorithmic_bytes(self) -> int:
        return 2 * self.n * self.V + 12 * self.n


def make_greedy_inputs(name, n, V, sigma, seed, tie_fraction=0.25, tie_spread_row=True) -> GreedyInputs:
    """logits ~ N(0, sigma^2) in bf16; in a seeded quarter of the rows the next bf16 value above
    the row maximum is written at 2-4 seeded random ids, so the row's argmax is a planted tie
    (expect the smallest id). One planted row puts its ids far apart along the row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = torch.randn((n, V), generator=torch.Generator().manual_seed(int(seed)), dtype=torch.float32)
    x *= float(np.float32(sigma))
    t = x.to(torch.bfloat16)
    del x
    bits = t.view(torch.int16)
    n_planted = int(round(tie_fraction * n))
    rows = np.sort(rng.choice(n, size=n_planted, replace=False)) if n_planted else np.zeros(0, np.int64)
    planted_ids = []
    for j, r in enumerate(rows):
        cnt = min(int(rng.integers(2, 5)), V)
        if tie_spread_row and j == 0 and V >= 16 and cnt >= 2:
            ids = np.array([3, V // 2 + 1, V - 2][:cnt] if cnt <= 3 else [3, V // 3, (2 * V) // 3, V - 2])
        else:
            ids = np.sort(rng.choice(V, size=cnt, replace=False))
        rowmax = t[r].float().max()
        up = torch.tensor([float(rowmax)], dtype=torch.float32).to(torch.bfloat16)
        # next representable bf16 above the row max (the max is positive here)
        up_bits = int(up.view(torch.int16).item()) & 0xFFFF
        if float(rowmax) >= 0:
            up_bits += 1
        else:
            up_bits -= 1
        val = np.int16(np.uint16(up_bits).view(np.int16))
        bits[r, torch.from_numpy(np.asarray(ids, dtype=np.int64))] = int(val)
        planted_ids.append(np.asarray(ids, dtype=np.int64))
    return GreedyInputs(name=name, n=n, V=V, logits=t, planted_rows=np.asarray(rows, np.int64),
                        planted_ids=planted_ids)


def config4() -> GreedyInputs:
    """Greedy large vocab: 256 rows x V=248320, N(0, 4^2), planted maxima in 25% of rows."""
    return make_greedy_inputs("cfg4: greedy n=256 V=248320 sigma=4 ties in 25% of rows", 256, 248320,
                              4.0, seed=4)


SAMPLE_CONFIGS = {"cfg1": config1, "cfg2": config2, "cfg3": config3, "cfg5": config5}
