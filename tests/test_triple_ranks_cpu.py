"""The vocabulary-sharded greedy exchange on CPU ranks ("perf: avoid full-vocab
all-gather for draft greedy sampling", Design and invariants): four gloo ranks
each own a slice of the vocabulary, reduce it with the oracle to (max, lse,
argmax), send exactly three FP32 words per token -- the global argmax's integer
bits carried in the third word -- with one all-gather, and merge. Every rank must
end with the unsharded result: max and argmax bit for bit, lse to double
rounding of fp32 shard values.
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N_ROWS, V = 12, 5003


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    sys.path.insert(0, ROOT)
    from vocab_wide_logit_gb300 import workloads as wl
    g = wl.make_greedy_inputs("ranks", n=N_ROWS, V=V, sigma=3.0, seed=21, tie_fraction=0.5)
    bits = wl.bf16_bits(g.logits).reshape(N_ROWS, V).copy()
    bits[2, 1000:4000] = 0xFF80  # a whole shard of row 2 is -inf
    return bits, g


def _worker(rank, world, port, bounds, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bits, _ = _inputs()
        b0, b1 = int(bounds[rank]), int(bounds[rank + 1])
        shard = np.ascontiguousarray(bits[:, b0:b1])
        loc = oracle.greedy_rows(shard, N_ROWS, b1 - b0)
        # the wire format: three fp32 words per token, the id's bits in the third
        words = np.empty((N_ROWS, 3), np.float32)
        words[:, 0] = loc["max"]
        words[:, 1] = loc["lse"].astype(np.float32)
        words[:, 2] = (loc["argmax"] + b0).astype(np.int32).view(np.float32)
        mine = torch.from_numpy(words)
        got = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)
        allw = torch.stack(got, dim=1).numpy()  # [rows, ranks, 3]
        merged = []
        for r in range(N_ROWS):
            ids = allw[r, :, 2].view(np.int32)
            m, l, a = oracle.merge_triples(allw[r, :, 0], allw[r, :, 1].astype(np.float64), ids,
                                           np.zeros(world, np.int32))
            merged.append((m, l, a))
        q.put((rank, merged))
    finally:
        dist.destroy_process_group()


def test_four_ranks_merge_to_the_unsharded_triple():
    sys.path.insert(0, ROOT)
    import oracle
    bounds = np.array([0, 1000, 4000, 4001, V])
    world = len(bounds) - 1
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, bounds, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    bits, g = _inputs()
    full = oracle.greedy_rows(bits, N_ROWS, V)
    for rank in range(world):
        for r, (m, l, a) in enumerate(res[rank]):
            assert m == float(full["max"][r])
            assert a == int(full["argmax"][r])
            assert abs(l - float(full["lse"][r])) <= 1e-6 * max(1.0, abs(float(full["lse"][r])))
    for r, ids in zip(g.planted_rows, g.planted_ids):
        assert res[0][r][2] == int(ids.min())
