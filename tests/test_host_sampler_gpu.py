"""The pipelined end-to-end path (HostSampler): steps submitted back to back from pinned host
memory give the same (tokens, logprobs) as ds_sample on device copies of the same inputs."""
import numpy as np
import pytest
import torch

import vocab_wide_logit_gb300 as pkg
from vocab_wide_logit_gb300 import workloads as wl
from vocab_wide_logit_gb300.api import HostSampler

pytestmark = pytest.mark.gpu


def test_pipelined_steps_match_device_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.load()
    dev = torch.device("cuda:0")
    inp = wl.config2()
    hs = HostSampler(torch.from_numpy(inp.request_ids), torch.from_numpy(inp.seq_lens.astype(np.int32)),
                     torch.from_numpy(inp.guidance), torch.from_numpy(inp.temperature), inp.C, inp.P, inp.P_u,
                     inp.V, device=dev, depth=2)
    c_h = inp.c_logits.pin_memory()
    u_h = inp.u_logits.pin_memory()
    its = [0, 1, 2, 7, 3]
    slots, got = [], {}
    for n, it in enumerate(its):
        slots.append(hs.submit(c_h, u_h, inp.top_ratio, inp.seed, it))
        if n >= 1:  # read each step's result before its slot is reused
            tok, lp = hs.result(slots[n - 1])
            got[its[n - 1]] = (tok.clone(), lp.clone())
    tok, lp = hs.result(slots[-1])
    got[its[-1]] = (tok.clone(), lp.clone())
    rid = torch.from_numpy(inp.request_ids).to(dev)
    sl = torch.from_numpy(inp.seq_lens.astype(np.int32)).to(dev)
    g = torch.from_numpy(inp.guidance).to(dev)
    tau = torch.from_numpy(inp.temperature).to(dev)
    c, u = inp.c_logits.to(dev), inp.u_logits.to(dev)
    for it in its:
        t, l = pkg.sample(rid, c, u, sl, g, tau, inp.top_ratio, inp.seed, it)
        torch.cuda.synchronize()
        assert torch.equal(t.cpu(), got[it][0]), it
        assert torch.equal(l.cpu(), got[it][1]), it
    assert hs.h2d_bytes() == 2 * inp.V * inp.C * (inp.P + inp.P_u)
    assert hs.d2h_bytes() == 8 * inp.C * inp.P
