"""GPU parity of fp32 top-p rows (the candidate-list path) against the CPU
oracle over a sweep of logit shapes, temperatures, p, min_p and V: the cut
falls in dense and in sparse value buckets, near the lists' bound and far
above it, and rows the path cannot settle go to the exact fallback."""

import numpy as np
import pytest
import torch

from paged_kv_gb300 import pkv

from parity import check_sampler

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _logits(shape: str, B: int, V: int, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    if shape == "zipf":
        base = -1.1 * torch.log(torch.arange(1, V + 1, dtype=torch.float64)).to(torch.float32)
        x = torch.empty(B, V)
        for b in range(B):
            x[b, torch.randperm(V, generator=g)] = base + 0.5 * torch.randn(V, generator=g)
        return x
    if shape == "gauss1":
        return torch.randn(B, V, generator=g)
    if shape == "gauss5":
        return 5.0 * torch.randn(B, V, generator=g)
    if shape == "flat":  # nearly uniform: large kept sets
        return 0.01 * torch.randn(B, V, generator=g)
    if shape == "spiky":  # a few large logits over a flat floor
        x = 0.1 * torch.randn(B, V, generator=g)
        for b in range(B):
            idx = torch.randint(0, V, (8,), generator=g)
            x[b, idx] += 10.0 * torch.rand(8, generator=g)
        return x
    raise ValueError(shape)


@pytest.mark.parametrize("shape", ["zipf", "gauss1", "gauss5", "flat", "spiky"])
@pytest.mark.parametrize("V", [1000, 32000, 151936])
def test_fp32_topp_sweep(shape, V):
    B = 24
    seed = 7 * sum(map(ord, shape)) + V  # fixed across processes
    logits = _logits(shape, B, V, seed)
    g = torch.Generator().manual_seed(seed + 1)
    t = torch.tensor([0.3, 0.7, 1.0, 2.0])[torch.randint(0, 4, (B,), generator=g)]
    p = torch.tensor([0.5, 0.9, 0.99, 0.999])[torch.randint(0, 4, (B,), generator=g)]
    mp = torch.where(torch.rand(B, generator=g) < 0.25, 0.02 + 0.2 * torch.rand(B, generator=g),
                     torch.zeros(B))
    u = torch.rand(B, generator=g)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    probs = torch.empty((B, V), dtype=torch.float32, device=DEV)
    tok = pkv.sample_batch(logits.to(DEV), t.to(DEV), None, p.to(DEV), u.to(DEV),
                           probs_out=probs, status=status, min_p=mp.to(DEV))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    stats = check_sampler(logits, t, None, p, u, tok.cpu().numpy(), gpu_probs=probs.cpu().numpy(),
                          min_p=mp)
    assert stats["greedy"] + stats["exact"] + stats["validated"] == B, stats


def test_fp32_topp_near_zero_spread():
    # About one element in 40 takes a value in [0, 1e-38] over a floor of
    # -10: most threads' maxima are such values, so the lists' bound lies
    # among them and the span up to the row maximum is far too small for a
    # finite bucket scale.  Small p puts the cut among the listed entries,
    # and equal weights make it a count in (value desc, index asc) order.
    B, V = 4, 20480
    g = torch.Generator().manual_seed(77)
    logits = torch.full((B, V), -10.0)
    hot = torch.rand(B, V, generator=g) < 1.0 / 40.0
    logits[hot] = 1e-38 * torch.rand(int(hot.sum()), generator=g)
    t = torch.ones(B)
    p = torch.tensor([0.05, 0.1, 0.03, 0.08])
    u = torch.rand(B, generator=g)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = pkv.sample_batch(logits.to(DEV), t.to(DEV), None, p.to(DEV), u.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    stats = check_sampler(logits, t, None, p, u, tok.cpu().numpy(), None)
    assert stats["greedy"] + stats["exact"] + stats["validated"] == B, stats
