"""GPU parity of the min_p filter (pkv_sample_batch_ex) against the CPU
oracle: tokens, and kept-set probabilities through the debug output."""

import numpy as np
import pytest
import torch

from paged_kv_gb300 import pkv, workloads

from parity import check_sampler

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _d(x):
    return None if x is None else x.to(DEV)


def _minp(B, seed, frac=0.5, lo=0.01, hi=0.5):
    g = torch.Generator().manual_seed(seed)
    v = lo + (hi - lo) * torch.rand(B, generator=g)
    on = torch.rand(B, generator=g) < frac
    return torch.where(on, v, torch.zeros(B))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_minp_mixed_rows_with_probs(dtype):
    w = workloads.mixed(B=48, V=20000)
    logits = w.logits.to(dtype)
    mp = _minp(w.B, 1)
    B, V = logits.shape
    probs = torch.empty((B, V), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = pkv.sample_batch(_d(logits), _d(w.temperature), _d(w.top_k), _d(w.top_p),
                           _d(w.uniform), probs_out=probs, status=status, min_p=_d(mp))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st = check_sampler(logits, w.temperature, w.top_k, w.top_p, w.uniform, tok.cpu().numpy(),
                       gpu_probs=probs.cpu().numpy(), min_p=mp)
    assert st["exact"] + st["excused_cdf"] >= 20


def test_minp_full_size_mixed_batch():
    w = workloads.mixed()
    mp = _minp(w.B, 2, frac=0.6, lo=0.001, hi=0.3)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = pkv.sample_batch(_d(w.logits), _d(w.temperature), _d(w.top_k), _d(w.top_p),
                           _d(w.uniform), status=status, min_p=_d(mp))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st = check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, tok.cpu().numpy(),
                       min_p=mp)
    assert st["exact"] >= 100


def test_minp_off_equals_the_plain_call_and_one_is_argmax():
    w = workloads.mixed(B=32, V=32768)
    args = (_d(w.logits), _d(w.temperature), _d(w.top_k), _d(w.top_p), _d(w.uniform))
    a = pkv.sample_batch(*args).cpu().numpy()
    b = pkv.sample_batch(*args, min_p=torch.zeros(w.B, device=DEV)).cpu().numpy()
    c = pkv.sample_batch(*args, min_p=torch.full((w.B,), -1.0, device=DEV)).cpu().numpy()
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)
    # min_p = 1 keeps the maxima only: the argmax, or a draw among tied maxima.
    ones = torch.full((w.B,), 1.0)
    one = pkv.sample_batch(*args, min_p=_d(ones)).cpu().numpy()
    check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, one, min_p=ones)
    lf = w.logits.float()
    assert (lf[torch.arange(w.B), torch.as_tensor(one, dtype=torch.long)] == lf.max(dim=1).values).all()


def test_minp_on_large_topk_histogram_rows():
    # top_k = 1024 then top_p = 0.95 (bf16 histogram rows with a top-k), plus min_p.
    w = workloads.large(B=24, V=65536)
    mp = _minp(w.B, 3, frac=0.7, lo=0.01, hi=0.6)
    B, V = w.logits.shape
    probs = torch.empty((B, V), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = pkv.sample_batch(_d(w.logits), _d(w.temperature), _d(w.top_k), _d(w.top_p),
                           _d(w.uniform), probs_out=probs, status=status, min_p=_d(mp))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st = check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, tok.cpu().numpy(),
                       gpu_probs=probs.cpu().numpy(), min_p=mp)
    assert st["exact"] + st["excused_cdf"] >= 12
