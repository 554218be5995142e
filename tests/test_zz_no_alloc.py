"""pkv_sample_batch_noalloc: the sampler with the library's static scratch.

This entry point serves callers that cannot allocate device memory where
they sample: a decode loop that must not stall on cudaMalloc (it can
synchronise the device), code inside a CUDA-graph stream capture, and
engines that gave their free memory to the KV pool.  The call uses the CUDA
runtime itself, so it is made from ordinary host code, not from a host
callback.  The source pages have no counterpart.  This file is collected
last so that a failure here comes after every other test has run; it also
passes alone in a fresh process.

CPU: the size limit and the argument checks answer before any CUDA call.
GPU: the tokens equal the oracle's (parity bar of tests/parity.py), equal
those of pkv_sample_batch with a caller workspace, and no device memory is
allocated by the call (the torch caching allocator's counters do not move).
"""

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_gb300 import pkv, workloads
from parity import check_sampler

DEV = "cuda"


def test_noalloc_rejects_batches_beyond_its_scratch():
    lib = pkv.load()
    p = ctypes.c_void_p(256)
    # B=1024, V=256000 bf16 needs about 320 MB of records and slice histograms;
    # the scratch holds 64 MiB.
    rc = lib.pkv_sample_batch_noalloc(p, pkv.PKV_BF16, 1024, 256000, 256000, None, None, None,
                                      None, p, None, 0, 0, None, None, None, None, None)
    assert rc == pkv.PKV_EUNSUPPORTED
    assert "static scratch" in pkv.last_error()


def test_noalloc_scratch_holds_the_benchmark_batches():
    # The mixed bf16 batch and the fp32 full-vocabulary nucleus batch (both
    # B=256, V=151936) fit the 64 MiB scratch; the large bf16 one does not.
    lib = pkv.load()
    assert lib.pkv_sample_workspace_bytes(256, 151936, pkv.PKV_BF16) <= 64 << 20
    assert lib.pkv_sample_workspace_bytes(256, 151936, pkv.PKV_FP32) <= 64 << 20
    assert lib.pkv_sample_workspace_bytes(1024, 256000, pkv.PKV_BF16) > 64 << 20


def test_noalloc_checks_arguments_first():
    lib = pkv.load()
    rc = lib.pkv_sample_batch_noalloc(None, pkv.PKV_BF16, 4, 100, 100, None, None, None, None,
                                      ctypes.c_void_p(256), None, 0, 0, None, None, None, None,
                                      None)
    assert rc == pkv.PKV_EINVAL and "logits" in pkv.last_error()
    p = ctypes.c_void_p(256)
    rc = lib.pkv_sample_batch_noalloc(p, pkv.PKV_BF16, 4, 100, 100, p, None, None, None, p, None,
                                      0, 0, None, None, None, None, None)
    assert rc == pkv.PKV_EINVAL and "uniform" in pkv.last_error()


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_workspace_path_without_allocating():
    w = workloads.mixed(B=96)
    L = w.logits.to(DEV)
    B, V = L.shape
    args = [None if x is None else x.to(DEV) for x in (w.temperature, w.top_k, w.top_p,
                                                       w.uniform)]
    out = torch.empty(B, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pool = torch.zeros(w.pool_shape, dtype=torch.int32, device=DEV)
    rows, cols = w.wb_rows.to(DEV), w.wb_cols.to(DEV)
    saved = torch.empty((3, B), dtype=torch.int32, device=DEV)  # each call's tokens
    # Warm up (library load, symbol lookup), then count allocations over calls.
    pkv.sample_batch_noalloc(L, *args, out_tokens=out, status=status)
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats(DEV).get("allocation.all.allocated", 0)
    for i in range(3):
        pkv.sample_batch_noalloc(L, *args, out_tokens=out, token_pool=pool, wb_rows=rows,
                                 wb_cols=cols, status=status)
        saved[i].copy_(out)
    torch.cuda.synchronize()
    after = torch.cuda.memory_stats(DEV).get("allocation.all.allocated", 0)
    assert after == before
    assert int(status.item()) == 0
    # Every call after the warm-up (three in a row) equals the workspace entry
    # point's tokens, and so the oracle's within the parity bar: the shared
    # scratch is left ready by each call.
    ref = pkv.sample_batch(L, *args).cpu().numpy()
    for i in range(3):
        tok = saved[i].cpu().numpy()
        np.testing.assert_array_equal(tok, ref)
        check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, tok)
    # The fused write-back went through as well.
    got = pool.cpu().numpy()
    r, c = w.wb_rows.numpy(), w.wb_cols.numpy()
    keep = c >= 0
    np.testing.assert_array_equal(got[r[keep], c[keep]], tok[keep])
