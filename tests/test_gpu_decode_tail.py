"""pkv_decode_tail: the sampler and the page fill of one decode step in one
call (the fill runs in extra CTAs of the sampler's finish kernel).  Its
tokens, token pool, page table, page total and status equal those of the two
separate calls, and the page table equals the oracle's, on every workload."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gb300 import pkv, workloads

DEV = "cuda"


def _d(x):
    return None if x is None else x.to(DEV)


def test_decode_tail_checks_fill_arguments_first():
    lib = pkv.load()
    p = ctypes.c_void_p(256)
    args = [p, pkv.PKV_BF16, 4, 1024, 1024, None, None, None, None, p, None, 0, 0, None, None,
            None, p, 1 << 24]
    # page_size 0, then a NULL length array: rejected before any launch.
    rc = lib.pkv_decode_tail(*args, p, p, p, 4, 0, p, 16, p, 4, 64, None, None)
    assert rc == pkv.PKV_EINVAL and "page_size" in pkv.last_error()
    rc = lib.pkv_decode_tail(*args, None, p, p, 4, 16, p, 16, p, 4, 64, None, None)
    assert rc == pkv.PKV_EINVAL and "NULL" in pkv.last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["pr1", "mixed", "nucleus", "large"])
def test_decode_tail_equals_the_two_calls(name):
    w = workloads.make(name)
    L = w.logits.to(DEV)
    B = L.shape[0]
    t, k, p, u = _d(w.temperature), _d(w.top_k), _d(w.top_p), _d(w.uniform)
    rows, cols = _d(w.wb_rows), _d(w.wb_cols)
    fill = (_d(w.cached_len), _d(w.device_len), _d(w.table_idx), w.page_size, _d(w.free_slots))

    def run(fused):
        pool = torch.full(w.pool_shape, -3, dtype=torch.int32, device=DEV)
        pt = torch.full(w.pt_shape, -7, dtype=torch.int32, device=DEV)
        total = torch.full((1,), -1, dtype=torch.int64, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = torch.empty(B, dtype=torch.int32, device=DEV)
        if fused:
            pkv.decode_tail(L, t, k, p, u, out, pool, rows, cols, *fill, pt, total, status)
        else:
            pkv.sample_batch(L, t, k, p, u, out_tokens=out, token_pool=pool, wb_rows=rows,
                             wb_cols=cols, status=status)
            pkv.fill_page_table(*fill, pt, total, status)
        torch.cuda.synchronize()
        return (out.cpu().numpy(), pool.cpu().numpy(), pt.cpu().numpy(), int(total.item()),
                int(status.item()))

    a, b = run(True), run(False)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    want = np.full(w.pt_shape, -7, np.int32)
    res = oracle.fill_page_table(w.cached_len, w.device_len, w.table_idx, w.page_size,
                                 w.free_slots, want)
    np.testing.assert_array_equal(a[2], want)
    assert a[3] == res["total"]
