"""GPU parity of pkv_free_pages and pkv_check_free_list against the CPU
oracle, bit-exact, through the C ABI ("CacheManager: allocation, release and
admission control", sections "Freeing, and freeing lazily" and "The
integrity check")."""

import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gb300 import pkv, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = -7


def _allocated_table(rb, ps):
    """Page table after every request of the release batch took its pages from
    position 0 (oracle fill on the CPU); returns the table and the free list left."""
    B = len(rb["device_len"])
    pt = np.full(rb["pt_shape"], SENTINEL, np.int32)
    free = rb["free_slots"].numpy()
    out = oracle.fill_page_table(np.zeros(B, np.int32), rb["device_len"], rb["table_idx"], ps,
                                 free, pt)
    assert out["rc"] == 0
    return pt, free[out["total"]:].copy()


def _both_free(table_idx, begin, end, ps, pt, live, capacity):
    cap_cpu = np.full(capacity, SENTINEL, np.int32)
    cap_cpu[: len(live)] = live
    want = oracle.free_pages(table_idx, begin, end, ps, pt, cap_cpu, len(live))
    cap_gpu = torch.full((capacity,), SENTINEL, dtype=torch.int32, device=DEV)
    cap_gpu[: len(live)] = torch.as_tensor(live, dtype=torch.int32)
    total = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.free_pages(torch.as_tensor(table_idx, dtype=torch.int32).to(DEV),
                   torch.as_tensor(begin, dtype=torch.int32).to(DEV),
                   torch.as_tensor(end, dtype=torch.int32).to(DEV), ps,
                   torch.as_tensor(pt).to(DEV), cap_gpu, len(live), total, status)
    torch.cuda.synchronize()
    return want, cap_cpu, cap_gpu.cpu().numpy(), int(total.item()), int(status.item())


@pytest.mark.parametrize("B,ps,ragged", [(1, 1, False), (37, 4, True), (256, 16, True),
                                         (256, 16, False), (1000, 64, True), (4096, 1, True)])
def test_free_bit_exact(B, ps, ragged):
    num_pages = 4096 * 2600 // ps + 1024
    rb = workloads.release_batch(B, ps, num_pages, seed=B * 131 + ps, ragged=ragged)
    pt, live = _allocated_table(rb, ps)
    want, cap_cpu, cap_gpu, total, status = _both_free(
        rb["table_idx"], rb["begin"], rb["end"], ps, pt, live, num_pages)
    assert want["rc"] == 0
    assert status == want["status"] and total == want["total"]
    np.testing.assert_array_equal(cap_gpu, cap_cpu)
    if not ragged:
        # Whole rows freed: every page is back, so the list passes the check.
        assert len(live) + total == num_pages
        assert oracle.check_free_list(cap_cpu, ps, num_pages, 0) == 0


def test_free_unaligned_slices_and_errors():
    rng = np.random.default_rng(5)
    pt = rng.integers(0, 10 ** 6, size=(9, 100)).astype(np.int32)
    table_idx = np.array([0, 9, 3, 4, 5, 6, -1, 8], np.int32)   # 9 and -1: rows out of range
    begin = np.array([3, 0, 7, 50, -2, 99, 0, 0], np.int32)     # -2: column out of range
    end = np.array([40, 5, 7, 101, 9, 100, 3, 100], np.int32)   # 101: past the table
    want, cap_cpu, cap_gpu, total, status = _both_free(table_idx, begin, end, 3, pt,
                                                       np.arange(5, dtype=np.int32), 200)
    assert want["status"] == pkv.ST_ROW_OOB | pkv.ST_COL_OOB
    assert status == want["status"] and total == want["total"]
    np.testing.assert_array_equal(cap_gpu, cap_cpu)


def test_free_capacity_overflow_writes_nothing():
    pt = np.arange(4 * 64, dtype=np.int32).reshape(4, 64)
    live = np.arange(10, dtype=np.int32)
    # 3 requests x 16 entries = 48 > 50 - 10 free places.
    want, cap_cpu, cap_gpu, total, status = _both_free([0, 1, 2], [0, 0, 0], [64, 64, 64], 4, pt,
                                                       live, 50)
    assert want["rc"] == -2 and want["status"] == pkv.ST_NOSPC
    assert status == pkv.ST_NOSPC and total == 0
    np.testing.assert_array_equal(cap_gpu, cap_cpu)
    assert (cap_gpu[10:] == SENTINEL).all()


def test_free_empty_batch():
    total = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    free = torch.zeros(4, dtype=torch.int32, device=DEV)
    pt = torch.zeros((1, 4), dtype=torch.int32, device=DEV)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    pkv.free_pages(e, e, e, 4, pt, free, 2, total)
    torch.cuda.synchronize()
    assert int(total.item()) == 0


def _gpu_check(free, ps, num_pages, cache_pages):
    bitmap = torch.full((max(1, math.ceil(num_pages / 32)),), -1, dtype=torch.int32, device=DEV)
    result = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    f = torch.as_tensor(np.asarray(free, np.int32)).to(DEV)
    pkv.check_free_list(f, len(free), ps, num_pages, cache_pages, bitmap, result)
    torch.cuda.synchronize()
    return int(result.item())


@pytest.mark.parametrize("ps,num_pages", [(1, 8), (4, 1000), (16, 65536), (64, 200000)])
def test_integrity_bits_match_oracle(ps, num_pages):
    rng = np.random.default_rng(num_pages + ps)
    full = (rng.permutation(num_pages) * ps).astype(np.int32)
    cases = {"full": (full, 0), "cache_holds_some": (full[: num_pages // 3], num_pages - num_pages // 3),
             "leak": (full[3:], 0)}
    dup = full.copy()
    dup[-1] = dup[0]
    cases["duplicate"] = (dup, 0)
    bad = full.copy()
    bad[num_pages // 2] = num_pages * ps  # one past the pool
    cases["range"] = (bad, 0)
    if ps > 1:
        mis = full.copy()
        mis[1] += 1
        cases["align"] = (mis, 0)
    neg = full.copy()
    neg[0] = -ps
    cases["negative"] = (neg, 0)
    for name, (lst, cache) in cases.items():
        want = oracle.check_free_list(lst, ps, num_pages, cache)
        assert _gpu_check(lst, ps, num_pages, cache) == want, name
    assert oracle.check_free_list(full, ps, num_pages, 0) == 0


def test_free_then_check_round_trip_mixed():
    # The benchmark's decode batch releases every request: all pages come back.
    w = workloads.mixed(B=256, V=64)
    ps = w.page_size
    num_pages = len(w.free_slots)
    rb = {"device_len": w.device_len, "table_idx": w.table_idx, "free_slots": w.free_slots,
          "pt_shape": w.pt_shape}
    pt, live = _allocated_table(rb, ps)
    zeros = np.zeros(256, np.int32)
    want, cap_cpu, cap_gpu, total, status = _both_free(w.table_idx, zeros, w.device_len, ps, pt,
                                                       live, num_pages)
    np.testing.assert_array_equal(cap_gpu, cap_cpu)
    assert status == 0 and total == want["total"] and len(live) + total == num_pages
    assert _gpu_check(cap_gpu, ps, num_pages, 0) == 0
