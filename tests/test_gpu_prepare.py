"""GPU parity of pkv_prepare_step (the step before the model: page fill,
packed positions, input_ids and out_loc gathers) against the CPU oracle,
bit-exact, through the C ABI; plus the hand-computed examples."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gb300 import pkv, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SENTINEL = -7


def _t(a, dtype=torch.int32):
    return torch.as_tensor(np.ascontiguousarray(a)).to(dtype).to(DEV)


def run_both(cached, device, table, ps, free, pt0, pool, cap):
    """The library and the oracle on the same inputs; returns both results."""
    pt = _t(pt0)
    pos = torch.full((cap,), SENTINEL, dtype=torch.int32, device=DEV)
    ids = torch.full((cap,), SENTINEL, dtype=torch.int32, device=DEV)
    loc = torch.full((cap,), SENTINEL, dtype=torch.int32, device=DEV)
    tp = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    tt = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.prepare_step(_t(cached), _t(device), _t(table), ps, _t(free), pt, _t(pool), cap,
                     positions=pos, input_ids=ids, out_loc=loc, total_pages=tp,
                     total_tokens=tt, status=status)
    torch.cuda.synchronize()
    got = {"pt": pt.cpu().numpy(), "positions": pos.cpu().numpy(), "input_ids": ids.cpu().numpy(),
           "out_loc": loc.cpu().numpy(), "total_pages": int(tp.item()),
           "total_tokens": int(tt.item()), "status": int(status.item())}
    want_pt = np.ascontiguousarray(pt0, dtype=np.int32).copy()
    want = oracle.prepare_step(cached, device, table, ps, free, want_pt, pool, cap)
    want["pt"] = want_pt
    return got, want


def assert_same(got, want):
    assert got["status"] == want["status"]
    assert got["total_tokens"] == want["total_tokens"]
    assert got["total_pages"] == want["total_pages"]
    np.testing.assert_array_equal(got["pt"], want["pt"])
    n = len(want["positions"])
    for k in ("positions", "input_ids", "out_loc"):
        np.testing.assert_array_equal(got[k][:n], want[k])
        assert (got[k][n:] == SENTINEL).all(), f"{k} written past the step's tokens"


def test_selftest_example():
    g = json.load(open(os.path.join(GOLDEN, "prepare_selftest.json")))
    pt = np.zeros(g["pt_shape"], np.int32)
    pt[1, :8] = g["pt_row1_prefix"]
    pool = np.zeros((2, 16), np.int32)
    pool[1] = g["pool_row1"]
    got, want = run_both(g["cached_len"], g["device_len"], g["table_idx"], g["page_size"],
                         g["free_slots"], pt, pool, 16)
    assert_same(got, want)
    assert got["out_loc"][:3].tolist() == g["expected_out_loc"]
    assert got["pt"][1].tolist() == g["expected_row1"]


def _state(cached, device, table, ps, rows, cols, pool_cols, seed):
    rng = np.random.default_rng(seed)
    pt = rng.integers(0, 1 << 24, (rows, cols)).astype(np.int32)
    pool = rng.integers(0, 1 << 17, (rows, pool_cols)).astype(np.int32)
    return pt, pool


@pytest.mark.parametrize("name", ["pr1", "mixed", "nucleus", "large"])
def test_workloads_match_oracle(name):
    w = workloads.make(name)
    cached, device = w.cached_len.numpy(), w.device_len.numpy()
    table, ps, free = w.table_idx.numpy(), w.page_size, w.free_slots.numpy()
    rows, cols = w.pt_shape
    pt, pool = _state(cached, device, table, ps, rows, cols, w.pool_shape[1], 11)
    ntok = int(np.maximum(device - cached, 0).sum())
    got, want = run_both(cached, device, table, ps, free, pt, pool, ntok + 37)
    assert want["rc"] == 0 and want["status"] == 0 and want["total_tokens"] == ntok
    assert_same(got, want)


def test_decode_step_one_token_each():
    # Decode: one token per request, a new page every ps steps.
    rng = np.random.default_rng(5)
    B, ps = 777, 16
    cached = rng.integers(0, 3000, B).astype(np.int32)
    device = cached + 1
    table = rng.permutation(B + 5)[:B].astype(np.int32)
    free = (rng.permutation(50000) * ps).astype(np.int32)
    pt, pool = _state(cached, device, table, ps, B + 5, 3008, 3008, 6)
    got, want = run_both(cached, device, table, ps, free, pt, pool, B)
    assert_same(got, want)
    np.testing.assert_array_equal(got["positions"], cached)


@pytest.mark.parametrize("ps", [1, 3, 4, 64])
def test_random_batches_with_empty_and_bad_requests(ps):
    rng = np.random.default_rng(ps)
    B = 180
    cached = rng.integers(0, 400, B).astype(np.int32)
    device = (cached + rng.integers(-5, 90, B)).astype(np.int32)  # some empty ranges
    # One table row per request, as in a real batch; -1 and 190..198 lie
    # outside the 190-row table and pool.
    table = (rng.permutation(200)[:B] - 1).astype(np.int32)
    cols = ((500 + ps) // ps + 1) * ps
    free = (rng.permutation(40000) * ps).astype(np.int32)
    pt, pool = _state(cached, device, table, ps, 190, cols, 450, 7)  # pool narrower than some ranges
    ntok = int(np.maximum(device - cached, 0).sum())
    got, want = run_both(cached, device, table, ps, free, pt, pool, ntok)
    assert want["rc"] == 0 and want["status"] & 4 and want["status"] & 8
    assert_same(got, want)


def test_capacity_and_no_space_write_nothing():
    g = json.load(open(os.path.join(GOLDEN, "prepare_batch4.json")))
    pt = np.full(g["pt_shape"], 9, np.int32)
    pool = np.arange(64, dtype=np.int32).reshape(g["pool_shape"])
    free = np.arange(64, dtype=np.int32) * 4
    args = (g["cached_len"], g["device_len"], g["table_idx"], 4)
    got, want = run_both(*args, free, pt, pool, 11)  # 12 tokens > 11
    assert got["status"] == 128 and got["total_tokens"] == 12 and got["total_pages"] == 0
    np.testing.assert_array_equal(got["pt"], pt)
    assert (got["positions"] == SENTINEL).all()
    assert want["rc"] == -3 and want["status"] == 128
    got, want = run_both(*args, free[:3], pt, pool, 64)  # 4 pages needed, 3 free
    assert got["status"] == 32 and got["total_pages"] == 0
    np.testing.assert_array_equal(got["pt"], pt)
    assert (got["positions"] == SENTINEL).all()
    assert want["rc"] == -2 and want["status"] == 32


def test_empty_batch_writes_zero_totals():
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    pt = torch.zeros((2, 8), dtype=torch.int32, device=DEV)
    pool = torch.zeros((2, 8), dtype=torch.int32, device=DEV)
    tp = torch.full((1,), 5, dtype=torch.int64, device=DEV)
    tt = torch.full((1,), 5, dtype=torch.int64, device=DEV)
    pkv.prepare_step(e, e, e, 4, torch.arange(4, dtype=torch.int32, device=DEV), pt, pool, 0,
                     total_pages=tp, total_tokens=tt)
    torch.cuda.synchronize()
    assert int(tp.item()) == 0 and int(tt.item()) == 0 and not pt.any()
