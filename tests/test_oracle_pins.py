"""Pins for the CPU oracle: it is checked against what the pages and the
mathematics fix, never against itself.

* worked examples printed on the pages (tests/golden/*.json, each cited);
* closed forms (softmax of two tokens, temperature scaling);
* special cases that reduce to a library routine (greedy == numpy.argmax,
  top_k=1 / top_p=1e-6 / tiny temperature == argmax);
* invariants (sum q == 1, q proportional to exp(l/T) on the kept set, the
  draw's measure equals q);
* an independent O(V^2) brute force for V <= 16 (tests/brute_force.py).

Each case is chosen so that a plausible slip in the oracle (top-p on the
inclusive instead of the exclusive cumulative sum, no renormalisation after
top-k, the draw in sorted instead of vocab order, multiplying by T instead of
dividing, a wrong tie rule) fails at least one test.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import brute_force
import oracle
from paged_kv_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _row(values, dtype=torch.float32):
    return torch.tensor([values], dtype=dtype)


def _sample1(values, T, k=-1, p=1.0, u=0.5, dtype=torch.float32, probs=True):
    res = oracle.sample(_row(values, dtype), torch.tensor([T]), torch.tensor([k], dtype=torch.int32),
                        torch.tensor([p]), torch.tensor([u]), want_probs=probs)
    return res


# ---------------------------------------------------------------- golden: sampler


def test_page_sampler_example_topk2():
    g = _golden("sampler_filters.json")
    row = g["rows"][0]
    q0 = 1.0 / (1.0 + math.exp(-1.0))  # e^5 / (e^5 + e^4)
    assert abs(q0 - row["q0_printed"]) < row["q0_printed_tol"]
    res = _sample1(g["logits"], row["temperature"], row["top_k"], row["top_p"], 0.5)
    q = res["probs"][0]
    assert abs(q[0] - q0) < 1e-12
    assert abs(q[1] - (1 - q0)) < 1e-12
    assert set(np.nonzero(q)[0].tolist()) == set(row["support"])
    # Inverse CDF in vocab order: u < q0 draws token 0, otherwise token 1.
    for u, want in [(0.0, 0), (q0 - 1e-6, 0), (q0 + 1e-6, 1), (0.999999, 1)]:
        assert _sample1(g["logits"], 1.0, 2, 1.0, u, probs=False)["tokens"][0] == want


def test_page_sampler_example_topp05_and_greedy():
    g = _golden("sampler_filters.json")
    logits = torch.tensor([g["logits"]] * 3, dtype=torch.float32)
    t = torch.tensor([r["temperature"] for r in g["rows"]])
    k = torch.tensor([r["top_k"] for r in g["rows"]], dtype=torch.int32)
    p = torch.tensor([r["top_p"] for r in g["rows"]])
    for u in np.linspace(0.0, 0.999, 41):
        res = oracle.sample(logits, t, k, p, torch.full((3,), float(u)), want_probs=True)
        assert res["tokens"][0] in g["rows"][0]["support"]
        assert res["tokens"][1] == 0 and res["kept"][1] == 1
        assert res["tokens"][2] == 0
    # The page says the top probability is "about 0.67"; exactly it is
    # e^5 / (e^5 + e^4 + e^3 + 3), which is > 0.5, so top-p keeps only token 0.
    q_top = math.exp(5) / (math.exp(5) + math.exp(4) + math.exp(3) + 3)
    assert 0.6 < q_top < 0.7


def test_all_greedy_batch_matches_numpy_argmax():
    logits = workloads.random_rows(16, 1000, torch.float32, seed=1, discrete=True)
    res = oracle.sample(logits)
    np.testing.assert_array_equal(res["tokens"], np.argmax(logits.numpy(), axis=1))
    bf = workloads.random_rows(16, 777, torch.bfloat16, seed=2)
    res = oracle.sample(bf)
    np.testing.assert_array_equal(res["tokens"], np.argmax(bf.float().numpy(), axis=1))


def test_greedy_signed_zero_ties_and_nan():
    # -0 and +0 are equal values: the lowest index wins.
    res = oracle.sample(torch.tensor([[-1.0, -0.0, 0.0, -2.0]]))
    assert res["tokens"][0] == 1
    res = oracle.sample(torch.tensor([[1.0, float("nan"), 2.0]]))
    assert res["tokens"][0] == -1 and res["row_status"][0] & 1


# ---------------------------------------------------------------- closed forms


def test_temperature_divides_logits():
    # Two tokens: q0 = 1 / (1 + exp(-(l0 - l1) / T)).
    for T in (0.25, 0.5, 2.0):
        q = _sample1([2.0, 0.0], T)["probs"][0]
        assert abs(q[0] - 1.0 / (1.0 + math.exp(-2.0 / T))) < 1e-12


def test_topp_renormalises_after_topk():
    # [5,4,3,0,0,0], k=2: renormalised q0 = 0.731 >= 0.7, so top_p=0.7 keeps only
    # token 0.  Without renormalisation q0 would be 0.656 < 0.7 and token 1 kept.
    res = _sample1([5.0, 4.0, 3.0, 0.0, 0.0, 0.0], 1.0, 2, 0.7)
    assert res["kept"][0] == 1 and res["probs"][0][0] == 1.0


def test_topp_uses_mass_before_token():
    # Exclusive cumulative sum: the top token is always kept even when its own
    # probability exceeds p.
    res = _sample1([10.0, 0.0, 0.0], 1.0, -1, 0.01)
    assert res["kept"][0] == 1
    # p just above the top token's probability keeps exactly two tokens.
    q0 = math.exp(10) / (math.exp(10) + 2)
    res = _sample1([10.0, 0.0, 0.0], 1.0, -1, q0 + 1e-6)
    assert res["kept"][0] == 2
    res = _sample1([10.0, 0.0, 0.0], 1.0, -1, q0 - 1e-6)
    assert res["kept"][0] == 1


def test_draw_walks_vocab_order():
    # The maximum sits at index 1; a small u must land on token 0, whose
    # interval comes first in vocab order.
    q0 = 1.0 / (1.0 + math.exp(5) + math.exp(4))
    assert _sample1([0.0, 5.0, 4.0], 1.0, -1, 1.0, q0 * 0.5)["tokens"][0] == 0
    assert _sample1([0.0, 5.0, 4.0], 1.0, -1, 1.0, q0 * 1.5)["tokens"][0] == 1
    assert _sample1([0.0, 5.0, 4.0], 1.0, -1, 1.0, 0.99)["tokens"][0] == 2


def test_topk_ties_take_lowest_index():
    # Values 3 at indices 4, 1, 6 (ties); k=2 keeps the two lowest indices.
    res = _sample1([0.0, 3.0, 0.0, 0.0, 3.0, 1.0, 3.0], 1.0, 2, 1.0)
    assert set(np.nonzero(res["probs"][0])[0].tolist()) == {1, 4}


# ---------------------------------------------------------------- reductions to argmax


@pytest.mark.parametrize("seed", [3, 4])
def test_degenerate_settings_reduce_to_argmax(seed):
    logits = workloads.random_rows(8, 300, torch.float32, seed=seed)
    want = np.argmax(logits.numpy(), axis=1)
    B = logits.shape[0]
    us = torch.linspace(0.0, 0.999, B)
    ones = torch.ones(B)
    res = oracle.sample(logits, ones, torch.ones(B, dtype=torch.int32), None, us)
    np.testing.assert_array_equal(res["tokens"], want)  # top_k = 1
    res = oracle.sample(logits, ones, None, torch.full((B,), 1e-6), us)
    np.testing.assert_array_equal(res["tokens"], want)  # top_p = 1e-6
    res = oracle.sample(logits, torch.full((B,), 1e-7), None, None, us)
    np.testing.assert_array_equal(res["tokens"], want)  # T clamps to 1e-6


# ---------------------------------------------------------------- invariants


def test_probabilities_sum_to_one_and_follow_softmax():
    logits = workloads.random_rows(12, 2000, torch.bfloat16, seed=5)
    t, k, p, u = workloads.random_params(12, seed=6, greedy_frac=0.0)
    res = oracle.sample(logits, t, k, p, u, want_probs=True)
    lf = logits.double().numpy()
    for b in range(12):
        q = res["probs"][b]
        assert abs(q.sum() - 1.0) < 1e-12
        s = np.nonzero(q)[0]
        assert len(s) == res["kept"][b]
        # Ratio test: q_i / q_j == exp((l_i - l_j) / T) on the kept set.
        i0 = s[np.argmax(lf[b, s])]
        ratio = q[s] / q[i0]
        want = np.exp((lf[b, s] - lf[b, i0]) / float(t[b]))
        np.testing.assert_allclose(ratio, want, rtol=1e-12)
        # The kept set is a prefix of the (logit desc, index asc) order.
        order = sorted(range(lf.shape[1]), key=lambda i: (-lf[b, i], i))
        assert set(order[:len(s)]) == set(s.tolist())


def test_draw_measure_equals_probability():
    rng = np.random.default_rng(7)
    for trial in range(20):
        V = int(rng.integers(2, 12))
        l = rng.integers(-3, 4, V).astype(np.float32).tolist()
        T, k, p = 0.7, int(rng.integers(0, V + 2)), float(rng.choice([1.0, 0.6, 0.9]))
        q = _sample1(l, T, k, p)["probs"][0]
        cuts = np.cumsum([q[i] for i in range(V)])
        points = sorted({0.0} | {min(max(c + d, 0.0), 1 - 1e-12)
                                  for c in cuts for d in (-1e-9, 1e-9)})
        measure = np.zeros(V)
        for a, bnd in zip(points[:-1], points[1:]):
            tok = _sample1(l, T, k, p, (a + bnd) / 2, probs=False)["tokens"][0]
            measure[tok] += bnd - a
        measure[_sample1(l, T, k, p, points[-1], probs=False)["tokens"][0]] += 1 - points[-1]
        np.testing.assert_allclose(measure, q, atol=1e-8)


# ---------------------------------------------------------------- brute force


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny_vocab(seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(40):
        V = int(rng.integers(1, 17))
        if rng.random() < 0.5:
            l = rng.integers(-3, 4, V).astype(np.float64)
        else:
            l = rng.normal(0, 2, V)
        l = np.asarray(l, np.float32).astype(np.float64).tolist()
        T = float(np.float32(rng.choice([0.3, 0.7, 1.0, 1.8])))
        k = int(rng.choice([-1, 1, 2, 3, V - 1, V, V + 3]))
        p = float(np.float32(rng.choice([1.0, 0.95, 0.6, 0.3, 1e-6])))
        u = float(np.float32(rng.random()))
        res = _sample1(l, T, k, p, u)
        q_bf = brute_force.kept_probabilities(l, T, k, p)
        q = res["probs"][0]
        assert set(np.nonzero(q)[0].tolist()) == set(i for i in q_bf if q_bf[i] > 0)
        for i, qi in q_bf.items():
            assert abs(q[i] - qi) < 1e-12
        if res["cdf_margin"][0] > 1e-9 and res["topp_margin"][0] > 1e-9:
            assert res["tokens"][0] == brute_force.sample_row(l, T, k, p, u)


def test_row_status_bits():
    res = oracle.sample(torch.tensor([[float("-inf")] * 4, [1.0, float("inf"), 0.0, 0.0],
                                      [0.0, 1.0, 2.0, 3.0]]),
                        torch.tensor([1.0, 1.0, 1.0]), None, None,
                        torch.tensor([0.5, 0.5, 1.5]))
    assert res["tokens"][0] == -1 and res["row_status"][0] == 2
    assert res["tokens"][1] == -1 and res["row_status"][1] == 1
    assert res["row_status"][2] == 16 and res["tokens"][2] == 3  # u clamped below 1


# ---------------------------------------------------------------- write-back


def test_writeback_golden():
    g = _golden("writeback_tuple.json")
    pool = np.zeros(g["pool_shape"], np.int32)
    st = oracle.writeback(g["tokens"], g["rows"], g["cols"], pool)
    assert st == 0
    np.testing.assert_array_equal(pool, np.array(g["expected_pool"], np.int32))
    pool2 = np.zeros(g["pool_shape"], np.int32)
    st = oracle.writeback([1, 2], [3, 0], [0, 5], pool2)
    assert st == (4 | 8) and not pool2.any()


# ---------------------------------------------------------------- pages


def test_pages_selftest_example():
    g = _golden("pages_selftest.json")
    res = oracle.alloc_pages([g["cached_len"]], [g["device_len"]], g["page_size"], 100)
    assert res["first_page"][0] == g["expected_first_page"]
    assert res["num_pages"][0] == g["expected_num_pages"] and res["total"] == 1
    pt = np.full((1, 16), -1, np.int32)
    free = np.arange(10, dtype=np.int32) * 4 + 40
    out = oracle.fill_page_table([6], [9], [0], 4, free, pt)
    assert out["rc"] == 0 and out["total"] == 1
    assert (np.nonzero(pt[0] >= 0)[0].tolist()) == g["expected_positions"]
    assert pt[0, 8:12].tolist() == [40, 41, 42, 43]


def test_pages_allocate_sequence():
    g = _golden("pages_allocate_sequence.json")
    ps, n = g["page_size"], g["num_pages"]
    free = np.arange(n, dtype=np.int32) * ps
    pt = np.zeros((4, 32), np.int32)
    for step in g["steps"]:
        out = oracle.fill_page_table([step["cached_len"]], [step["device_len"]],
                                     [g["table_idx"]], ps, free, pt)
        assert out["rc"] == 0
        free = free[out["total"]:]
        assert len(free) == step["free_after"]
        if "row_prefix" in step:
            assert pt[g["table_idx"], :8].tolist() == step["row_prefix"]
        if "aligned_column" in step:
            assert pt[g["table_idx"], step["aligned_column"]] % ps == 0
            assert pt[g["table_idx"], 8:12].tolist() == [8, 9, 10, 11]


def test_pages_trace_page_size_one():
    g = _golden("pages_trace_ps1.json")
    free = np.arange(g["num_pages"], dtype=np.int32)
    lens = np.array(g["prompt_lens"], np.int32)
    pt = np.zeros((5, 64), np.int32)
    out = oracle.fill_page_table(np.zeros(4, np.int32), lens, np.arange(4), 1, free, pt)
    free = free[out["total"]:]
    assert len(free) == g["free_after_prefill"]
    for want in g["free_after_each_decode"]:
        out = oracle.fill_page_table(lens, lens + 1, np.arange(4), 1, free, pt)
        free = free[out["total"]:]
        lens = lens + 1
        assert len(free) == want


def test_pages_hand_example_and_invariants():
    # ps=4, cached {0,6,3,10}, device {5,9,4,13}: pages [0,2), [2,3), none, [3,4).
    w = workloads.pr1()
    res = oracle.alloc_pages(w.cached_len, w.device_len, 4, 64)
    assert res["num_pages"].tolist() == [2, 1, 0, 1] and res["total"] == 4
    assert res["offset"].tolist() == [0, 2, 3, 3]
    pt = np.full(w.pt_shape, -1, np.int32)
    out = oracle.fill_page_table(w.cached_len, w.device_len, w.table_idx, 4,
                                 w.free_slots, pt)
    assert out["rc"] == 0
    assert pt[0, :8].tolist() == list(range(8))
    assert pt[1, 8:12].tolist() == [8, 9, 10, 11]
    assert pt[3, 12:16].tolist() == [12, 13, 14, 15]
    assert (pt[2] == -1).all()
    assert (pt >= 0).sum() == 16


def test_pages_disjoint_aligned_and_enospc():
    w = workloads.mixed(B=32, V=64)
    free = w.free_slots.numpy()
    pt = np.full(w.pt_shape, -1, np.int32)
    out = oracle.fill_page_table(w.cached_len, w.device_len, w.table_idx, w.page_size,
                                 free, pt)
    N = out["total"]
    taken = pt[pt >= 0]
    assert len(taken) == N * w.page_size
    assert len(np.unique(taken)) == len(taken)  # no location handed out twice
    starts = taken[taken % w.page_size == 0]
    assert set(starts.tolist()) == set(free[:N].tolist())  # exactly the front of the list
    # Not enough pages: nothing is written.
    pt2 = np.full(w.pt_shape, -1, np.int32)
    out = oracle.fill_page_table(w.cached_len, w.device_len, w.table_idx, w.page_size,
                                 free[: N - 1], pt2)
    assert out["rc"] == -2 and (pt2 == -1).all()


# ---------------------------------------------------------------- golden + brute force: free path


def test_pages_free_roundtrip():
    g = _golden("pages_free_roundtrip.json")
    ps, n, t = g["page_size"], g["num_pages"], g["table_idx"]
    free = np.arange(n, dtype=np.int32) * ps
    pt = np.zeros((4, 32), np.int32)
    for c, d in g["alloc_steps"]:
        out = oracle.fill_page_table([c], [d], [t], ps, free, pt)
        assert out["rc"] == 0
        free = free[out["total"]:]
    cap = np.full(n, -1, np.int32)
    cap[: len(free)] = free
    out = oracle.free_pages([t], [g["free_begin"]], [g["free_end"]], ps, pt, cap, len(free))
    assert out["rc"] == 0 and out["status"] == 0 and out["total"] == 3
    assert cap.tolist() == g["expected_free_list"]
    assert oracle.check_free_list(cap, ps, n, 0) == g["expected_integrity_bits"]


def test_pages_integrity_detects_leak():
    g = _golden("pages_integrity_leak.json")
    n, ps = g["num_pages"], g["page_size"]
    free = np.arange(n, dtype=np.int32) * ps
    assert oracle.check_free_list(free, ps, n, 0) == g["expected_bits_fresh"]
    assert oracle.check_free_list(free[g["leaked"]:], ps, n, 0) == g["expected_bits_after_leak"]


def test_integrity_bits_by_hand():
    # 4 pages of 4 tokens: a full list in any order passes; each fault sets its bit.
    assert oracle.check_free_list([12, 0, 8, 4], 4, 4, 0) == 0
    assert oracle.check_free_list([12, 0], 4, 4, 2) == 0      # two pages held by the cache
    assert oracle.check_free_list([12, 0], 4, 4, 1) == 1      # one page missing
    assert oracle.check_free_list([12, 1, 8, 4], 4, 4, 0) == 2  # not a page start
    assert oracle.check_free_list([12, 16, 8, 4], 4, 4, 0) == 4  # past the pool
    assert oracle.check_free_list([12, 4, 8, 4], 4, 4, 0) == 8   # page 1 twice (page 0 lost)
    assert oracle.check_free_list([-4, 0, 8, 4], 4, 4, 0) == 4   # negative start
    assert oracle.check_free_list([3, 0, 1, 2], 1, 4, 0) == 0    # ps=1: every slot is a start


@pytest.mark.parametrize("seed", range(6))
def test_free_matches_the_pages_slicing(seed):
    # The pages' own expression, free_slots = cat([free_slots] + [row[b:e][::ps] ...]),
    # evaluated with numpy slicing on random tables, ragged and unaligned ranges.
    rng = np.random.default_rng(seed)
    ps = int(rng.choice([1, 2, 4, 16]))
    R, C, B = 6, 40, int(rng.integers(0, 9))
    pt = rng.integers(0, 1000, size=(R, C)).astype(np.int32)
    t = rng.integers(0, R, size=B).astype(np.int32)
    b = rng.integers(0, C, size=B).astype(np.int32)
    e = np.minimum(C, b + rng.integers(-3, 30, size=B)).astype(np.int32)
    base = rng.integers(0, 1000, size=int(rng.integers(0, 5))).astype(np.int32)
    want = np.concatenate([base] + [pt[t[i], b[i]:e[i]][::ps] for i in range(B)]).astype(np.int32)
    cap = np.full(len(want) + 3, -7, np.int32)
    cap[: len(base)] = base
    out = oracle.free_pages(t, b, e, ps, pt, cap, len(base))
    assert out["rc"] == 0 and out["status"] == 0 and out["total"] == len(want) - len(base)
    assert cap[: len(want)].tolist() == want.tolist()
    assert (cap[len(want):] == -7).all()


def test_free_errors_write_nothing_or_skip():
    pt = np.arange(24, dtype=np.int32).reshape(3, 8)
    cap = np.full(4, -1, np.int32)
    # Capacity: 2 + 3 entries do not fit in 4: nothing is appended.
    cap[:2] = [100, 101]
    out = oracle.free_pages([0], [0], [5], 2, pt, cap, 2)
    assert out["rc"] == -2 and out["status"] == 32 and out["total"] == 0
    assert cap.tolist() == [100, 101, -1, -1]
    # A row outside the table and a range past its end are flagged and skipped.
    out = oracle.free_pages([5, 1, 2], [0, 6, 0], [2, 9, 3], 2, pt, cap, 2)
    assert out["rc"] == 0 and out["status"] == 4 | 8 and out["total"] == 2
    assert cap.tolist() == [100, 101, 16, 18]


# ---------------------------------------------------------------- golden + second statement: the step before the model


def test_prepare_selftest_example():
    # The pages' self-test 4 numbers run through _prepare_batch by hand.
    g = _golden("prepare_selftest.json")
    pt = np.zeros(g["pt_shape"], np.int32)
    pt[1, :8] = g["pt_row1_prefix"]
    pool = np.zeros((2, 16), np.int32)
    pool[1] = g["pool_row1"]
    r = oracle.prepare_step(g["cached_len"], g["device_len"], g["table_idx"], g["page_size"],
                            g["free_slots"], pt, pool, 16)
    assert r["rc"] == 0 and r["status"] == 0
    assert r["positions"].tolist() == g["expected_positions"]
    assert r["input_ids"].tolist() == g["expected_input_ids"]
    assert r["out_loc"].tolist() == g["expected_out_loc"]
    assert pt[1].tolist() == g["expected_row1"]
    assert (r["total_pages"], r["total_tokens"]) == (g["expected_total_pages"],
                                                     g["expected_total_tokens"])


def _batch4_state(g):
    ps = g["page_size"]
    pt = np.zeros(g["pt_shape"], np.int32)
    for i, (c, t) in enumerate(zip(g["cached_len"], g["table_idx"])):
        first = -(-c // ps)
        pt[t, :first * ps] = 1000 * (t + 1) + np.arange(first * ps)
    pool = (100 * np.arange(g["pool_shape"][0])[:, None] + np.arange(g["pool_shape"][1])[None, :])
    free = np.arange(g["num_free_pages"], dtype=np.int32) * ps
    return pt, pool.astype(np.int32), free


def test_prepare_batch_hand_example():
    g = _golden("prepare_batch4.json")
    pt, pool, free = _batch4_state(g)
    r = oracle.prepare_step(g["cached_len"], g["device_len"], g["table_idx"], g["page_size"],
                            free, pt, pool, 64)
    assert r["rc"] == 0 and r["status"] == 0
    assert r["positions"].tolist() == g["expected_positions"]
    assert r["input_ids"].tolist() == g["expected_input_ids"]
    assert r["out_loc"].tolist() == g["expected_out_loc"]
    assert (r["total_pages"], r["total_tokens"]) == (g["expected_total_pages"],
                                                     g["expected_total_tokens"])


@pytest.mark.parametrize("seed", range(4))
def test_prepare_matches_the_offline_slices(seed):
    # The offline example on the same page builds the same three arrays from
    # slices: positions = cat(arange(cached, device)), the inputs =
    # cat(token row[cached:device]), out_loc = cat(page_table[row,
    # cached:device]).  The oracle gathers token by token through the input
    # tuple; the two statements must agree (page table taken after the fill).
    rng = np.random.default_rng(100 + seed)
    B, ps = 12, int(rng.choice([1, 4, 16]))
    cached = rng.integers(0, 60, B).astype(np.int32)
    device = (cached + rng.integers(0, 40, B)).astype(np.int32)
    tidx = rng.permutation(B + 3)[:B].astype(np.int32)
    cols = ((int(device.max()) + ps - 1) // ps) * ps
    pt = rng.integers(0, 1 << 20, (B + 3, cols)).astype(np.int32)
    pool = rng.integers(0, 1 << 17, (B + 3, cols + 5)).astype(np.int32)
    free = (rng.permutation(4096) * ps).astype(np.int32)
    pt_after = pt.copy()
    fill = oracle.fill_page_table(cached, device, tidx, ps, free, pt_after)
    assert fill["rc"] == 0
    r = oracle.prepare_step(cached, device, tidx, ps, free, pt, pool, 1 << 14)
    assert r["rc"] == 0 and r["status"] == 0
    np.testing.assert_array_equal(pt, pt_after)
    want_pos = np.concatenate([np.arange(c, d) for c, d in zip(cached, device)]).astype(np.int32)
    want_ids = np.concatenate([pool[t, c:d] for t, c, d in zip(tidx, cached, device)])
    want_loc = np.concatenate([pt_after[t, c:d] for t, c, d in zip(tidx, cached, device)])
    np.testing.assert_array_equal(r["positions"], want_pos)
    np.testing.assert_array_equal(r["input_ids"], want_ids)
    np.testing.assert_array_equal(r["out_loc"], want_loc)
    assert r["total_tokens"] == int((device - cached).sum())
    # Page-aligned free list: every position in a new page lands at the same
    # offset inside its page ("writes page-aligned token positions"), and the
    # new pages are the free list's first entries in batch order.
    first = np.concatenate([np.full(d - c, -(-c // ps)) for c, d in zip(cached, device)])
    new = r["positions"] // ps >= first
    assert ((r["out_loc"][new] - r["positions"][new]) % ps == 0).all()
    starts = r["out_loc"][new] - r["positions"][new] % ps
    assert list(dict.fromkeys(starts.tolist())) == free[:r["total_pages"]].tolist()


def test_prepare_errors_write_nothing_or_skip():
    g = _golden("prepare_batch4.json")
    pt, pool, free = _batch4_state(g)
    # Above the token capacity: nothing written, the count still reported.
    pt0 = pt.copy()
    r = oracle.prepare_step(g["cached_len"], g["device_len"], g["table_idx"], 4, free, pt, pool, 11)
    assert r["rc"] == -3 and r["status"] == 128 and r["total_tokens"] == 12
    np.testing.assert_array_equal(pt, pt0)
    # Not enough free pages: nothing written.
    r = oracle.prepare_step(g["cached_len"], g["device_len"], g["table_idx"], 4, free[:3], pt,
                            pool, 64)
    assert r["rc"] == -2 and r["status"] == 32 and r["total_pages"] == 0
    np.testing.assert_array_equal(pt, pt0)
    # A request in a row outside the pool keeps its positions, gathers -1.
    small_pool = pool[:3].copy()
    r = oracle.prepare_step(g["cached_len"], g["device_len"], g["table_idx"], 4, free, pt,
                            small_pool, 64)
    assert r["rc"] == 0 and r["status"] == 4
    assert r["positions"].tolist() == g["expected_positions"]
    assert r["input_ids"].tolist()[-3:] == [-1, -1, -1]
    assert r["out_loc"].tolist()[-3:] == [-1, -1, -1]
    assert r["out_loc"].tolist()[:-3] == g["expected_out_loc"][:-3]



# ---------------------------------------------------------------- library routine: the counter-based uniforms


def _numpy_block(counter, key):
    # numpy's Philox advances its counter before producing a block, so the
    # block of counter c comes out of a generator whose counter is c - 1.
    c = [int(x) for x in counter]
    i = 0
    while c[i] == 0:
        c[i] = (1 << 64) - 1
        i += 1
    c[i] -= 1
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=np.array(c, dtype=np.uint64))
    return bg.random_raw(4).astype(np.uint64)


@pytest.mark.parametrize("counter,key", [
    ((1, 0, 0, 0), (0, 0)),
    ((5, 42, 0, 0), (42, 0)),
    ((0, 3, 0, 0), (7, 9)),                      # a borrow into the second word
    ((2**64 - 1, 2**64 - 1, 5, 1), (2**64 - 1, 2**64 - 1)),
    ((123456789, 987654321, 2**40, 2**63), (0xDEADBEEF, 0xC0FFEE)),
])
def test_philox_block_matches_numpy(counter, key):
    np.testing.assert_array_equal(oracle.philox4x64(counter, key), _numpy_block(counter, key))


def test_uniforms_are_the_top_24_bits_of_word_0():
    seed, offset, B = 42, 17, 300
    u = oracle.uniforms(seed, offset, B)
    assert u.dtype == np.float32 and ((u >= 0) & (u < 1)).all()
    for b in (0, 1, 2, 299):
        x0 = int(_numpy_block((b, offset, 0, 0), (seed, 0))[0])
        assert u[b] == np.float32((x0 >> 40) / 2**24)
    # Closed form of the conversion at its ends: 24-bit values k map to k / 2^24.
    k = (u.astype(np.float64) * 2**24)
    np.testing.assert_array_equal(k, np.floor(k))
    # Calls and seeds give different streams; the same (seed, call) repeats.
    assert not np.array_equal(u, oracle.uniforms(seed, offset + 1, B))
    assert not np.array_equal(u, oracle.uniforms(seed + 1, offset, B))
    np.testing.assert_array_equal(u, oracle.uniforms(seed, offset, B))


# ---------------------------------------------------------------- closed forms + brute force: min_p


def _sample_minp(values, T, min_p, k=-1, p=1.0, u=0.5):
    return oracle.sample(_row(values), torch.tensor([T]), torch.tensor([k], dtype=torch.int32),
                         torch.tensor([p]), torch.tensor([u]), want_probs=True,
                         min_p=torch.tensor([min_p]))


def test_min_p_page_example_closed_forms():
    # The pages' test row [5, 4, 3, 0, 0, 0] at T = 1: probabilities relative
    # to the largest are 1, e^-1 = 0.368, e^-2 = 0.135, e^-5 = 0.0067.
    l = [5.0, 4.0, 3.0, 0.0, 0.0, 0.0]
    q = _sample_minp(l, 1.0, 0.3)["probs"][0]  # keeps tokens 0 and 1
    assert np.count_nonzero(q) == 2
    assert abs(q[0] - math.e ** 5 / (math.e ** 5 + math.e ** 4)) < 1e-12  # 0.73106
    assert np.count_nonzero(_sample_minp(l, 1.0, 0.5)["probs"][0]) == 1
    q = _sample_minp(l, 1.0, 0.1)["probs"][0]  # e^-2 >= 0.1 > e^-5
    z = math.e ** 5 + math.e ** 4 + math.e ** 3
    np.testing.assert_allclose(q[:3], [math.e ** 5 / z, math.e ** 4 / z, math.e ** 3 / z],
                               atol=1e-12)
    assert not q[3:].any()
    # Temperature scales the threshold: at T = 2, e^(-1/2) = 0.61 >= 0.5.
    assert np.count_nonzero(_sample_minp(l, 2.0, 0.5)["probs"][0]) == 2


def test_min_p_intersects_with_top_k_and_top_p():
    l = [5.0, 4.0, 3.0, 0.0, 0.0, 0.0]
    # top_k = 2 keeps {0, 1}; min_p = 0.1 alone keeps {0, 1, 2}: the intersection.
    assert set(np.nonzero(_sample_minp(l, 1.0, 0.1, k=2)["probs"][0])[0]) == {0, 1}
    # top_p = 0.5 keeps {0}; min_p = 0.3 keeps {0, 1}.
    assert set(np.nonzero(_sample_minp(l, 1.0, 0.3, p=0.5)["probs"][0])[0]) == {0}
    # min_p = 1 keeps the maximum only (tie-free row): the argmax.
    rng = np.random.default_rng(4)
    row = rng.normal(0, 3, 500).astype(np.float32)
    r = _sample_minp(row.tolist(), 0.8, 1.0, u=0.77)
    assert r["tokens"][0] == int(np.argmax(row)) and np.count_nonzero(r["probs"][0]) == 1
    # Off (0 or negative) and tiny values change nothing on a narrow row.
    narrow = (rng.random(200) * 2).astype(np.float32).tolist()
    base = _sample1(narrow, 1.0, u=0.3)["probs"][0]
    for mp in (0.0, -1.0, 1e-30):
        np.testing.assert_array_equal(_sample_minp(narrow, 1.0, mp, u=0.3)["probs"][0], base)


@pytest.mark.parametrize("seed", range(4))
def test_min_p_brute_force_tiny_vocab(seed):
    rng = np.random.default_rng(300 + seed)
    for _ in range(40):
        V = int(rng.integers(1, 17))
        l = np.asarray(rng.normal(0, 2, V), np.float32).astype(np.float64).tolist()
        T = float(np.float32(rng.choice([0.3, 0.7, 1.0, 1.8])))
        k = int(rng.choice([-1, 2, 3, V]))
        p = float(np.float32(rng.choice([1.0, 0.9, 0.5])))
        mp = float(np.float32(rng.choice([0.01, 0.1, 0.4, 0.9])))
        u = float(np.float32(rng.random()))
        res = _sample_minp(l, T, mp, k=k, p=p, u=u)
        q_bf = brute_force.kept_probabilities(l, T, k, p, mp)
        q = res["probs"][0]
        if res["minp_margin"][0] > 1e-9 and res["topp_margin"][0] > 1e-9:
            assert set(np.nonzero(q)[0].tolist()) == set(i for i in q_bf if q_bf[i] > 0)
            for i, qi in q_bf.items():
                assert abs(q[i] - qi) < 1e-12
            if res["cdf_margin"][0] > 1e-9:
                assert res["tokens"][0] == brute_force.sample_row(l, T, k, p, u, mp)
