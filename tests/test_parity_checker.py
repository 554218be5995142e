"""The parity checker itself (CPU): it accepts the oracle's own tokens, every
excused row is validated rather than skipped, and a planted wrong token in an
exact or an excused row is caught.  A checker that let excused rows through
unchecked would pass any token there."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gb300 import workloads
from parity import TOL, admissible_sets, check_sampler


def _case(name, **kw):
    w = workloads.make(name, **kw)
    r = oracle.sample(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, threads=8)
    return w, r


def test_oracle_tokens_pass_and_every_excused_row_is_validated():
    w, r = _case("mixed", B=96, V=40000)
    st = check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, r["tokens"],
                       ores=r)
    excused = st["excused_cdf"] + st["excused_topp"] + st["excused_minp"]
    assert excused > 0, st  # the case exercises the excused branch
    assert st["validated"] == excused
    assert st["greedy"] + st["exact"] + st["validated"] == w.B


@pytest.mark.parametrize("kind", ["exact", "topp"])
def test_wrong_token_is_caught(kind):
    w, r = _case("mixed", B=96, V=40000)
    t = w.temperature.numpy()
    sampled = t > 0
    if kind == "exact":
        rows = np.nonzero(sampled & (r["topp_margin"] >= TOL) & (r["cdf_margin"] >= TOL))[0]
    else:
        rows = np.nonzero(sampled & (r["topp_margin"] < TOL))[0]
    assert len(rows) > 0
    b = int(rows[0])
    bad = r["tokens"].copy()
    bad[b] = (bad[b] + 1) % w.V
    with pytest.raises(AssertionError):
        check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, bad, ores=r)


def test_token_outside_the_vocabulary_is_caught():
    w, r = _case("mixed", B=32, V=20000)
    t = w.temperature.numpy()
    b = int(np.nonzero(t > 0)[0][0])
    bad = r["tokens"].copy()
    bad[b] = -1
    with pytest.raises(AssertionError):
        check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, bad, ores=r)


def test_admissible_sets_are_the_prefixes_between_the_bounding_cuts():
    # Four equal logits and a -inf one: with p = 0.5 the mass before the
    # j-th of them is exactly j / 4 of the total, so p = 0.5 sits on a
    # boundary and the admissible cuts keep 2 or 3 of them (p - TOL, p + TOL).
    row = torch.tensor([1.0, 1.0, 1.0, 1.0, float("-inf")])
    sets = admissible_sets(row, 1.0, -1, 0.5, None, topp_free=True, minp_free=False)
    assert [s.tolist() for s in sets] == [[0, 1], [0, 1, 2]]
    # Without the top-p freedom there is exactly the oracle's set.
    one = admissible_sets(row, 1.0, -1, 0.5, None, topp_free=False, minp_free=False)
    assert [s.tolist() for s in one] == [[0, 1]]


def test_probs_of_an_excused_row_must_match_an_admissible_set():
    row = torch.tensor([[1.0, 1.0, 1.0, 1.0, float("-inf")]])
    t = torch.tensor([1.0])
    p = torch.tensor([0.5])
    u = torch.tensor([0.1])
    r = oracle.sample(row, t, None, p, u, want_probs=True)
    assert r["topp_margin"][0] < TOL
    good = np.zeros((1, 5), np.float32)
    good[0, :3] = 1.0 / 3.0  # the cut that keeps three
    check_sampler(row, t, None, p, u, np.array([0]), gpu_probs=good, ores=r)
    bad = np.zeros((1, 5), np.float32)
    bad[0, :4] = 0.25  # keeps all four: not admissible
    with pytest.raises(AssertionError):
        check_sampler(row, t, None, p, u, np.array([0]), gpu_probs=bad, ores=r)
