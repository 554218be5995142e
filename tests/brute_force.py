"""Brute-force restatement of the sampler for tiny vocabularies (V <= 16).

Used only to pin the oracle.  It is written from the rank definition rather
than from a sort: token i's rank is the number of tokens that come before it in
the order (logit descending, index ascending); top-k keeps rank < k; the top-p
"mass before i" is summed over the kept tokens of smaller rank; the draw walks
the kept set in vocab order.  O(V^2) pure Python, fp64.

Source: "mini-sglang from Scratch", page "The engine and the sampler",
section "The sampler" (sample_torch), with multinomial replaced by an inverse
CDF against a supplied uniform.
"""

from __future__ import annotations

import math


def rank_of(l, i):
    return sum(1 for j in range(len(l)) if l[j] > l[i] or (l[j] == l[i] and j < i))


def kept_probabilities(l, T, k, p, min_p=0.0):
    """{token: q} over the kept set S of one sampled row.  min_p > 0 keeps
    only the tokens whose probability is at least min_p times the largest
    (exercise 2 of the same page), intersected with the top-k / top-p set."""
    V = len(l)
    if k < 1 or k >= V:
        k = V
    ranks = [rank_of(l, i) for i in range(V)]
    K = [i for i in range(V) if ranks[i] < k]
    m = max(l)
    w = {i: math.exp((l[i] - m) / T) for i in K}
    zk = sum(w.values())
    if p < 1.0:
        S = [i for i in K
             if sum(w[j] for j in K if ranks[j] < ranks[i]) / zk < p]
    else:
        S = K
    if min_p > 0.0:
        pmax = max(math.exp((l[j] - m) / T) for j in range(V))  # 1 at the maximum
        S = [i for i in S if w[i] / pmax >= min(min_p, 1.0)]
    zs = sum(w[i] for i in S)
    return {i: w[i] / zs for i in S}


def draw(q, u):
    """Inverse CDF over the kept set in ascending vocab index."""
    c = 0.0
    for i in sorted(q):
        c += q[i]
        if u < c:
            return i
    return max(i for i in q if q[i] > 0)


def sample_row(l, T, k, p, u, min_p=0.0):
    return draw(kept_probabilities(l, T, k, p, min_p), u)
