"""Comparison of the CUDA sampler's output with the CPU oracle.

Rules (the parity bar):
  * greedy rows: tokens bit-exact;
  * sampled rows: tokens exact unless the uniform lies within TOL of a CDF
    boundary (oracle ``cdf_margin`` < TOL), the top-p cut is within TOL of a
    boundary (``topp_margin`` < TOL) or a kept token's probability is within
    TOL (relative) of the min_p threshold (``minp_margin`` < TOL);
  * kept-set probabilities (``probs_out``) within TOL absolute of the
    oracle's, with the same kept set, on every row that is not excused.

Excused rows are validated, never skipped.  Their kept set may be any cut the
tolerance allows: the oracle's kept sets at (p - TOL, min_p * (1 + TOL)) and
(p + TOL, min_p * (1 - TOL)) bound it, and every set in between is a prefix
of the (logit desc, index asc) order whose length lies between theirs.  The
GPU token must be in one such set S with the uniform inside the token's CDF
interval (S renormalised, vocab order) up to TOL; with ``probs_out`` the GPU's
own set must be one of them and its probabilities the renormalised
exp((l - m) / T) of that set within TOL.  A row excused by the CDF margin
alone has exactly one admissible set: the oracle's.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = 1e-5


def _as_np(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().numpy()
    return np.asarray(x)


def _oracle_set(row: torch.Tensor, T: float, k: int, p: float, mp: float | None) -> np.ndarray:
    """Indices the oracle keeps (nonzero probability) for one row."""
    r = oracle.sample(row[None], torch.tensor([T], dtype=torch.float32),
                      torch.tensor([k], dtype=torch.int32),
                      torch.tensor([p], dtype=torch.float32),
                      torch.tensor([0.5], dtype=torch.float32), want_probs=True,
                      min_p=None if mp is None else torch.tensor([mp], dtype=torch.float32))
    return np.nonzero(r["probs"][0])[0]


def admissible_sets(row: torch.Tensor, T: float, k: int, p: float, mp: float | None,
                    topp_free: bool, minp_free: bool) -> list[np.ndarray]:
    """Every kept set the tolerance admits for one row (sorted index arrays)."""
    p_lo, p_hi = (max(p - TOL, 1e-6), min(p + TOL, 1.0)) if topp_free else (p, p)
    if mp is not None and minp_free:
        m_lo, m_hi = mp * (1 + TOL), mp * (1 - TOL)
    else:
        m_lo = m_hi = mp
    lo = _oracle_set(row, T, k, p_lo, m_lo)
    hi = _oracle_set(row, T, k, p_hi, m_hi)
    assert set(lo.tolist()) <= set(hi.tolist()), "oracle kept sets are not nested"
    if len(lo) == len(hi):
        return [hi]
    lf = row.double().numpy()
    extra = np.setdiff1d(hi, lo)
    extra = extra[np.lexsort((extra, -lf[extra]))]  # (logit desc, index asc)
    return [np.sort(np.concatenate([lo, extra[:j]])) for j in range(len(extra) + 1)]


def _interval_ok(lf: np.ndarray, T: float, s: np.ndarray, tok: int, u: float) -> bool:
    """tok is in s and u lies in tok's CDF interval of s (renormalised exp((l - m) / T),
    vocab order) up to TOL."""
    if tok < 0 or tok not in set(s.tolist()):
        return False
    w = np.exp((lf[s] - np.max(lf[np.isfinite(lf)])) / T)
    q = w / w.sum()
    c = np.cumsum(q)
    j = int(np.searchsorted(s, tok))
    return q[j] > 0 and c[j] - q[j] - TOL <= u < c[j] + TOL


def validate_excused(row: torch.Tensor, T: float, k: int, p: float, mp: float | None, u: float,
                     tok: int, topp_free: bool, minp_free: bool, gq_row=None) -> int:
    """Asserts that an excused row's token (and GPU kept set, if given) is one
    the tolerance admits; returns the number of admissible sets."""
    lf = row.double().numpy()
    sets = admissible_sets(row, T, k, p, mp, topp_free, minp_free)
    if gq_row is not None:
        sg = np.nonzero(gq_row)[0]
        match = [s for s in sets if np.array_equal(s, sg)]
        assert match, f"gpu kept set ({len(sg)}) is not an admissible cut " \
                      f"({len(sets[0])}..{len(sets[-1])})"
        w = np.exp((lf[sg] - np.max(lf[np.isfinite(lf)])) / T)
        err = np.max(np.abs(gq_row[sg].astype(np.float64) - w / w.sum()))
        assert err <= TOL, f"probability error {err:.3g} on the gpu kept set"
        sets = match
    assert any(_interval_ok(lf, T, s, tok, u) for s in sets), \
        f"token {tok} with u={u} is in no admissible set's interval"
    return len(sets)


def check_sampler(logits: torch.Tensor, temperature, top_k, top_p, uniform,
                  gpu_tokens, gpu_probs=None, ores=None, min_p=None) -> dict:
    """Asserts parity; returns counts of exact, greedy and excused rows (every
    excused row is validated: ``validated`` counts them)."""
    logits = logits.detach().cpu()
    B, V = logits.shape
    if ores is None:
        ores = oracle.sample(logits, temperature, top_k, top_p, uniform,
                             want_probs=gpu_probs is not None, threads=8, min_p=min_p)
    mp = _as_np(min_p)
    t = _as_np(temperature)
    k = _as_np(top_k)
    p = _as_np(top_p)
    u = _as_np(uniform)
    gt = _as_np(gpu_tokens).astype(np.int64)
    gq = _as_np(gpu_probs)
    stats = {"greedy": 0, "exact": 0, "excused_cdf": 0, "excused_topp": 0, "excused_minp": 0,
             "validated": 0, "probs_checked": 0}
    for b in range(B):
        ot = int(ores["tokens"][b])
        greedy = t is None or not (t[b] > 0)
        if greedy or ot < 0:
            assert gt[b] == ot, f"row {b}: gpu {gt[b]} oracle {ot} (greedy/error row)"
            stats["greedy"] += 1
            if gq is not None and ot >= 0:
                assert gq[b, ot] == 1.0 and np.count_nonzero(gq[b]) == 1
            continue
        assert 0 <= gt[b] < V, f"row {b}: gpu token {gt[b]} outside [0, {V})"
        mpb = float(mp[b]) if mp is not None and mp[b] > 0 else None
        minp_free = mpb is not None and ores["minp_margin"][b] < TOL
        topp_free = ores["topp_margin"][b] < TOL
        cdf_free = ores["cdf_margin"][b] < TOL
        if not (minp_free or topp_free or cdf_free):
            assert gt[b] == ot, (f"row {b}: gpu token {gt[b]} oracle {ot} "
                                 f"(margins topp {ores['topp_margin'][b]:.3g}, "
                                 f"cdf {ores['cdf_margin'][b]:.3g})")
            stats["exact"] += 1
            if gq is not None:
                qg = gq[b].astype(np.float64)
                qo = ores["probs"][b]
                sg, so = np.nonzero(qg)[0], np.nonzero(qo)[0]
                assert np.array_equal(sg, so), f"row {b}: kept sets differ ({len(sg)} vs {len(so)})"
                err = np.max(np.abs(qg - qo))
                assert err <= TOL, f"row {b}: kept-set probability error {err:.3g}"
                stats["probs_checked"] += 1
            continue
        if minp_free:
            stats["excused_minp"] += 1
        elif topp_free:
            stats["excused_topp"] += 1
        else:
            stats["excused_cdf"] += 1
        T = float(t[b])
        kk = -1 if k is None else int(k[b])
        pp = 1.0 if p is None else float(p[b])
        try:
            validate_excused(logits[b], T, kk, pp, mpb, float(u[b]), int(gt[b]), topp_free,
                             minp_free, None if gq is None else gq[b])
        except AssertionError as e:
            raise AssertionError(f"row {b} (excused: minp {minp_free}, topp {topp_free}, "
                                 f"cdf {cdf_free}): {e}") from None
        stats["validated"] += 1
        if gq is not None:
            stats["probs_checked"] += 1
    return stats
