"""Comparison of the CUDA sampler's output with the CPU oracle.

Rules (the parity bar):
  * greedy rows: tokens bit-exact;
  * sampled rows: tokens exact unless the uniform lies within TOL of a CDF
    boundary (oracle ``cdf_margin`` < TOL) or the top-p cut is within TOL of
    a boundary (oracle ``topp_margin`` < TOL);
  * kept-set probabilities (``probs_out``) within TOL absolute of the
    oracle's, with the same kept set, on every row whose top-p cut is not
    excused.
Excused rows are still checked for validity: the GPU's kept set must lie
between the oracle's kept sets at p - TOL and p + TOL, its probabilities must
be the renormalised exp(l / T) of that set within TOL, and the token must be
in it with the uniform inside the token's CDF interval up to TOL.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = 1e-5


def _row_params(temperature, top_k, top_p, uniform, b):
    T = None if temperature is None else float(temperature[b])
    k = -1 if top_k is None else int(top_k[b])
    p = 1.0 if top_p is None else float(top_p[b])
    u = None if uniform is None else float(uniform[b])
    return T, k, p, u


def _as_np(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().numpy()
    return np.asarray(x)


def check_sampler(logits: torch.Tensor, temperature, top_k, top_p, uniform,
                  gpu_tokens, gpu_probs=None, ores=None, min_p=None) -> dict:
    """Asserts parity; returns counts of checked / excused rows.  Rows whose
    min_p boundary lies within TOL of a kept token's relative probability are
    excused like the top-p boundary rows (and only counted)."""
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
    lf = logits.double().numpy()
    stats = {"greedy": 0, "exact": 0, "excused_cdf": 0, "excused_topp": 0, "excused_minp": 0,
             "probs_checked": 0}
    for b in range(B):
        ot = int(ores["tokens"][b])
        greedy = t is None or not (t[b] > 0)
        if greedy or ot < 0:
            assert gt[b] == ot, f"row {b}: gpu {gt[b]} oracle {ot} (greedy/error row)"
            stats["greedy"] += 1
            if gq is not None and ot >= 0:
                assert gq[b, ot] == 1.0 and np.count_nonzero(gq[b]) == 1
            continue
        if ores["minp_margin"][b] < TOL:
            stats["excused_minp"] += 1
            continue
        topp_ok = ores["topp_margin"][b] >= TOL
        cdf_ok = ores["cdf_margin"][b] >= TOL
        if not topp_ok and mp is not None and mp[b] > 0:
            stats["excused_topp"] += 1
            continue
        if topp_ok and cdf_ok:
            assert gt[b] == ot, (f"row {b}: gpu token {gt[b]} oracle {ot} "
                                 f"(margins topp {ores['topp_margin'][b]:.3g}, "
                                 f"cdf {ores['cdf_margin'][b]:.3g})")
            stats["exact"] += 1
        elif topp_ok:
            stats["excused_cdf"] += 1
        else:
            stats["excused_topp"] += 1
        if gq is None and topp_ok and not cdf_ok:
            # Kept set is exact; the token must sit in an interval within TOL of u.
            q = ores["probs"][b] if ores["probs"] is not None else None
            if q is not None:
                c = np.cumsum(q)
                lo = c[gt[b]] - q[gt[b]]
                assert q[gt[b]] > 0 and lo - TOL <= u[b] < c[gt[b]] + TOL
        if gq is None:
            continue
        qg = gq[b].astype(np.float64)
        sg = np.nonzero(qg)[0]
        assert gt[b] in set(sg.tolist()), f"row {b}: token {gt[b]} not in the gpu kept set"
        if topp_ok:
            qo = ores["probs"][b]
            so = np.nonzero(qo)[0]
            assert np.array_equal(sg, so), f"row {b}: kept sets differ ({len(sg)} vs {len(so)})"
            err = np.max(np.abs(qg - qo))
            assert err <= TOL, f"row {b}: kept-set probability error {err:.3g}"
            if not cdf_ok:
                c = np.cumsum(qo)
                lo = c[gt[b]] - qo[gt[b]]
                assert lo - TOL <= u[b] < c[gt[b]] + TOL, f"row {b}: token outside its interval"
        else:
            # Excused top-p cut: the gpu set must be a valid cut within TOL.
            T, kk, pp, _ = _row_params(t, k, p, u, b)
            lo_set, hi_set = [], []
            for pad, acc in ((-TOL, lo_set), (TOL, hi_set)):
                pq = float(np.clip(pp + pad, 1e-6, 1.0))
                r = oracle.sample(logits[b:b + 1], torch.tensor([T]),
                                  torch.tensor([kk], dtype=torch.int32), torch.tensor([pq]),
                                  torch.tensor([0.5]), want_probs=True)
                acc.extend(np.nonzero(r["probs"][0])[0].tolist())
            sset = set(sg.tolist())
            assert set(lo_set) <= sset <= set(hi_set), f"row {b}: gpu kept set is not a valid cut"
            w = np.exp((lf[b, sg] - lf[b].max()) / T)
            err = np.max(np.abs(qg[sg] - w / w.sum()))
            assert err <= TOL, f"row {b}: probability error {err:.3g} on the gpu kept set"
            c = np.cumsum(qg)
            lo = c[gt[b]] - qg[gt[b]]
            assert lo - TOL <= u[b] < c[gt[b]] + TOL, f"row {b}: token outside its interval"
        stats["probs_checked"] += 1
    return stats
