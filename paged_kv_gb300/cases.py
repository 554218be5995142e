"""A few pkv_sample_batch calls on one row mix, for profilers.

``python -m paged_kv_gb300.cases <case> [calls]`` runs `calls` (default 6)
sampler calls on the mixed workload's logits (B=256, V=151936 bf16, four
rotating buffers) with the parameters of one case: ``greedy`` (temperature
0), ``plain`` (T=1), ``topk50``, ``topp`` (p=0.9, no top-k), ``topk50_topp``
or ``mixed`` (the benchmark's own parameters); or on one of the other
workloads with its own parameters: ``pr1``, ``greedy_batch`` (B=64, V=128256
bf16, all greedy), ``nucleus`` (fp32) or ``large``.  Needs a GPU and the built
library.
"""

from __future__ import annotations

import sys

import torch

from paged_kv_gb300 import pkv, workloads


def params(case: str, w):
    B = w.B
    one = torch.ones(B)
    k50 = torch.full((B,), 50, dtype=torch.int32)
    p09 = torch.full((B,), 0.9)
    table = {"greedy": (torch.zeros(B), None, None), "plain": (one, None, None),
             "topk50": (one, k50, None), "topp": (one, None, p09),
             "topk50_topp": (one, k50, p09), "mixed": (w.temperature, w.top_k, w.top_p)}
    if case not in table:
        raise SystemExit(f"unknown case {case!r}; one of {sorted(table)}")
    return table[case]


WORKLOADS = {"pr1": "pr1", "greedy_batch": "greedy", "nucleus": "nucleus", "large": "large"}


def main(argv=None) -> None:
    argv = sys.argv[1:] if argv is None else argv
    case = argv[0] if argv else "mixed"
    calls = int(argv[1]) if len(argv) > 1 else 6
    dev = torch.device("cuda")
    if case in WORKLOADS:
        w = workloads.make(WORKLOADS[case])
        t, k, p = (None if x is None else x.to(dev) for x in (w.temperature, w.top_k, w.top_p))
    else:
        w = workloads.mixed()
        t, k, p = (None if x is None else x.to(dev) for x in params(case, w))
    base = w.logits.to(dev)
    bufs = [base] + [base.clone() for _ in range(3 if w.B * w.V * w.elt < (1 << 30) else 0)]
    u = w.uniform.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for i in range(calls):
        pkv.sample_batch(bufs[i % len(bufs)], t, k, p, u, status=status)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise SystemExit(f"status word {int(status.item())}")
    print("ok", case, calls)


if __name__ == "__main__":
    main()
