"""GB300-native decode-step tail: batched per-request sampling with fused
token write-back, and paged-KV page allocation / page-table fill.

The work runs in the CUDA library ``libpkv.so`` (C ABI in ``include/pkv.h``);
``paged_kv_gb300.pkv`` is its thin Python binding and
``paged_kv_gb300.workloads`` draws seeded synthetic inputs.
"""

__all__ = ["pkv", "workloads"]
