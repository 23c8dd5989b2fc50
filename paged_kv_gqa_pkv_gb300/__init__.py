"""GB300-native attention over a paged KV cache.

The compute lives in ``libpkv.so`` (hand-written CUDA for sm_103a, C ABI
declared in ``include/pkv.h``). ``paged_kv_gqa_pkv_gb300.binding`` is the thin
ctypes layer over it; ``paged_kv_gqa_pkv_gb300.graphs`` captures one decode
step per batch-size bucket as a CUDA graph; ``paged_kv_gqa_pkv_gb300.workloads``
draws seeded synthetic inputs; ``paged_kv_gqa_pkv_gb300.sharding`` holds the
host-side logic of a multi-rank run (per-rank seeds, max-over-ranks timing).
"""

__all__ = ["binding", "graphs", "sharding", "workloads"]
