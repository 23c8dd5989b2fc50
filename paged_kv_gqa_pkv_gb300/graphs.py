"""Bucketed CUDA-graph decode: append + split-KV decode captured once per
batch-size bucket and replayed (by default as the fused append + decode
call, two kernels a step; ``fused=False`` captures the separate append).

This follows the pages' engine: one CUDA graph per batch-size bucket, decode
dispatched to the smallest bucket that fits, and the unused rows of the
bucket padded with batch slot 0, the reserved no-op slot
("flex_paged_attention.py" commit log, "Why this works", item 3;
"qwen3_flex_inference.py", ``capture_decode_cudagraph`` and ``_decode_step``).
Graph replay was the pages' largest single lever ("flex_vs_vllm.md", "What
each option did": eager ~420 tok/s, +CUDA graphs 4279).

The graphs hold fixed device pointers: the KV pools and the page table are
the caller's tensors (updated in place between steps), while q, the new k/v,
batch_idx, input_pos and seq_lens live in static buffers that ``step`` fills.
Padding rows get batch_idx 0, so the append skips them and decode returns
zeros and -inf for them. Every kernel is the library's; PyTorch only captures
and replays.
"""

from __future__ import annotations

import torch

from . import binding

DEFAULT_BUCKETS = (1, 2, 4, 8, 16, 32, 48, 64)


class DecodeGraphs:
    """Captured append + decode graphs for a fixed paged cache.

    Args:
        k_pool, v_pool: bf16 ``[P*ps, H_kv, D]`` CUDA tensors (kept by pointer).
        page_table: int32 ``[max_batch, max_blocks]`` CUDA tensor (kept by pointer).
        page_size: tokens per page.
        num_q_heads: query heads per row.
        scale: softmax scale.
        buckets: batch sizes to capture, ascending.
        fused: capture ``pkv_decode_append_attention`` (the new token is
            written at ``seq_lens - 1``, so ``input_pos`` must equal
            ``seq_lens - 1`` on live rows) instead of ``pkv_append`` followed by
            ``pkv_decode_attention``.
    """

    def __init__(self, k_pool, v_pool, page_table, page_size: int, num_q_heads: int,
                 scale: float, buckets=DEFAULT_BUCKETS, fused: bool = True):
        self.k_pool, self.v_pool, self.page_table = k_pool, v_pool, page_table
        self.page_size, self.scale = page_size, float(scale)
        self.fused = bool(fused)
        self.buckets = tuple(sorted(int(b) for b in buckets))
        if not self.buckets or self.buckets[0] < 1:
            raise ValueError("buckets must be positive batch sizes")
        dev = k_pool.device
        hkv, d = k_pool.shape[1], k_pool.shape[2]
        bmax = self.buckets[-1]
        self.q = torch.zeros((bmax, num_q_heads, d), dtype=torch.bfloat16, device=dev)
        self.k_new = torch.zeros((bmax, hkv, d), dtype=torch.bfloat16, device=dev)
        self.v_new = torch.zeros((bmax, hkv, d), dtype=torch.bfloat16, device=dev)
        self.batch_idx = torch.zeros(bmax, dtype=torch.int32, device=dev)
        self.input_pos = torch.zeros(bmax, dtype=torch.int32, device=dev)
        self.seq_lens = torch.zeros(bmax, dtype=torch.int32, device=dev)
        self.out = torch.zeros((bmax, num_q_heads, d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.zeros((bmax, num_q_heads), dtype=torch.float32, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = binding.pkv_decode_workspace_size(k_pool, page_table, page_size, bmax, num_q_heads)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.graphs = {}
        # largest bucket first, as the pages do; a warm-up call per bucket does
        # the library's one-time set-up outside capture
        for b in reversed(self.buckets):
            self._launch(b)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._launch(b)
            self.graphs[b] = g
        torch.cuda.synchronize()

    def _launch(self, b: int) -> None:
        if self.fused:
            binding.pkv_decode_append_attention(
                self.k_pool, self.v_pool, self.page_table, self.q[:b], self.k_new[:b],
                self.v_new[:b], self.batch_idx[:b], self.seq_lens[:b], self.page_size,
                self.scale, out=self.out[:b], lse=self.lse[:b], workspace=self.workspace,
                dev_err=self.dev_err)
            return
        binding.pkv_append(self.k_pool, self.v_pool, self.page_table, self.k_new[:b],
                           self.v_new[:b], self.batch_idx[:b], self.input_pos[:b],
                           self.page_size, dev_err=self.dev_err)
        binding.pkv_decode_attention(self.k_pool, self.v_pool, self.page_table, self.q[:b],
                                     self.batch_idx[:b], self.seq_lens[:b], self.page_size,
                                     self.scale, out=self.out[:b], lse=self.lse[:b],
                                     workspace=self.workspace, dev_err=self.dev_err)

    def bucket_for(self, batch: int) -> int:
        for b in self.buckets:
            if b >= batch:
                return b
        raise ValueError(f"batch {batch} exceeds the largest bucket {self.buckets[-1]}")

    def step(self, q, k_new, v_new, batch_idx, input_pos, seq_lens):
        """One decode step for ``B = q.shape[0]`` rows: copies the inputs into the
        static buffers, pads the bucket with slot-0 rows, replays the bucket's
        graph. Returns views ``(out[:B], lse[:B])`` of the static outputs (valid
        until the next step)."""
        B = q.shape[0]
        b = self.bucket_for(B)
        for dst, src in ((self.q, q), (self.k_new, k_new), (self.v_new, v_new),
                         (self.batch_idx, batch_idx), (self.input_pos, input_pos),
                         (self.seq_lens, seq_lens)):
            dst[:B].copy_(src, non_blocking=True)
            if b > B:
                dst[B:b].zero_()
        self.graphs[b].replay()
        return self.out[:B], self.lse[:B]
