"""Seeded synthetic workloads for paged-KV GQA attention.

This module only draws inputs: sequence lengths, page tables, pools and
q/k/v. It holds none of the attention arithmetic, so both sides can use it.
One address computation appears here, in ``chunked_prefill``: to place real
prefix data in a pool otherwise filled with a marker value it maps each
prefix token to its pool row. Neither the kernels nor the oracle use it.

The shapes follow the Qwen3-4B attention layer the source pages benchmark
(32 query heads, 8 KV heads, head dim 128; "qwen3_flex_inference.py",
``patch_qwen3_model``; "flex_vs_vllm.md", "Setup"). The pages measure on real
prompts of a public math dataset; these seeded N(0, 1) tensors stand in for
them, with lengths drawn to the same ranges (prompt plus 512 generated
tokens).

Every tensor is produced on the CPU from a ``torch.Generator`` seeded per
workload, so a workload is reproducible bit for bit.

Conventions shared by all workloads:

* ``k_pool``/``v_pool``: bf16 ``[num_pages * page_size, H_kv, D]``.
* ``page_table``: int32 ``[max_batch, max_blocks]``; row 0 (padding slot) and
  page 0 are reserved; unassigned entries are -1.
* Decode row b reads batch slot ``batch_idx[b]`` (1-based for live rows, 0 for
  padding rows) and attends ``seq_lens[b]`` keys; its new token sits at
  ``input_pos[b] = seq_lens[b] - 1``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 128


@dataclass
class DecodeCase:
    """Inputs of one decode step: append of the new tokens, then attention."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    max_batch: int
    max_blocks: int
    scale: float
    k_pool: torch.Tensor        # bf16 [P*ps, Hkv, D] (prior context filled)
    v_pool: torch.Tensor
    page_table: torch.Tensor    # int32 [max_batch, max_blocks]
    q: torch.Tensor             # bf16 [B, Hq, D]
    k_new: torch.Tensor         # bf16 [B, Hkv, D]
    v_new: torch.Tensor
    batch_idx: torch.Tensor     # int32 [B]
    input_pos: torch.Tensor     # int32 [B]
    seq_lens: torch.Tensor      # int32 [B]
    info: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])


@dataclass
class PrefillCase:
    """Inputs of one packed prefill: attention over the packed k/v and the
    append of the same k/v into the paged pools."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    max_batch: int
    max_blocks: int
    scale: float
    q: torch.Tensor             # bf16 [T, Hq, D]
    k: torch.Tensor             # bf16 [T, Hkv, D]
    v: torch.Tensor
    batch_idx: torch.Tensor     # int32 [T]
    input_pos: torch.Tensor     # int32 [T]
    doc_lens: list
    k_pool: torch.Tensor        # bf16 pools the packed k/v are appended to
    v_pool: torch.Tensor
    page_table: torch.Tensor
    info: dict = field(default_factory=dict)

    @property
    def n_tokens(self) -> int:
        return int(self.q.shape[0])


@dataclass
class ChunkedCase:
    """Inputs of one chunked-prefill step over the paged cache: each sequence
    already holds a prefix in the pools and brings a chunk of new tokens (a
    decode token is a chunk of one); the chunk's K/V are appended, then every
    packed query token attends its slot's keys 0..input_pos through the
    pages."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    max_batch: int
    max_blocks: int
    scale: float
    q: torch.Tensor             # bf16 [T, Hq, D]
    k_new: torch.Tensor         # bf16 [T, Hkv, D] (the chunks' own K/V)
    v_new: torch.Tensor
    batch_idx: torch.Tensor     # int32 [T]
    input_pos: torch.Tensor     # int32 [T]
    prefix_lens: list           # per slot 1.., tokens already in the pools
    chunk_lens: list            # per slot 1.., new tokens in this step
    k_pool: torch.Tensor        # bf16 [P*ps, Hkv, D], prefixes filled
    v_pool: torch.Tensor
    page_table: torch.Tensor
    info: dict = field(default_factory=dict)

    @property
    def n_tokens(self) -> int:
        return int(self.q.shape[0])


def _randn_bf16(shape, gen) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def _blocks(n_tokens: int, page_size: int) -> int:
    return -(-n_tokens // page_size)


def assign_pages(blocks_per_slot, num_pages: int, max_batch: int,
                 max_blocks: int, gen, permute: bool) -> torch.Tensor:
    """Page table giving slot s (1-based) ``blocks_per_slot[s-1]`` pages.

    ``permute=False`` hands out pages 1, 2, 3, ... in order, so every slot's
    pages are consecutive (what a fresh sequential allocator does;
    "flex_vs_vllm.md", "What each option did", BLOCKS_ARE_CONTIGUOUS).
    ``permute=True`` hands them out in a seeded random order of pages
    1..num_pages-1. Page 0 and slot 0 stay reserved; unused entries are -1.
    """
    need = sum(blocks_per_slot)
    if need > num_pages - 1:
        raise ValueError(f"need {need} pages, pool has {num_pages - 1} free")
    if len(blocks_per_slot) > max_batch - 1:
        raise ValueError("more slots than the table holds")
    order = torch.arange(1, num_pages, dtype=torch.int64)
    if permute:
        order = order[torch.randperm(num_pages - 1, generator=gen)]
    table = torch.full((max_batch, max_blocks), -1, dtype=torch.int32)
    nxt = 0
    for s, nb in enumerate(blocks_per_slot, start=1):
        if nb > max_blocks:
            raise ValueError("sequence longer than max_blocks pages")
        table[s, :nb] = order[nxt:nxt + nb].to(torch.int32)
        nxt += nb
    return table


def _decode_case(name, gen, *, lens, n_pad, hq, hkv, page_size, permute,
                 max_blocks=None, pool_slack=1.0, num_pages=None,
                 fill=None) -> DecodeCase:
    """Common builder. ``lens`` are keys attended per live row (the new token
    included); live rows use slots 1..len(lens); ``n_pad`` padding rows use
    slot 0 and trail the live rows (a batch-size bucket padded at its end)."""
    d = HEAD_DIM
    live = len(lens)
    blocks = [_blocks(n, page_size) for n in lens]
    if max_blocks is None:
        max_blocks = max(blocks) if blocks else 1
    if num_pages is None:
        num_pages = 1 + int(math.ceil(sum(blocks) * pool_slack))
    max_batch = live + 1
    table = assign_pages(blocks, num_pages, max_batch, max_blocks, gen, permute)
    rows = num_pages * page_size
    if fill is None:
        k_pool = _randn_bf16((rows, hkv, d), gen)
        v_pool = _randn_bf16((rows, hkv, d), gen)
    else:
        k_pool = torch.full((rows, hkv, d), fill, dtype=torch.bfloat16)
        v_pool = torch.full((rows, hkv, d), fill, dtype=torch.bfloat16)
    B = live + n_pad
    q = _randn_bf16((B, hq, d), gen)
    k_new = _randn_bf16((B, hkv, d), gen)
    v_new = _randn_bf16((B, hkv, d), gen)
    batch_idx = torch.zeros(B, dtype=torch.int32)
    batch_idx[:live] = torch.arange(1, live + 1, dtype=torch.int32)
    seq_lens = torch.ones(B, dtype=torch.int32)   # padding rows: input_pos 0
    seq_lens[:live] = torch.tensor(lens, dtype=torch.int32)
    input_pos = seq_lens - 1
    return DecodeCase(
        name=name, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
        page_size=page_size, num_pages=num_pages, max_batch=max_batch,
        max_blocks=max_blocks, scale=1.0 / math.sqrt(d), k_pool=k_pool,
        v_pool=v_pool, page_table=table, q=q, k_new=k_new, v_new=v_new,
        batch_idx=batch_idx, input_pos=input_pos, seq_lens=seq_lens,
        info={"live": live, "pad": n_pad, "permuted": permute,
              "kv_tokens": int(sum(lens))})


def tiny_decode(seed: int = 0, permute: bool = True) -> DecodeCase:
    """B=4, Hq=8, Hkv=2, page 16, 32 physical pages. Each sequence holds
    {17, 64, 100, 130} tokens; the new token goes to position len and is then
    attended, so len+1 keys are attended. Pages by seeded permutation."""
    gen = torch.Generator().manual_seed(seed)
    ctx = [17, 64, 100, 130]
    lens = [n + 1 for n in ctx]
    return _decode_case("tiny_decode", gen, lens=lens, n_pad=0, hq=8, hkv=2,
                        page_size=16, permute=permute, num_pages=32,
                        max_blocks=16)


def qwen3_b64_decode(seed: int = 0, permute: bool = False, batch: int = 64,
                     page_size: int = 128) -> DecodeCase:
    """Qwen3-4B-shaped decode, one layer: B=64, Hq=32, Hkv=8, page 128 (or
    ``page_size``; the pages also ran 256), keys attended uniform in
    [512, 1024]. Sequential pages (contiguous fast path) or a seeded
    permutation."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(512, 1025, (batch,), generator=gen).tolist()
    suffix = "" if page_size == 128 else f"_ps{page_size}"
    return _decode_case(f"qwen3_b{batch}_decode_{'perm' if permute else 'seq'}{suffix}",
                        gen, lens=lens, n_pad=0, hq=32, hkv=8, page_size=page_size,
                        permute=permute, max_blocks=(1024 + page_size - 1) // page_size)


def padded_bucket_decode(seed: int = 0) -> DecodeCase:
    """B=64 bucket with 40 live sequences (keys uniform in [1, 2048]) and 24
    padding rows on batch slot 0; Hq=32, Hkv=8, page 128, permuted pages."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, 2049, (40,), generator=gen).tolist()
    return _decode_case("padded_bucket_decode", gen, lens=lens, n_pad=24,
                        hq=32, hkv=8, page_size=128, permute=True,
                        max_blocks=16)


def long_context_decode(seed: int = 0, batch: int = 256) -> DecodeCase:
    """B=256, Hq=32, Hkv=8, page 128, keys log-uniform in [128, 8192],
    permuted pages; pool sized to the need plus 10 %."""
    gen = torch.Generator().manual_seed(seed)
    u = torch.rand(batch, generator=gen, dtype=torch.float64)
    lens = torch.exp(math.log(128) + u * (math.log(8192) - math.log(128)))
    lens = lens.round().clamp(128, 8192).to(torch.int64).tolist()
    return _decode_case(f"long_context_b{batch}_decode", gen, lens=lens,
                        n_pad=0, hq=32, hkv=8, page_size=128, permute=True,
                        max_blocks=64, pool_slack=1.1)


def custom_decode(seed: int, lens, *, hq=32, hkv=8, page_size=128, n_pad=0,
                  permute=True, max_blocks=None, num_pages=None,
                  fill=None) -> DecodeCase:
    """Arbitrary decode case for edge tests (lengths of 0 are allowed: such a
    row has a slot but attends nothing)."""
    gen = torch.Generator().manual_seed(seed)
    return _decode_case("custom_decode", gen, lens=list(lens), n_pad=n_pad,
                        hq=hq, hkv=hkv, page_size=page_size, permute=permute,
                        max_blocks=max_blocks, num_pages=num_pages, fill=fill)


def packed_prefill(seed: int = 0, n_docs: int = 64, lo: int = 64,
                   hi: int = 1024, hq: int = 32, hkv: int = 8,
                   page_size: int = 128, permute: bool = True,
                   doc_lens=None) -> PrefillCase:
    """Packed document-causal prefill: ``n_docs`` prompts with lengths uniform
    in [lo, hi] concatenated into one sequence; token t of document s (slot
    s+1) has ``batch_idx = s+1`` and ``input_pos = t``. The pools the packed
    k/v are appended to hold exactly the pages the documents need."""
    gen = torch.Generator().manual_seed(seed)
    if doc_lens is None:
        doc_lens = torch.randint(lo, hi + 1, (n_docs,), generator=gen).tolist()
    doc_lens = [int(n) for n in doc_lens]
    T = sum(doc_lens)
    d = HEAD_DIM
    q = _randn_bf16((T, hq, d), gen)
    k = _randn_bf16((T, hkv, d), gen)
    v = _randn_bf16((T, hkv, d), gen)
    batch_idx = torch.cat([torch.full((n,), s + 1, dtype=torch.int32)
                           for s, n in enumerate(doc_lens)]) if T else \
        torch.zeros(0, dtype=torch.int32)
    input_pos = torch.cat([torch.arange(n, dtype=torch.int32)
                           for n in doc_lens]) if T else \
        torch.zeros(0, dtype=torch.int32)
    blocks = [_blocks(n, page_size) for n in doc_lens]
    max_blocks = max(blocks) if blocks else 1
    num_pages = 1 + sum(blocks)
    max_batch = len(doc_lens) + 1
    table = assign_pages(blocks, num_pages, max_batch, max_blocks, gen, permute)
    rows = num_pages * page_size
    k_pool = torch.zeros((rows, hkv, d), dtype=torch.bfloat16)
    v_pool = torch.zeros((rows, hkv, d), dtype=torch.bfloat16)
    return PrefillCase(
        name=f"packed_prefill_{len(doc_lens)}docs", num_q_heads=hq,
        num_kv_heads=hkv, head_dim=d, page_size=page_size,
        num_pages=num_pages, max_batch=max_batch, max_blocks=max_blocks,
        scale=1.0 / math.sqrt(d), q=q, k=k, v=v, batch_idx=batch_idx,
        input_pos=input_pos, doc_lens=doc_lens, k_pool=k_pool, v_pool=v_pool,
        page_table=table,
        info={"tokens": T, "pairs": int(sum(n * (n + 1) // 2 for n in doc_lens))})


def chunked_prefill(seed: int = 0, *, prefix_lens=None, chunk_lens=None, n_chunks: int = 16,
                    chunk: int = 512, prefix_lo: int = 512, prefix_hi: int = 4096,
                    n_decode: int = 48, decode_lo: int = 512, decode_hi: int = 2048,
                    hq: int = 32, hkv: int = 8, page_size: int = 128, permute: bool = True,
                    shuffle: bool = True, n_pad: int = 0, fill=None) -> ChunkedCase:
    """One mixed step of chunked prefill, the pages' missing piece (prefill
    and decode in one pass; "flex_vs_vllm.md", "What's left on the table"):
    ``n_chunks`` sequences with a prefix of U[prefix_lo, prefix_hi] tokens in
    the cache bring ``chunk`` new tokens each, and ``n_decode`` sequences with
    a prefix of U[decode_lo, decode_hi] bring one. ``prefix_lens`` and
    ``chunk_lens`` (per slot) override the draw. Each sequence's chunk is
    contiguous in the packed order; the sequences come in a seeded random
    order (``shuffle``) and ``n_pad`` padding tokens (slot 0) trail them. The
    pools hold random prefixes; rows past a sequence's prefix hold random
    values, or ``fill`` when given (e.g. NaN)."""
    gen = torch.Generator().manual_seed(seed)
    if prefix_lens is None:
        pre = torch.randint(prefix_lo, prefix_hi + 1, (n_chunks,), generator=gen).tolist()
        pre += torch.randint(decode_lo, decode_hi + 1, (n_decode,), generator=gen).tolist()
        chunk_lens = [chunk] * n_chunks + [1] * n_decode
    else:
        pre = list(prefix_lens)
        chunk_lens = list(chunk_lens)
    pre = [int(x) for x in pre]
    chunk_lens = [int(x) for x in chunk_lens]
    S = len(pre)
    d = HEAD_DIM
    # the packed order is drawn before anything whose size depends on the
    # page size, so that page sizes are compared on the same token order
    order = torch.randperm(S, generator=gen).tolist() if shuffle else list(range(S))
    blocks = [_blocks(p + c, page_size) for p, c in zip(pre, chunk_lens)]
    max_blocks = max(blocks) if blocks else 1
    num_pages = 1 + sum(blocks)
    table = assign_pages(blocks, num_pages, S + 1, max_blocks, gen, permute)
    rows = num_pages * page_size
    if fill is None:
        k_pool = _randn_bf16((rows, hkv, d), gen)
        v_pool = _randn_bf16((rows, hkv, d), gen)
    else:
        k_pool = torch.full((rows, hkv, d), fill, dtype=torch.bfloat16)
        v_pool = torch.full((rows, hkv, d), fill, dtype=torch.bfloat16)
        for s in range(S):   # the prefixes are real data
            for t in range(pre[s]):
                r = int(table[s + 1, t // page_size]) * page_size + t % page_size
                k_pool[r] = _randn_bf16((hkv, d), gen)
                v_pool[r] = _randn_bf16((hkv, d), gen)
    bidx, pos = [], []
    for s in order:
        bidx += [s + 1] * chunk_lens[s]
        pos += list(range(pre[s], pre[s] + chunk_lens[s]))
    bidx += [0] * n_pad
    pos += [0] * n_pad
    T = len(bidx)
    q = _randn_bf16((T, hq, d), gen)
    k_new = _randn_bf16((T, hkv, d), gen)
    v_new = _randn_bf16((T, hkv, d), gen)
    return ChunkedCase(
        name=f"chunked_prefill_{S}seq_T{T}", num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
        page_size=page_size, num_pages=num_pages, max_batch=S + 1, max_blocks=max_blocks,
        scale=1.0 / math.sqrt(d), q=q, k_new=k_new, v_new=v_new,
        batch_idx=torch.tensor(bidx, dtype=torch.int32),
        input_pos=torch.tensor(pos, dtype=torch.int32), prefix_lens=pre,
        chunk_lens=chunk_lens, k_pool=k_pool, v_pool=v_pool, page_table=table,
        info={"tokens": T, "pairs": int(sum((p + 1) for b, p in zip(bidx, pos) if b != 0))})


def rope_tables(max_pos: int, head_dim: int = HEAD_DIM, theta: float = 1.0e6):
    """fp32 cos/sin tables ``[max_pos, head_dim/2]`` of the standard rotary
    embedding: angle ``p * theta**(-2i/head_dim)`` for row p, column i
    (Qwen3's ``rope_theta`` is 1e6). These are inputs to the RoPE-fused
    append, the way the model passes cos/sin to its attention layers."""
    i = torch.arange(0, head_dim // 2, dtype=torch.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv_freq[None, :]
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "qwen3_b64_decode": qwen3_b64_decode,
    "padded_bucket_decode": padded_bucket_decode,
    "long_context_decode": long_context_decode,
    "packed_prefill": packed_prefill,
    "chunked_prefill": chunked_prefill,
}


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a CPU bf16 tensor as a numpy uint16 array
    (a reinterpretation, no arithmetic)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
