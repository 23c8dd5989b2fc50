"""K1 pkv_append on the GPU: bit-exact against the oracle on every pool byte,
including slots it must not touch, and error bits instead of faults for
unreserved or out-of-range entries."""

import numpy as np
import pytest
import torch

import oracle.paged_attention as orc
from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from paged_kv_gqa_pkv_gb300.workloads import bf16_bits
from tests.parity import gpu, new_dev_err

pytestmark = pytest.mark.gpu


def _append_gpu(kp, vp, table, k_new, v_new, bidx, pos, ps):
    kp, vp = gpu(kp), gpu(vp)
    err = new_dev_err()
    binding.pkv_append(kp, vp, gpu(table), gpu(k_new), gpu(v_new), gpu(bidx), gpu(pos), ps,
                       dev_err=err)
    torch.cuda.synchronize()
    return bf16_bits(kp.cpu()), bf16_bits(vp.cpu()), int(err.item())


@pytest.mark.parametrize("maker", [W.tiny_decode, W.qwen3_b64_decode, W.padded_bucket_decode])
def test_decode_append_bit_exact(maker):
    c = maker(0)
    kb, vb, err = _append_gpu(c.k_pool, c.v_pool, c.page_table, c.k_new, c.v_new,
                              c.batch_idx, c.input_pos, c.page_size)
    ek, ev, bad = orc.append(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                             bf16_bits(c.k_new), bf16_bits(c.v_new), c.batch_idx.numpy(),
                             c.input_pos.numpy(), c.page_size)
    assert not bad and err == 0
    assert np.array_equal(kb, ek) and np.array_equal(vb, ev)


def test_prefill_append_full_size_bit_exact():
    """The packed prefill tokens (64 documents, lengths 64..1024) appended
    into page_size-128 pools."""
    c = W.packed_prefill(0)
    kb, vb, err = _append_gpu(c.k_pool, c.v_pool, c.page_table, c.k, c.v, c.batch_idx,
                              c.input_pos, c.page_size)
    ek, ev, bad = orc.append(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                             bf16_bits(c.k), bf16_bits(c.v), c.batch_idx.numpy(),
                             c.input_pos.numpy(), c.page_size)
    assert not bad and err == 0
    assert np.array_equal(kb, ek) and np.array_equal(vb, ev)


def test_bad_entries_flagged_and_skipped():
    gen = torch.Generator().manual_seed(3)
    ps, P, hkv, maxb, nb = 16, 40, 2, 6, 4
    kp = torch.randn((P * ps, hkv, 128), generator=gen).to(torch.bfloat16)
    vp = torch.randn((P * ps, hkv, 128), generator=gen).to(torch.bfloat16)
    table = torch.full((maxb, nb), -1, dtype=torch.int32)
    table[1:, :3] = (torch.randperm(P - 1, generator=gen)[:15] + 1).view(5, 3).int()
    table[0, :] = 0
    table[2, 1] = -1          # unreserved inside a sequence
    table[3, 0] = P + 7       # past the pool
    bidx = torch.tensor([1, 2, 2, 3, 0, 4, 9, 5, -1, 1], dtype=torch.int32)
    pos = torch.tensor([0, 5, 20, 1, 3, 47, 0, 2 * ps + 3, 0, nb * ps], dtype=torch.int32)
    N = len(bidx)
    k_new = torch.randn((N, hkv, 128), generator=gen).to(torch.bfloat16)
    v_new = torch.randn((N, hkv, 128), generator=gen).to(torch.bfloat16)
    kb, vb, err = _append_gpu(kp, vp, table, k_new, v_new, bidx, pos, ps)
    ek, ev, bad = orc.append(bf16_bits(kp), bf16_bits(vp), table.numpy(), bf16_bits(k_new),
                             bf16_bits(v_new), bidx.numpy(), pos.numpy(), ps)
    assert sorted(bad) == [2, 3, 6, 8, 9]
    assert np.array_equal(kb, ek) and np.array_equal(vb, ev)
    assert err & binding.DEV_ERR_BAD_PAGE
    assert err & binding.DEV_ERR_BAD_SLOT
    assert err & binding.DEV_ERR_BAD_POS


def test_empty_append_is_a_no_op():
    c = W.tiny_decode(0)
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    empty_i = torch.zeros(0, dtype=torch.int32, device="cuda")
    empty_kv = torch.zeros((0, c.num_kv_heads, 128), dtype=torch.bfloat16, device="cuda")
    binding.pkv_append(kp, vp, gpu(c.page_table), empty_kv, empty_kv, empty_i, empty_i,
                       c.page_size)
    torch.cuda.synchronize()
    assert torch.equal(kp.cpu(), c.k_pool) and torch.equal(vp.cpu(), c.v_pool)
