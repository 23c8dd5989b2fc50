"""K2/K3 split-KV decode on the GPU against the float64 oracle, on the four
decode workloads at full size and on edge cases (tile edges, empty rows,
padding rows, NaN garbage in unused slots, bad entries, other GQA groups,
changing batch sizes in one process)."""

import ctypes

import numpy as np
import pytest
import torch

import oracle.paged_attention as orc
from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from paged_kv_gqa_pkv_gb300.workloads import bf16_bits
from tests.parity import (assert_attention_close, gpu, new_dev_err, oracle_decode_step,
                          run_decode_step)

pytestmark = pytest.mark.gpu


def _full_parity(case):
    kp, vp, out, lse, err = run_decode_step(case)
    ek, ev, ref_o, ref_l, bad_tok, bad_rows = oracle_decode_step(case)
    assert err == 0 and not bad_tok and not bad_rows
    assert np.array_equal(bf16_bits(kp), ek) and np.array_equal(bf16_bits(vp), ev)
    return assert_attention_close(out, lse, ref_o, ref_l, tag=case.name)


def test_tiny_decode():
    _full_parity(W.tiny_decode(0))


@pytest.mark.parametrize("permute", [False, True], ids=["sequential", "permuted"])
def test_qwen3_b64_decode(permute):
    _full_parity(W.qwen3_b64_decode(0, permute=permute))


def test_padded_bucket_decode():
    c = W.padded_bucket_decode(0)
    _, _, out, lse, err = run_decode_step(c)
    assert err == 0
    assert torch.all(out[40:] == 0) and torch.all(torch.isneginf(lse[40:]))
    _full_parity(c)


def test_long_context_b256_decode():
    _full_parity(W.long_context_decode(0))


def _permute_pages(case, seed):
    """Same logical content, pages moved by a random permutation."""
    P, ps = case.num_pages, case.page_size
    rng = np.random.default_rng(seed)
    sigma = np.concatenate([[0], rng.permutation(np.arange(1, P))])
    kp = torch.empty_like(case.k_pool)
    vp = torch.empty_like(case.v_pool)
    for p in range(P):
        kp[sigma[p] * ps:(sigma[p] + 1) * ps] = case.k_pool[p * ps:(p + 1) * ps]
        vp[sigma[p] * ps:(sigma[p] + 1) * ps] = case.v_pool[p * ps:(p + 1) * ps]
    t = case.page_table.numpy()
    t2 = np.where(t >= 0, sigma[np.maximum(t, 0)], -1).astype(np.int32)
    import copy
    c2 = copy.copy(case)
    c2.k_pool, c2.v_pool, c2.page_table = kp, vp, torch.from_numpy(t2)
    return c2


def test_contiguous_fast_path_bitwise_equals_general_path():
    seq = W.qwen3_b64_decode(0, permute=False)
    perm = _permute_pages(seq, 1)
    _, _, o1, l1, e1 = run_decode_step(seq)
    _, _, o2, l2, e2 = run_decode_step(perm)
    assert e1 == 0 and e2 == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 4), (8, 2)])
def test_other_gqa_groups(hq, hkv):
    lens = [1, 15, 16, 17, 31, 32, 33, 100, 0, 257]
    c = W.custom_decode(5, lens, hq=hq, hkv=hkv, page_size=32, permute=True)
    # a live row with no keys has no position to append to: attend only
    kp, vp, out, lse, err = run_decode_step(c, append=False)
    _, _, ref_o, ref_l, _, bad_rows = oracle_decode_step(c, append=False)
    assert err == 0 and not bad_rows
    assert_attention_close(out, lse, ref_o, ref_l, tag=f"G={hq // hkv}")
    assert torch.all(out[8] == 0) and torch.all(torch.isneginf(lse[8]))


def test_single_key_returns_its_value_row():
    c = W.custom_decode(7, [1, 1, 1], hq=32, hkv=8, page_size=128)
    kp, vp, out, lse, err = run_decode_step(c)
    g = 4
    for b in range(3):
        for h in range(32):
            assert torch.equal(out[b, h], c.v_new[b, h // g])


def test_unused_slots_hold_nan_garbage():
    """Slots past each sequence's length (inside its last page) hold NaN; the
    kernel must never let them into a result."""
    c = W.custom_decode(9, [5, 17, 130, 40], hq=32, hkv=8, page_size=128, fill=float("nan"))
    gen = torch.Generator().manual_seed(2)
    for s, n in enumerate(c.seq_lens.tolist(), start=1):
        for t in range(n):
            row = int(c.page_table[s, t // 128]) * 128 + t % 128
            c.k_pool[row] = torch.randn((8, 128), generator=gen).to(torch.bfloat16)
            c.v_pool[row] = torch.randn((8, 128), generator=gen).to(torch.bfloat16)
    _full_parity(c)


def test_bad_page_entry_flagged_other_rows_exact():
    c = W.custom_decode(11, [40, 300, 90], hq=32, hkv=8, page_size=128, permute=True)
    c.page_table[2, 1] = -1
    kp, vp, out, lse, err = run_decode_step(c, append=False)
    assert err & binding.DEV_ERR_BAD_PAGE
    _, _, ref_o, ref_l, _, bad_rows = oracle_decode_step(c, append=False)
    assert bad_rows == [1]
    assert_attention_close(out, lse, ref_o, ref_l, rows=[0, 2])


def test_bad_slot_and_overlong_rows_give_zero():
    c = W.custom_decode(13, [40, 70, 90], hq=32, hkv=8, page_size=128, permute=True)
    c.batch_idx[0] = 77                      # slot past the table
    c.seq_lens[1] = c.max_blocks * 128 + 1   # longer than the table allows
    _, _, out, lse, err = run_decode_step(c, append=False)
    assert err & binding.DEV_ERR_BAD_SLOT and err & binding.DEV_ERR_BAD_POS
    assert torch.all(out[:2] == 0) and torch.all(torch.isneginf(lse[:2]))
    _, _, ref_o, ref_l, _, _ = oracle_decode_step(c, append=False, rows=[2])
    assert_attention_close(out, lse, ref_o, ref_l, rows=[2])


def test_changing_batch_sizes_in_one_process():
    """One library, many shapes: no per-shape state may leak between calls."""
    for B in (1, 64, 3, 200, 2):
        lens = torch.randint(1, 700, (B,), generator=torch.Generator().manual_seed(B)).tolist()
        c = W.custom_decode(B, lens, hq=32, hkv=8, page_size=128, permute=True)
        _full_parity(c)


def test_decode_rejects_bad_host_arguments():
    c = W.tiny_decode(0)
    kp, vp, table = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    q, bidx, lens = gpu(c.q), gpu(c.batch_idx), gpu(c.seq_lens)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.PkvError) as e:
        binding.pkv_decode_attention(kp, vp, table, q, bidx, lens, c.page_size, c.scale,
                                     workspace=small)
    assert e.value.status == 4
    with pytest.raises(binding.PkvError) as e:   # page size not a multiple of 16
        binding.pkv_decode_attention(kp, vp, table, q, bidx, lens, 8, c.scale)
    assert e.value.status == 1
    q_off = torch.empty(q.numel() + 4, dtype=torch.bfloat16, device="cuda")[4:].view(q.shape)
    with pytest.raises(binding.PkvError) as e:   # 16-byte misaligned q
        binding.pkv_decode_attention(kp, vp, table, q_off, bidx, lens, c.page_size, c.scale)
    assert e.value.status == 2
    q6 = torch.zeros((4, 6, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.PkvError) as e:   # group 3 unsupported
        binding.pkv_decode_attention(kp, vp, table, q6, bidx, lens, c.page_size, c.scale)
    assert e.value.status == 1


def _decode_with(case, ws, err):
    kp, vp, table = gpu(case.k_pool), gpu(case.v_pool), gpu(case.page_table)
    return binding.pkv_decode_attention(kp, vp, table, gpu(case.q), gpu(case.batch_idx),
                                        gpu(case.seq_lens), case.page_size, case.scale,
                                        workspace=ws, dev_err=err)


def test_one_workspace_serves_every_shape():
    """One workspace (uninitialised) across batch sizes, GQA groups and KV-head
    counts: nothing of a call's scratch may leak into the next."""
    shapes = [(64, 32, 8, 600), (3, 32, 8, 9000), (200, 8, 8, 300), (1, 16, 2, 5000),
              (17, 64, 8, 1200), (64, 32, 8, 600)]
    cases = []
    for i, (B, hq, hkv, lmax) in enumerate(shapes):
        lens = torch.randint(1, lmax, (B,), generator=torch.Generator().manual_seed(i)).tolist()
        cases.append(W.custom_decode(40 + i, lens, hq=hq, hkv=hkv, page_size=128, permute=True))
    need = max(binding.pkv_decode_workspace_size(gpu(c.k_pool), gpu(c.page_table), 128,
                                                 c.batch, c.num_q_heads) for c in cases)
    ws = torch.full((need,), 0x7f, dtype=torch.uint8, device="cuda")
    for c in cases:
        err = new_dev_err()
        out, lse = _decode_with(c, ws, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _, _, ref_o, ref_l, _, _ = oracle_decode_step(c, append=False)
        assert_attention_close(out.cpu(), lse.cpu(), ref_o, ref_l, tag=c.name)


def test_single_long_row_merges_many_segments():
    """One 8192-key row: each item is cut into ~128 segments, more than one
    merge pass of 32 lanes."""
    c = W.custom_decode(21, [8192], hq=32, hkv=8, page_size=128, permute=True)
    _full_parity(c)


def test_short_rows_finish_whole_items_in_one_worker():
    """512 rows of 1..40 keys: most items fall inside one worker's range and
    are normalised without a partial."""
    lens = torch.randint(1, 41, (512,), generator=torch.Generator().manual_seed(5)).tolist()
    c = W.custom_decode(23, lens, hq=32, hkv=8, page_size=16, permute=True)
    _full_parity(c)



@pytest.mark.parametrize("lens,hq,hkv,ps", [([5000, 12, 7000], 32, 8, 128),
                                            ([9000, 8191], 8, 2, 64),
                                            ([20000], 32, 8, 16)],
                         ids=["b3_h8", "b2_g4_h2", "b1_20k_ps16"])
def test_long_rows_small_batch_combined_per_cta(lens, hq, hkv, ps):
    """Few rows with many keys: items are split over dozens of warps, and the
    CTAs combine their parts before the merge (the launch picks that path
    for small batch x kv heads)."""
    c = W.custom_decode(29, lens, hq=hq, hkv=hkv, page_size=ps, permute=True)
    _full_parity(c)


@pytest.mark.parametrize("ps,permute", [(48, True), (48, False), (80, True), (256, True),
                                        (256, False)],
                         ids=["ps48_perm", "ps48_seq", "ps80_perm", "ps256_perm", "ps256_seq"])
def test_page_sizes_that_are_not_powers_of_two_or_above_a_tile_row(ps, permute):
    """Any multiple of 16 is a valid page size: lengths on both sides of tile
    (16) and page edges, over permuted pages (table walk) and sequential ones
    (contiguous fast path)."""
    lens = [1, 15, 16, 17, ps - 1, ps, ps + 1, 2 * ps + 16, 3 * ps + 5, 700]
    c = W.custom_decode(31, lens, hq=32, hkv=8, page_size=ps, permute=permute)
    _full_parity(c)


@pytest.mark.parametrize("fill", ["random", "ones", "zeros"])
def test_workspace_needs_no_initialisation(fill):
    """The decode workspace's contents need no initialisation: whatever bits
    it starts with, and however often it is reused (eager calls, and replays
    of captured back-to-back calls), every call matches the oracle and every
    result is bit-identical to the first."""
    c = W.qwen3_b64_decode(3, permute=True)
    kp, vp, table = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    q, bi, sl = gpu(c.q), gpu(c.batch_idx), gpu(c.seq_lens)
    need = binding.pkv_decode_workspace_size(kp, table, c.page_size, c.batch, c.num_q_heads)
    if fill == "random":
        g = torch.Generator(device="cuda").manual_seed(9)
        ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda", generator=g)
    else:
        ws = torch.full((need,), 0xFF if fill == "ones" else 0, dtype=torch.uint8, device="cuda")
    err = new_dev_err()
    out = torch.empty((c.batch, c.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((c.batch, c.num_q_heads), dtype=torch.float32, device="cuda")

    def call():
        binding.pkv_decode_attention(kp, vp, table, q, bi, sl, c.page_size, c.scale, out=out,
                                     lse=lse, workspace=ws, dev_err=err)

    _, _, ref_o, ref_l, _, _ = oracle_decode_step(c, append=False)
    call()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out.cpu(), lse.cpu(), ref_o, ref_l, tag=f"{c.name}-{fill}")
    o0, l0 = out.clone(), lse.clone()
    for _ in range(2):  # eager calls on the same workspace
        out.zero_()
        call()
        torch.cuda.synchronize()
        assert torch.equal(out, o0) and torch.equal(lse, l0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()
        s.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for _ in range(3):  # back-to-back calls on one workspace
                call()
    torch.cuda.synchronize()
    for _ in range(3):  # replays of the captured calls
        out.zero_()
        lse.zero_()
        gr.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, o0) and torch.equal(lse, l0)
    assert int(err.item()) == 0
    del gr  # release the graph's memory pool now, not at some later collection
    torch.cuda.synchronize()


def _pinned(t):
    return t.contiguous().pin_memory()


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 8), (32, 4)])
def test_host_resident_inputs_give_the_same_bits(hq, hkv):
    """q, batch_idx and seq_lens in pinned host memory (the kernels read them
    over the host link; q's rows by cp.async) give the bits the same call
    gives on device copies, for GQA groups 1, 4 and 8."""
    lens = torch.randint(1, 3000, (33,), generator=torch.Generator().manual_seed(hq + hkv)).tolist()
    lens[3] = 0
    c = W.custom_decode(60 + hq, lens, hq=hq, hkv=hkv, page_size=128, permute=True, n_pad=3)
    kp, vp, table = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    err = new_dev_err()
    o_dev, l_dev = binding.pkv_decode_attention(kp, vp, table, gpu(c.q), gpu(c.batch_idx),
                                                gpu(c.seq_lens), c.page_size, c.scale,
                                                dev_err=err)
    o_host, l_host = binding.pkv_decode_attention(kp, vp, table, _pinned(c.q),
                                                  _pinned(c.batch_idx), _pinned(c.seq_lens),
                                                  c.page_size, c.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o_host, o_dev) and torch.equal(l_host, l_dev)
    _, _, ref_o, ref_l, _, _ = oracle_decode_step(c, append=False)
    assert_attention_close(o_host.cpu(), l_host.cpu(), ref_o, ref_l, tag="host inputs")


def test_host_resident_inputs_fused_step_and_graph_replay():
    """The fused append + decode with q, k_new, v_new, batch_idx and
    seq_lens in pinned host memory and out/lse written to pinned host memory:
    the pools and results equal those of the same step on device inputs, and
    a captured step replayed after the host rewrote its inputs in place gives
    the new step's bits."""
    c = W.qwen3_b64_decode(4, permute=True)
    c2 = W.qwen3_b64_decode(5, permute=True)  # other q / k_new / v_new, same lengths
    kp_d, vp_d = gpu(c.k_pool), gpu(c.v_pool)
    kp_h, vp_h = gpu(c.k_pool), gpu(c.v_pool)
    table = gpu(c.page_table)
    err = new_dev_err()
    o_d, l_d = binding.pkv_decode_append_attention(
        kp_d, vp_d, table, gpu(c.q), gpu(c.k_new), gpu(c.v_new), gpu(c.batch_idx),
        gpu(c.seq_lens), c.page_size, c.scale, dev_err=err)
    hq_, hk, hv = _pinned(c.q), _pinned(c.k_new), _pinned(c.v_new)
    hb, hs = _pinned(c.batch_idx), _pinned(c.seq_lens)
    out_h = torch.empty((c.batch, c.num_q_heads, 128), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((c.batch, c.num_q_heads), dtype=torch.float32).pin_memory()
    binding.pkv_decode_append_attention(kp_h, vp_h, table, hq_, hk, hv, hb, hs, c.page_size,
                                        c.scale, out=out_h, lse=lse_h, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(kp_h, kp_d) and torch.equal(vp_h, vp_d)
    assert torch.equal(out_h, o_d.cpu()) and torch.equal(lse_h, l_d.cpu())
    # capture the host-input step, then rewrite the inputs in place and replay
    ws = torch.empty(binding.pkv_decode_workspace_size(kp_h, table, c.page_size, c.batch,
                                                       c.num_q_heads),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def step():
        binding.pkv_decode_append_attention(kp_h, vp_h, table, hq_, hk, hv, hb, hs,
                                            c.page_size, c.scale, out=out_h, lse=lse_h,
                                            workspace=ws, dev_err=err)

    with torch.cuda.stream(s):
        step()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.synchronize()
    hq_.copy_(c2.q)
    hk.copy_(c2.k_new)
    hv.copy_(c2.v_new)
    kp2, vp2 = gpu(c.k_pool), gpu(c.v_pool)
    o2, l2 = binding.pkv_decode_append_attention(
        kp2, vp2, table, gpu(c2.q), gpu(c2.k_new), gpu(c2.v_new), gpu(c.batch_idx),
        gpu(c.seq_lens), c.page_size, c.scale, dev_err=err)
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(kp_h, kp2) and torch.equal(vp_h, vp2)
    assert torch.equal(out_h, o2.cpu()) and torch.equal(lse_h, l2.cpu())
    del g


def test_pageable_host_q_is_rejected():
    """q in pageable host memory, which the GPU cannot read, is refused at the
    C boundary (PKV_ERR_ARG) before any launch."""
    c = W.tiny_decode(0)
    kp, vp, table = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    q_pageable = c.q.clone()  # not pinned
    lib = binding.load_library()
    desc = binding.cache_desc(kp, table, c.page_size)
    need = lib.pkv_decode_workspace_size(ctypes.byref(desc), c.batch, c.num_q_heads, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty((c.batch, c.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((c.batch, c.num_q_heads), dtype=torch.float32, device="cuda")
    bi, sl = gpu(c.batch_idx), gpu(c.seq_lens)
    st = lib.pkv_decode_attention(
        ctypes.byref(desc), ctypes.c_void_p(kp.data_ptr()), ctypes.c_void_p(vp.data_ptr()),
        ctypes.c_void_p(table.data_ptr()), ctypes.c_void_p(q_pageable.data_ptr()),
        c.num_q_heads, ctypes.c_void_p(bi.data_ptr()), ctypes.c_void_p(sl.data_ptr()), c.batch,
        ctypes.c_float(c.scale), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(need), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 1  # PKV_ERR_ARG
    with pytest.raises(ValueError):
        binding.pkv_decode_attention(kp, vp, table, q_pageable, bi, sl, c.page_size, c.scale)


def test_batches_above_512_rows_run_as_equal_launches():
    """1100 rows (five of them padding) run as three launches of at most 367
    rows over one workspace, whose size is that of one launch: every row
    against the oracle, and the same bits with q, batch_idx and seq_lens in
    pinned host memory (each launch reads its rows at an offset there)."""
    lens = torch.randint(1, 200, (1095,), generator=torch.Generator().manual_seed(11)).tolist()
    c = W.custom_decode(11, lens, hq=32, hkv=8, page_size=16, permute=True, n_pad=5)
    assert c.batch == 1100
    kp, vp, table = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    size = lambda b: binding.pkv_decode_workspace_size(kp, table, c.page_size, b, c.num_q_heads)
    assert size(1100) == size(367) < size(512)
    assert size(1536) == size(512)
    _, _, o_dev, l_dev, err = run_decode_step(c, append=False)
    assert err == 0
    _, _, ref_o, ref_l, _, bad_rows = oracle_decode_step(c, append=False)
    assert not bad_rows
    assert_attention_close(o_dev, l_dev, ref_o, ref_l, tag="1100 rows")
    e2 = new_dev_err()
    o_host, l_host = binding.pkv_decode_attention(kp, vp, table, _pinned(c.q),
                                                  _pinned(c.batch_idx), _pinned(c.seq_lens),
                                                  c.page_size, c.scale, dev_err=e2)
    torch.cuda.synchronize()
    assert int(e2.item()) == 0
    assert torch.equal(o_host.cpu(), o_dev) and torch.equal(l_host.cpu(), l_dev)
