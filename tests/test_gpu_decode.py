"""GPU paged decode attention (fused NVFP4 dequant) vs the oracle's fp64 attention.

Decode dequantises inside the attention kernel ("nvfp4-kv-cache-memory-wall",
section 3, item 3).  Bar: per (sequence, query head) row,
max_d |out - ref| <= 2e-3 * ||ref||_2 (gpu_util.ATTN_TOL).
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import (bf16_dev, check_rows, decode_gpu, dev, fill_workload_gpu, fill_workload_oracle, gpu_append,
                      gpu_cache, gpu_global_scales, pool_host, status_word)

pytestmark = pytest.mark.gpu


def _full_compare(wl):
    prompts = wl.all_prompt_kv()
    new = wl.new_kv() if wl.append else None
    q = wl.q()
    g = fill_workload_gpu(wl, prompts, new)
    st = status_word()
    out, ws = decode_gpu(wl, g, q, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o = fill_workload_oracle(wl, prompts, new)
    ref, rs = oracle.decode_attention(o, q, wl.page_table, wl.seq_lens, wl.softmax_scale)
    assert rs == 0
    worst = check_rows(out.cpu().numpy(), ref)
    # the workspace is scratch that needs no initialisation: filled with
    # garbage, a second call gives the same bits
    ws.fill_(0xA5)
    out2, _ = decode_gpu(wl, g, q, workspace=ws)
    assert torch.equal(out, out2)
    return worst


def test_tiny_workload(cuda_lib):
    _full_compare(inputs.decode_config(1))


@pytest.mark.parametrize("index,scale", [(2, 1 / 32), (3, 1 / 256), (4, 1 / 32)])
def test_scaled_workloads(cuda_lib, index, scale):
    _full_compare(inputs.decode_config(index, scale))


def _custom(lens, hq, hkv, seed=0, dist=None, pool_factor=1.0, append=False):
    dist = dist or inputs.KVDist("normal", 1.0)
    return inputs.DecodeWorkload("custom", seed, np.array(lens, np.int64), append, hq, hkv, dist,
                                 pool_factor=pool_factor)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (4, 2), (16, 4), (64, 8), (24, 8)])
def test_group_sizes(cuda_lib, hq, hkv):
    _full_compare(_custom([1, 15, 16, 17, 33, 200], hq, hkv, seed=hq))


def test_ragged_tails_empty_and_many_tiny_sequences(cuda_lib):
    rng = np.random.default_rng(9)
    lens = list(rng.integers(0, 40, 300)) + [0, 1, 2, 16, 4096]
    _full_compare(_custom(lens, 32, 8, seed=5, pool_factor=1.3))


@pytest.mark.parametrize("batch", [1024, 1025, 3000])
def test_batches_past_the_combines_length_scan(cuda_lib, batch):
    # up to 1024 sequences the combine works out where a cut pair's records
    # are from the lengths; past that, from the page prefix the decode wrote
    rng = np.random.default_rng(batch)
    lens = list(rng.integers(0, 120, batch - 2)) + [3000, 0]
    _full_compare(_custom(lens, 4, 2, seed=batch, pool_factor=1.2))


def test_long_single_sequence_across_many_ctas(cuda_lib):
    _full_compare(_custom([65536 + 7], 8, 1, seed=11, append=True,
                          dist=inputs.KVDist("normal", 0.02, outlier=6.0, per_chunk=8)))


def test_large_scores_and_calibrated_scales(cuda_lib):
    wl = _custom([300, 1000], 16, 2, seed=12, dist=inputs.KVDist("channel", lo=0.1, hi=10.0))
    wl.q_sigma = 30.0           # sharp softmax: exercises the running-max rescale
    wl.calibrated = True
    _full_compare(wl)


def test_bad_page_ids_and_lengths_are_flagged_and_skipped(cuda_lib):
    wl = _custom([40, 70], 8, 2, seed=13)
    prompts = wl.all_prompt_kv()
    q = wl.q()
    g = fill_workload_gpu(wl, prompts)
    o = fill_workload_oracle(wl, prompts)
    pt = wl.page_table.copy()
    pt[1, 2] = wl.num_pages + 100          # sequence 1, tokens 32..47 -> skipped
    st = status_word()
    B, Hq = wl.batch, wl.num_q_heads
    ws = torch.zeros(kv.nvfp4kv_decode_workspace_size(g, B, Hq), dtype=torch.uint8, device="cuda")
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    from gpu_util import bf16_dev
    kv.nvfp4kv_decode_attention(g, bf16_dev(q), out, dev(pt), dev(wl.seq_lens), wl.softmax_scale, ws,
                                device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kv.NVFP4KV_DEVERR_PAGE
    ref, rs = oracle.decode_attention(o, q, pt, wl.seq_lens, wl.softmax_scale)
    assert rs == 1
    check_rows(out.cpu().numpy(), ref)
    # a length past the page table is clamped and flagged
    lens = wl.seq_lens.copy()
    lens[0] = wl.max_pages * 16 + 5
    st.zero_()
    kv.nvfp4kv_decode_attention(g, bf16_dev(q), out, dev(wl.page_table), dev(lens), wl.softmax_scale, ws,
                                device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kv.NVFP4KV_DEVERR_LENGTH


@pytest.mark.parametrize("index,scale", [(1, 1.0), (2, 1 / 32), (4, 1 / 32), (3, 1 / 256)])
def test_fused_append_decode_matches_two_calls(cuda_lib, index, scale):
    # nvfp4kv_append_decode_attention gives exactly the bits of
    # nvfp4kv_quantize_append followed by nvfp4kv_decode_attention
    wl = inputs.decode_config(index, scale)
    prompts = wl.all_prompt_kv()
    new = wl.new_kv() if wl.append else None
    q = wl.q()
    gk, gv = gpu_global_scales(wl, prompts, new)

    def prompts_only():                         # the step itself appends the new token
        c = gpu_cache(wl.num_pages, wl.num_kv_heads, gk, gv)
        for bb in range(wl.batch):
            kk, vv = prompts[bb]
            if kk.shape[0]:
                gpu_append(c, kk, vv, wl.slots(bb, 0, kk.shape[0]))
        return c

    a = prompts_only()
    b = prompts_only()
    if new is not None:
        slots = dev(wl.append_slots())
        k, v = bf16_dev(new[0]), bf16_dev(new[1])
    else:
        slots = dev(np.zeros(0, np.int64))
        k = v = bf16_dev(np.zeros((0, wl.num_kv_heads, 128), np.uint16))
    qd, pt, lens = bf16_dev(q), dev(wl.page_table), dev(wl.seq_lens.astype(np.int32))
    n = kv.nvfp4kv_decode_workspace_size(a, wl.batch, wl.num_q_heads)
    ws_a = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ws_b = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out_a = torch.full((wl.batch, wl.num_q_heads, 128), float("nan"), device="cuda")
    out_b = torch.full_like(out_a, float("nan"))
    st = status_word()
    kv.nvfp4kv_append_decode_attention(a, k, v, slots, qd, out_a, pt, lens, wl.softmax_scale, ws_a,
                                       device_status=st)
    if new is not None:
        kv.nvfp4kv_quantize_append(b, k, v, slots)
    kv.nvfp4kv_decode_attention(b, qd, out_b, pt, lens, wl.softmax_scale, ws_b)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out_a, out_b)
    for x, y in zip(pool_host(a), pool_host(b)):
        np.testing.assert_array_equal(x, y)


def test_workspace_bytes_from_the_batch_shape_covers_the_call(cuda_lib):
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    for B, hq, hkv in ((32, 64, 8), (256, 32, 8), (2, 8, 2), (7, 24, 8)):
        cache = kv.Cache.empty(4, hkv)
        need = kv.nvfp4kv_decode_workspace_size(cache, B, hq)
        assert kv.nvfp4kv_decode_workspace_bytes(B, hq, 8193, nsm) >= need
