"""The decode workloads at full size, every (sequence, KV head) pair against the oracle.

The 8K workload (32 x 8193 tokens, 64 q / 8 KV heads) runs through the call
the benchmark times, nvfp4kv_append_decode_attention (append of the 32 new
tokens, then the decode with its split-K combine), in the benchmark's launch
configuration; the 128K workload (4 x 131072 tokens, calibrated global
scales) through nvfp4kv_decode_attention.  At full size the stream-K split
cuts pairs at places the scaled-down tests never reach, so every pair's
output is compared with the oracle's fp64 decode (per row, max |out - ref| <=
2e-3 * ||ref||), and the whole cache pool with the oracle's, byte for byte.
The oracle runs in spawned host processes, one sequence each.
"""
import os

import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import (bf16_dev, check_rows, dev, fill_workload_oracle, gpu_append, gpu_cache, gpu_global_scales,
                      oracle_global_scales, pool_host, status_word)
from oracle_workers import oracle_workload

pytestmark = pytest.mark.gpu

PROCS = max(1, min(32, os.cpu_count() or 1))


def _compare_pools(g, o):
    for got, want in zip(pool_host(g), (o.k_data, o.v_data, o.k_scale, o.v_scale)):
        assert np.array_equal(got, want)


def _compare_every_pair(wl, out, refs):
    G = wl.num_q_heads // wl.num_kv_heads
    worst = 0.0
    for b in range(wl.batch):
        for h in range(wl.num_kv_heads):
            worst = max(worst, check_rows(out[b, h * G:(h + 1) * G], refs[b][h]))
    return worst


def test_full_size_8k_step_every_pair(cuda_lib):
    wl = inputs.decode_config(2)
    prompts = wl.all_prompt_kv(threads=16)
    new = wl.new_kv()
    q = wl.q()
    # the cache before the step: the prompts only; the step appends the new tokens
    g = gpu_cache(wl.num_pages, wl.num_kv_heads)
    for b, (k, v) in enumerate(prompts):
        gpu_append(g, k, v, wl.slots(b, 0, k.shape[0]))
    ws = torch.zeros(kv.nvfp4kv_decode_workspace_size(g, wl.batch, wl.num_q_heads), dtype=torch.uint8, device="cuda")
    out = torch.full((wl.batch, wl.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = status_word()
    kv.nvfp4kv_append_decode_attention(g, bf16_dev(new[0]), bf16_dev(new[1]), dev(wl.append_slots()), bf16_dev(q),
                                       out, dev(wl.page_table), dev(wl.seq_lens.astype(np.int32)), wl.softmax_scale,
                                       ws, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _compare_pools(g, fill_workload_oracle(wl, prompts, new))
    del prompts
    refs = oracle_workload(2, 1.0, 1.0, range(wl.batch), PROCS)
    worst = _compare_every_pair(wl, out.cpu().numpy(), refs)
    print(f"\n8K step, all {wl.batch * wl.num_kv_heads} pairs: worst row error {worst:.2e} of the row norm")


def test_full_size_128k_every_pair(cuda_lib):
    wl = inputs.decode_config(3)
    prompts = wl.all_prompt_kv(threads=16)
    q = wl.q()
    gk, gv = gpu_global_scales(wl, prompts)
    ogk, ogv = oracle_global_scales(wl, prompts)
    assert (np.float32(gk), np.float32(gv)) == (np.float32(ogk), np.float32(ogv))   # calibration, bit for bit
    g = gpu_cache(wl.num_pages, wl.num_kv_heads, gk, gv)
    for b, (k, v) in enumerate(prompts):
        gpu_append(g, k, v, wl.slots(b, 0, k.shape[0]))
    ws = torch.zeros(kv.nvfp4kv_decode_workspace_size(g, wl.batch, wl.num_q_heads), dtype=torch.uint8, device="cuda")
    out = torch.full((wl.batch, wl.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = status_word()
    kv.nvfp4kv_decode_attention(g, bf16_dev(q), out, dev(wl.page_table), dev(wl.seq_lens.astype(np.int32)),
                                wl.softmax_scale, ws, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _compare_pools(g, fill_workload_oracle(wl, prompts))
    del prompts
    refs = oracle_workload(3, float(ogk), float(ogv), range(wl.batch), PROCS)
    worst = _compare_every_pair(wl, out.cpu().numpy(), refs)
    print(f"\n128K, all {wl.batch * wl.num_kv_heads} pairs: worst row error {worst:.2e} of the row norm")


def test_full_size_ragged_many_pairs(cuda_lib):
    # 256 sequences of 512..32768 tokens (+1), 32 q / 8 KV heads, fragmented
    # pool: every KV head of 48 sequences (the longest, the shortest and an
    # even spread) against the oracle; the cache is filled a sequence at a time
    wl = inputs.decode_config(4)
    order = np.argsort(wl.seq_lens)
    pick = sorted(set(order[:8].tolist() + order[-8:].tolist() + list(range(0, wl.batch, 8))))
    new = wl.new_kv()
    q = wl.q()
    g = gpu_cache(wl.num_pages, wl.num_kv_heads)
    from concurrent.futures import ThreadPoolExecutor

    with ThreadPoolExecutor(max_workers=16) as ex:          # drawn in threads, appended as they come
        for b, (k, v) in enumerate(ex.map(wl.prompt_kv, range(wl.batch))):
            gpu_append(g, k, v, wl.slots(b, 0, k.shape[0]))
    gpu_append(g, new[0], new[1], wl.append_slots())
    ws = torch.zeros(kv.nvfp4kv_decode_workspace_size(g, wl.batch, wl.num_q_heads), dtype=torch.uint8, device="cuda")
    out = torch.full((wl.batch, wl.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = status_word()
    kv.nvfp4kv_decode_attention(g, bf16_dev(q), out, dev(wl.page_table), dev(wl.seq_lens.astype(np.int32)),
                                wl.softmax_scale, ws, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert not torch.isnan(out).any()
    refs = oracle_workload(4, 1.0, 1.0, pick, PROCS)
    G = wl.num_q_heads // wl.num_kv_heads
    o = out.cpu().numpy()
    for b in pick:
        for h in range(wl.num_kv_heads):
            check_rows(o[b, h * G:(h + 1) * G], refs[b][h])
