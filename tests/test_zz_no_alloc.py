"""nvfp4kv_decode_attention_static: decode for callers that cannot allocate.

Some callers cannot hand the decode a device workspace: they run inside an
allocator hook, or they are plug-ins whose host runtime owns all device memory.
For them the library keeps a fixed 32 MiB scratch array in its device image
and nvfp4kv_decode_attention_static uses it instead.

The static entry point runs the same kernels, on the same split of the work,
as nvfp4kv_decode_attention with a caller workspace, so its output must equal
that call's bit for bit; one call is also checked against the oracle.  Between
the two calls on the target workload the static entry point decodes another
workload, whose (sequence, KV head) pairs are cut at other places, so the
second call finds the scratch full of someone else's split records and
page prefixes.  This file is named to run last: the scratch is process-wide state.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import (ATTN_TOL, bf16_dev, check_rows, decode_gpu, dev, fill_workload_gpu, fill_workload_oracle,
                      status_word)

pytestmark = pytest.mark.gpu


def _static(lib, cache, q_dev, out, pt_dev, lens_dev, B, Hq, scale, status):
    c = cache.c_struct()
    return lib.nvfp4kv_decode_attention_static(
        ctypes.byref(c), q_dev.data_ptr(), out.data_ptr(), pt_dev.data_ptr(), int(pt_dev.shape[1]),
        lens_dev.data_ptr(), B, Hq, float(scale), status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _static_decode(lib, wl, cache, q_bits):
    """One static-entry decode of workload wl; returns the fp32 output (device)."""
    out = torch.full((wl.batch, wl.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    status = status_word()
    rc = _static(lib, cache, bf16_dev(q_bits), out, dev(wl.page_table), dev(wl.seq_lens.astype(np.int32)),
                 wl.batch, wl.num_q_heads, wl.softmax_scale, status)
    assert rc == kv.NVFP4KV_OK, kv.nvfp4kv_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


def _other_workload():
    """Ragged lengths, another GQA shape: cut points unlike the target's."""
    rng = np.random.default_rng(77)
    lens = np.array(list(rng.integers(1, 3000, 37)) + [9000], np.int64)
    return inputs.DecodeWorkload("custom", 77, lens, True, 16, 4, inputs.KVDist("normal", 1.0), pool_factor=1.1)


@pytest.mark.parametrize("index,scale", [(1, 1.0), (4, 1 / 16), (2, 1 / 8)])
def test_static_scratch_equals_workspace_decode_bit_for_bit(cuda_lib, index, scale):
    lib = kv.load()
    wl = inputs.decode_config(index, scale)
    prompts = wl.all_prompt_kv()
    new = wl.new_kv() if wl.append else None
    cache = fill_workload_gpu(wl, prompts, new)
    q = wl.q()
    ref, _ = decode_gpu(wl, cache, q)                     # ordinary entry point, caller workspace
    torch.cuda.synchronize()

    first = _static_decode(lib, wl, cache, q)
    assert torch.equal(first, ref)
    o = fill_workload_oracle(wl, prompts, new)
    exp, rs = oracle.decode_attention(o, q, wl.page_table, wl.seq_lens, wl.softmax_scale)
    assert rs == 0
    check_rows(first.cpu().numpy(), exp, tol=ATTN_TOL)

    other = _other_workload()
    oc = fill_workload_gpu(other, other.all_prompt_kv(), other.new_kv())
    oq = other.q()
    other_out = _static_decode(lib, other, oc, oq)
    other_ref, _ = decode_gpu(other, oc, oq)
    assert torch.equal(other_out, other_ref)

    second = _static_decode(lib, wl, cache, q)
    assert torch.equal(second, ref)


def test_static_scratch_rejects_a_batch_that_does_not_fit(cuda_lib):
    lib = kv.load()
    cache = kv.Cache.empty(4, 1, zero=True)
    Hq = 1
    # the scratch holds the split records and one page-prefix word per sequence:
    # the smallest batch past 32 MiB
    B = 1
    while kv.nvfp4kv_decode_workspace_size(cache, B, Hq) <= (32 << 20):
        B *= 2
    lo = B // 2
    while lo + 1 < B:
        mid = (lo + B) // 2
        if kv.nvfp4kv_decode_workspace_size(cache, mid, Hq) <= (32 << 20):
            lo = mid
        else:
            B = mid
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    pt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    status = status_word()
    rc = _static(lib, cache, q, out, pt, lens, B, Hq, 0.1, status)
    assert rc == kv.NVFP4KV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not out.any()             # nothing was enqueued
