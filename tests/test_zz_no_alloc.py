"""nvfp4kv_decode_attention_static: decode for callers that cannot allocate.

Some callers cannot hand the decode a device workspace: they run inside an
allocator hook, or they are plug-ins whose host runtime owns all device memory.
For them the library keeps a fixed 16 MiB scratch array in its device image
and nvfp4kv_decode_attention_static uses it instead.  These tests call the new
entry point through the C ABI and compare it with the ordinary entry point
(caller workspace) on the same cache, twice in a row, since the second call
finds the first call's leftovers in the shared scratch.  This file is named to
run last: the scratch is process-wide state.
"""
import ctypes

import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import ATTN_TOL, bf16_dev, check_rows, decode_gpu, dev, fill_workload_gpu, status_word

pytestmark = pytest.mark.gpu


def _static(lib, cache, q_dev, out, pt_dev, lens_dev, B, Hq, scale, status):
    c = cache.c_struct()
    return lib.nvfp4kv_decode_attention_static(
        ctypes.byref(c), q_dev.data_ptr(), out.data_ptr(), pt_dev.data_ptr(), int(pt_dev.shape[1]),
        lens_dev.data_ptr(), B, Hq, float(scale), status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("index,scale", [(1, 1.0), (4, 1 / 16), (2, 1 / 8)])
def test_static_scratch_matches_workspace_decode_twice(cuda_lib, index, scale):
    lib = kv.load()
    wl = inputs.decode_config(index, scale)
    prompts = wl.all_prompt_kv()
    new = wl.new_kv() if wl.append else None
    cache = fill_workload_gpu(wl, prompts, new)
    q = wl.q()
    ref, _ = decode_gpu(wl, cache, q)                     # ordinary entry point, caller workspace
    ref = ref.cpu().numpy().astype(np.float64)
    q_dev, pt_dev, lens_dev = bf16_dev(q), dev(wl.page_table), dev(wl.seq_lens.astype(np.int32))
    for call in range(2):
        out = torch.full((wl.batch, wl.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
        status = status_word()
        rc = _static(lib, cache, q_dev, out, pt_dev, lens_dev, wl.batch, wl.num_q_heads, wl.softmax_scale,
                     status)
        assert rc == kv.NVFP4KV_OK, kv.nvfp4kv_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        check_rows(out.cpu().numpy(), ref, tol=ATTN_TOL)


def test_static_scratch_rejects_a_batch_that_does_not_fit(cuda_lib):
    lib = kv.load()
    cache = kv.Cache.empty(4, 8, zero=True)
    Hq = 8
    B = 4096                         # grow the batch until its workspace exceeds the 16 MiB scratch
    while kv.nvfp4kv_decode_workspace_size(cache, B, Hq) <= (16 << 20):
        B *= 2
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    pt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    status = status_word()
    rc = _static(lib, cache, q, out, pt, lens, B, Hq, 0.1, status)
    assert rc == kv.NVFP4KV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not out.any()             # nothing was enqueued
