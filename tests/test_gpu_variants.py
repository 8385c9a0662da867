"""Quantize-append of the format variants on the GPU against the oracle, bit for bit.

"NVFP4: breaking the memory wall" (cloud.tencent.com): stochastic rounding and
a Hadamard rotation before quantisation; MXFP4's blocks of 32 ("NVIDIA NVFP4:
LLM memory doubled, inference 3x" (nmedialink), figure 6).  The oracle side
applies the oracle's per-block functions to every row at its slot.
"""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import bf16_dev, dev, status_word
from variant_util import oracle_variant_pools

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", [kv.NVFP4KV_VARIANT_SR, kv.NVFP4KV_VARIANT_HADAMARD, kv.NVFP4KV_VARIANT_MXFP4])
@pytest.mark.parametrize("gk,gv", [(1.0, 1.0), (0.37, 3e-3)])
def test_variant_quantize_bit_exact(cuda_lib, variant, gk, gv):
    rng = np.random.default_rng(40 + variant)
    n, H, pages = 77, 2, 8                                 # 308 rows: the last warp is partly past the end
    x = (rng.standard_normal((n, H, 128)) * 2.0 ** rng.integers(-12, 6, (n, H, 1))).astype(np.float32)
    x[3, 1, 7] = 6.0 * 448                                  # an outlier block
    x[4, 0, :] = 0.0                                       # a zero row (all blocks zero)
    k, v = inputs.bf16_bits(x), inputs.bf16_bits(-0.5 * x[::-1].copy())
    slots = rng.permutation(pages * 16)[:n].astype(np.int64)
    slots[::13] = -1
    slots[9] = pages * 16 + 1                               # outside the pool
    rk = inputs.rounding_bytes(2, n * H * 128).reshape(n, H, 128)
    rv = inputs.rounding_bytes(3, n * H * 128).reshape(n, H, 128)
    cache = kv.Cache.empty(pages, H, k_global_scale=gk, v_global_scale=gv, zero=True,
                           mxfp4=variant == kv.NVFP4KV_VARIANT_MXFP4)
    st = status_word()
    kv.nvfp4kv_quantize_append_variant(variant, cache, bf16_dev(k), bf16_dev(v), dev(slots), dev(rk), dev(rv),
                                       device_status=st)
    torch.cuda.synchronize()
    assert st.item() & kv.NVFP4KV_DEVERR_SLOT
    want = oracle_variant_pools(variant, k, v, slots, pages, H, np.float32(gk), np.float32(gv), rk, rv)
    rows = pages * H * 16
    for name, (data, scale) in want.items():
        gd = (cache.k_data if name == "k" else cache.v_data).reshape(rows, -1).cpu().numpy()
        gs = (cache.k_scale if name == "k" else cache.v_scale).reshape(rows, -1).cpu().numpy()
        assert np.array_equal(gd, data), f"{name} data"
        assert np.array_equal(gs, scale), f"{name} scales"


def test_variant_argument_checks(cuda_lib):
    cache = kv.Cache.empty(2, 1, zero=True)
    k = bf16_dev(inputs.bf16_bits(np.ones((2, 1, 128), np.float32)))
    with pytest.raises(kv.Nvfp4kvError):
        kv.nvfp4kv_quantize_append_variant(9, cache, k, k, dev(np.array([0, 1], np.int64)))
    with pytest.raises(kv.Nvfp4kvError):                   # stochastic rounding needs its random bytes
        kv.nvfp4kv_quantize_append_variant(kv.NVFP4KV_VARIANT_SR, cache, k, k, dev(np.array([0, 1], np.int64)))
