"""Global-scale calibration on the GPU against the oracle, bit for bit.

"nvfp4-kv-cache-memory-wall", section 2: the FP32 per-tensor scale is 1 in the
uncalibrated public setting; a calibrated one maps the tensor's largest
magnitude onto E2M1 6 x E4M3 448.  nvfp4kv_tensor_amax is the device pass
(max |x| of a bf16 tensor), nvfp4kv_calibrated_global_scale the host division.
Inputs are finite: the pages define no NaN handling (the library propagates a
NaN, the oracle skips it).
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import (bf16_dev, fill_workload_gpu, fill_workload_oracle, gpu_global_scales, oracle_global_scales,
                      pool_host)

pytestmark = pytest.mark.gpu


def _amax_gpu(bits, start=None):
    """The library's amax of bf16 bit patterns; start: accumulate onto this value
    (else the output holds garbage that the call must overwrite)."""
    out = torch.full((1,), 123.0 if start is None else start, dtype=torch.float32, device="cuda")
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    x = bf16_dev(bits) if bits.size else torch.empty(0, dtype=torch.bfloat16, device="cuda")
    kv.nvfp4kv_tensor_amax(x, out, accumulate=start is not None)
    return out.cpu().numpy()[0]


def _same(a, b):
    return np.float32(a).tobytes() == np.float32(b).tobytes()


def _wide_range(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n) * 2.0 ** rng.integers(-140, 110, n)
    return inputs.bf16_bits(x.astype(np.float32))


# sizes around the 8-value vector, the 4-vector unroll of a thread, a block's
# 256 threads, and a grid-stride pass over every SM
@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 15, 16, 17, 31, 33, 255, 8191, 8192, 8193,
                               152 * 8 * 256 * 8 * 4 + 13, 3_000_001])
def test_amax_bit_exact(cuda_lib, n):
    bits = _wide_range(n, n)
    assert _same(_amax_gpu(bits), oracle.tensor_amax(bits))


@pytest.mark.parametrize("where", ["first", "in_vector", "last_vector", "tail", "last", "middle"])
def test_amax_wherever_the_largest_value_sits(cuda_lib, where):
    n = 100_003                                  # 12500 vectors and a 3-value tail
    rng = np.random.default_rng(11)
    bits = inputs.bf16_bits((rng.standard_normal(n) * 0.5).astype(np.float32))
    pos = {"first": 0, "in_vector": 8 * 777 + 5, "last_vector": 8 * 12499 + 7, "tail": n - 2, "last": n - 1,
           "middle": n // 2}[where]
    bits[pos] = inputs.bf16_bits(np.array([-37.25], np.float32))[0]
    got = _amax_gpu(bits)
    assert got == 37.25 and _same(got, oracle.tensor_amax(bits))


def test_amax_of_zeros_subnormals_and_infinities(cuda_lib):
    rng = np.random.default_rng(5)
    zeros = np.where(rng.random(1000) < 0.5, 0x8000, 0x0000).astype(np.uint16)
    assert _same(_amax_gpu(zeros), 0.0)                                   # +0, never -0
    sub = (rng.integers(1, 0x80, 5001) | (rng.integers(0, 2, 5001) << 15)).astype(np.uint16)
    assert _same(_amax_gpu(sub), oracle.tensor_amax(sub))
    assert _amax_gpu(sub) == inputs.bf16_bits_to_f32(np.array([(sub & 0x7FFF).max()], np.uint16))[0]
    inf = _wide_range(4099, 9)
    inf[4097] = 0xFF80                                                     # -inf
    assert _same(_amax_gpu(inf), oracle.tensor_amax(inf)) and np.isinf(_amax_gpu(inf))


def test_amax_accumulates(cuda_lib):
    bits = inputs.bf16_bits(np.array([1.0, -3.0, 2.5] * 700, np.float32))
    assert _amax_gpu(bits, start=5.0) == 5.0
    assert _amax_gpu(bits, start=0.0) == 3.0
    assert _amax_gpu(bits[:0], start=7.5) == 7.5                           # nothing to fold
    assert _amax_gpu(bits[:0]) == 0.0                                     # zeroed


def test_amax_on_a_slice(cuda_lib):
    # a tensor that starts 16 bytes into its allocation
    bits = _wide_range(4096 + 8, 21)
    x = bf16_dev(bits)[8:]
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    kv.nvfp4kv_tensor_amax(x, out)
    assert _same(out.item(), oracle.tensor_amax(bits[8:]))


def test_misaligned_slice_refused(cuda_lib):
    x = bf16_dev(_wide_range(64, 1))[1:]
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    with pytest.raises(kv.Nvfp4kvError):
        kv.nvfp4kv_tensor_amax(x, out)


@pytest.mark.parametrize("scale", [1 / 64, 1 / 8])
def test_calibrated_workload_scales_and_cache_bytes(cuda_lib, scale):
    # the long-context workload (per-channel magnitudes over two decades): the
    # library's scales equal the oracle's, and the caches both fill are equal
    wl = inputs.decode_config(3, scale)
    prompts = wl.all_prompt_kv()
    g = gpu_global_scales(wl, prompts)
    o = oracle_global_scales(wl, prompts)
    assert all(_same(a, b) for a, b in zip(g, o)) and g != (1.0, 1.0)
    gc = fill_workload_gpu(wl, prompts)
    oc = fill_workload_oracle(wl, prompts)
    for got, want in zip(pool_host(gc), (oc.k_data, oc.v_data, oc.k_scale, oc.v_scale)):
        assert np.array_equal(got, want)
    assert max(int(oc.k_scale.max()), int(oc.v_scale.max())) == 0x7E       # the amax block reaches 448
