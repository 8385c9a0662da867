"""Oracle global-scale calibration: the per-tensor amax and g = amax / (6 * 448).

"nvfp4-kv-cache-memory-wall", section 2: the FP32 per-tensor scale is left at
1 in the uncalibrated public setting; a calibrated one maps the tensor's
largest magnitude onto the top of the two-level range (E2M1 6 times E4M3 448).
"""
import numpy as np
import pytest

import oracle
from nvfp4_quantized_paged_quantize_gb300 import inputs


def _bf16(x):
    return inputs.bf16_bits(np.asarray(x, np.float32))


@pytest.mark.parametrize("n", [0, 1, 7, 8, 1000, 65537])
def test_amax_matches_numpy(n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * 2.0 ** rng.integers(-140, 100, n)).astype(np.float32)
    bits = _bf16(x)
    ref = float(np.abs(inputs.bf16_bits_to_f32(bits)).max()) if n else 0.0
    assert oracle.tensor_amax(bits) == ref


def test_amax_of_negative_and_subnormal_values():
    bits = np.array([0x8001, 0x0003, 0x807F, 0x0000, 0x8000], np.uint16)  # bf16 subnormals, +-0
    assert oracle.tensor_amax(bits) == float(inputs.bf16_bits_to_f32(np.array([0x007F], np.uint16))[0])
    assert oracle.tensor_amax(_bf16([-3.5, 2.0, -0.0])) == 3.5


@pytest.mark.parametrize("amax", [2688.0, 1.0, 6.0, 0.06, 3.3e38, 1e-38])
def test_calibrated_scale_is_binary32_division(amax):
    a = np.float32(amax)
    assert oracle.calibrated_global_scale(float(a)) == float(a / np.float32(2688.0))
    assert oracle.calibrated_global_scale(0.0) == 1.0
    assert oracle.calibrated_global_scale(2688.0) == 1.0


@pytest.mark.parametrize("amax", [0.06, 6.0, 17.25, 3.0e5])
def test_calibrated_scale_maps_amax_to_top_of_range(amax):
    # the block holding the tensor's amax gets scale 448 and the amax code +-6
    rng = np.random.default_rng(3)
    x = (rng.uniform(-1, 1, 16) * amax * 0.5).astype(np.float32)
    x[5] = -amax
    x = inputs.bf16_bits_to_f32(_bf16(x))
    g = oracle.calibrated_global_scale(oracle.tensor_amax(_bf16(x)))
    packed, sb = oracle.quantize_block(x, g)
    assert sb == 0x7E and oracle.e4m3_value(sb) == 448.0
    assert (packed[2] >> 4) & 0xF == 0xF                             # element 5 (high nibble of byte 2): -6


def test_workload_generator_uses_the_calibrated_scale():
    # the long-context workload's global scales are this calibration of its K and V
    wl = inputs.decode_config(3, 1 / 1024)
    prompts = wl.all_prompt_kv()
    gk, gv = wl.global_scales(prompts)
    ak = max(oracle.tensor_amax(k) for k, _ in prompts)
    av = max(oracle.tensor_amax(v) for _, v in prompts)
    assert gk == oracle.calibrated_global_scale(ak)
    assert gv == oracle.calibrated_global_scale(av)
