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


def test_calibrated_workload_reaches_the_top_scale():
    # over the long-context workload, the calibrated scale of each of K and V
    # gives the block holding that tensor's amax E4M3 scale 448 (code 0x7E) and
    # no block a larger one; with scale 1 the same data stays far below it
    wl = inputs.decode_config(3, 1 / 1024)
    prompts = wl.all_prompt_kv()
    pairs = wl.calibration_tensors(prompts)
    assert len(pairs) == wl.batch
    ak = max(oracle.tensor_amax(k) for k, _ in pairs)
    av = max(oracle.tensor_amax(v) for _, v in pairs)
    for gk, gv, top in ((oracle.calibrated_global_scale(ak), oracle.calibrated_global_scale(av), 0x7E),
                        (1.0, 1.0, None)):
        c = oracle.Cache(wl.num_pages, wl.num_kv_heads, 128, 16, gk, gv)
        for b, (k, v) in enumerate(prompts):
            assert oracle.quantize_append(c, k, v, wl.slots(b, 0, k.shape[0])) == 0
        for sc in (c.k_scale, c.v_scale):
            if top is None:
                assert sc.max() < 0x60                                  # below 32: far from 448
            else:
                assert sc.max() == top


def test_uncalibrated_workloads_have_no_calibration_tensors():
    for index in (1, 2, 4):
        assert inputs.decode_config(index, 1 / 64).calibration_tensors() == []


def _rmse_report(wl, prompts, gk, gv):
    """RMSE of the oracle's dequantised cache against the bf16 inputs, K and V."""
    import math

    H = wl.num_kv_heads
    c = oracle.Cache(wl.num_pages, H, 128, 16, gk, gv)
    err = {"k": 0.0, "v": 0.0}
    n = 0
    for b, (k, v) in enumerate(prompts):
        s = wl.slots(b, 0, k.shape[0])
        assert oracle.quantize_append(c, k, v, s) == 0
        rows = ((((s >> 4) * H)[:, None] + np.arange(H)[None, :]) * 16 + (s & 15)[:, None]).reshape(-1)
        for which, x in (("k", k), ("v", v)):
            xh = oracle.dequantize_rows(c, which, rows)
            err[which] += float(((xh - inputs.bf16_bits_to_f32(x).reshape(-1, 128).astype(np.float64)) ** 2).sum())
        n += k.size
    return {w: math.sqrt(e / n) for w, e in err.items()}


@pytest.mark.parametrize("index,scale", [(2, 1 / 64), (3, 1 / 256)])
def test_rmse_report_unit_vs_calibrated(index, scale, capsys):
    # the RMSE of g = 1 against the calibrated scale on the decode workloads:
    # calibration never does worse here (it moves block scales out of E4M3's
    # subnormal range when values are small, as in the 8K workload's N(0, 0.02))
    wl = inputs.decode_config(index, scale)
    prompts = wl.all_prompt_kv()
    g = [oracle.calibrated_global_scale(max(oracle.tensor_amax(p[i]) for p in prompts)) for i in range(2)]
    unit = _rmse_report(wl, prompts, 1.0, 1.0)
    cal = _rmse_report(wl, prompts, *g)
    with capsys.disabled():
        print(f"\n{wl.name} (x{scale:g}): RMSE g=1 K {unit['k']:.6g} V {unit['v']:.6g}; "
              f"calibrated (gK {g[0]:.6g}, gV {g[1]:.6g}) K {cal['k']:.6g} V {cal['v']:.6g}")
    for w in ("k", "v"):
        assert cal[w] <= unit[w]


def test_rmse_small_values_need_calibration():
    # values of N(0, 0.002): with g = 1 most block scales round below E4M3's
    # smallest subnormal (2^-9) and the blocks store zeros; the calibrated
    # scale keeps the usual NVFP4 error (a few percent of the RMS value)
    rng = np.random.default_rng(8)
    x = inputs.bf16_bits((rng.standard_normal(4096 * 16) * 0.002).astype(np.float32))
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    rms = float(np.sqrt(np.mean(xf ** 2)))

    def rmse(g):
        err = 0.0
        for blk in xf.reshape(-1, 16):
            packed, sb = oracle.quantize_block(blk.astype(np.float32), g)
            codes = np.stack([np.asarray(packed) & 0xF, np.asarray(packed) >> 4], axis=-1).reshape(-1)
            xh = np.array([oracle.dequant_value(int(c), int(sb), g) for c in codes])
            err += float(((xh - blk) ** 2).sum())
        return float(np.sqrt(err / xf.size))

    g_cal = oracle.calibrated_global_scale(oracle.tensor_amax(x))
    assert rmse(1.0) > 0.6 * rms
    assert rmse(g_cal) < 0.15 * rms
