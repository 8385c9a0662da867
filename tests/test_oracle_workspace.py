"""Pins of the oracle's FP8 E4M3 workspace dequantisation.

Chunked prefill / extend ("nvfp4-kv-cache-memory-wall", section 3, item 2):
the NVFP4 prefix is dequantised into one FP8 workspace reused by every layer.
Pinned by the per-element closed form with unit scales (a plain E4M3 cast of
the dequantised value, via ml_dtypes), E4M3's rounding bound for other
scales, and the row mapping.
"""
import numpy as np
import pytest

import oracle
from nvfp4_quantized_paged_quantize_gb300 import inputs


def _make(lens, H=2, gk=1.0, gv=1.0, seed=0, extra_rows=3):
    rng = np.random.default_rng(seed)
    maxp = max((L + 15) // 16 for L in lens)
    num_pages = sum((L + 15) // 16 for L in lens)
    perm = rng.permutation(num_pages).astype(np.int32)
    pt = np.full((len(lens), maxp), -1, np.int32)
    pos = 0
    cache = oracle.Cache(num_pages, H, 128, 16, gk, gv)
    for b, L in enumerate(lens):
        n = (L + 15) // 16
        pt[b, :n] = perm[pos:pos + n]
        pos += n
        x = rng.standard_t(4, (2, L, H, 128)) * 0.05
        x[:, rng.random((L, H, 128)) < 0.002] = 6.0
        t = np.arange(L)
        slots = pt[b, t // 16].astype(np.int64) * 16 + t % 16
        oracle.quantize_append(cache, inputs.bf16_bits(x[0].astype(np.float32)),
                               inputs.bf16_bits(x[1].astype(np.float32)), slots)
    cu = np.concatenate([[0], np.cumsum(np.array(lens) + extra_rows)]).astype(np.int64)
    return cache, pt, np.array(lens, np.int32), cu


def test_unit_scales_equal_plain_e4m3_cast():
    mld = pytest.importorskip("ml_dtypes")
    lens = (33, 16, 7)
    cache, pt, pl, cu = _make(lens)
    ws_k, ws_v, st = oracle.dequant_to_fp8_workspace(cache, pt, pl, cu, int(cu[-1]))
    assert st == 0
    from test_oracle_attention import _dense_dequant

    for which, ws in (("k", ws_k), ("v", ws_v)):
        dense = _dense_dequant(cache, pt, lens, which)
        for b, L in enumerate(lens):
            ref = dense[b].transpose(1, 0, 2).astype(np.float32)       # [L][H][d]
            ref = np.clip(ref, -448, 448).astype(mld.float8_e4m3fn).view(np.uint8)
            np.testing.assert_array_equal(ws[cu[b]:cu[b] + L], ref)
            assert not ws[cu[b] + L:cu[b + 1]].any()            # gap rows untouched


def test_all_codes_and_scales_unit_scales():
    mld = pytest.importorskip("ml_dtypes")
    # every (E2M1 code, E4M3 scale) pair once: closed form E4M3(e2m1 * scale)
    for sb in range(0x7F):
        s = oracle.e4m3_value(sb)
        for code in range(16):
            ref = np.array([oracle.e2m1_value(code) * s], np.float32)
            ref = np.clip(ref, -448, 448).astype(mld.float8_e4m3fn).view(np.uint8)[0]
            assert oracle.e4m3_encode(np.float32(oracle.e2m1_value(code) * s)) == ref


@pytest.mark.parametrize("gk,gv,sk,sv", [(0.37, 2.5, 1.0, 1.0), (1.0, 1.0, 0.25, 3.0),
                                         (1e-3, 4e-3, 6e-3, 2.4e-2)])
def test_general_scales_within_e4m3_rounding(gk, gv, sk, sv):
    lens = (20, 45)
    cache, pt, pl, cu = _make(lens, gk=gk, gv=gv, seed=1, extra_rows=0)
    ws_k, ws_v, st = oracle.dequant_to_fp8_workspace(cache, pt, pl, cu, int(cu[-1]), sk, sv)
    assert st == 0
    from test_oracle_attention import _dense_dequant

    for which, ws, s in (("k", ws_k, sk), ("v", ws_v, sv)):
        dense = _dense_dequant(cache, pt, lens, which)
        for b, L in enumerate(lens):
            ref = dense[b].transpose(1, 0, 2) / np.float64(np.float32(s))
            got = np.array([oracle.e4m3_value(int(c)) for c in ws[cu[b]:cu[b] + L].reshape(-1)])
            ref = ref.reshape(-1)
            sat = np.abs(ref) > 448
            assert np.all(np.abs(got[sat]) == 448)
            r = ref[~sat]
            # half an E4M3 step: 2^-4 relative for normals, 2^-10 absolute below 2^-6
            bound = np.maximum(np.abs(r) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
            assert np.all(np.abs(got[~sat] - r) <= bound)


def test_bad_page_writes_zeros_and_flags():
    lens = (40,)
    cache, pt, pl, cu = _make(lens)
    bad = pt.copy()
    bad[0, 2] = 10_000
    ws_k, _, st = oracle.dequant_to_fp8_workspace(cache, bad, pl, cu, int(cu[-1]))
    assert st == 1
    assert not ws_k[32:40].any() and ws_k[:32].any()
