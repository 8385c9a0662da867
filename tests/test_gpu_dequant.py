"""GPU NVFP4 -> FP8 E4M3 workspace vs the oracle (bit-exact).

Chunked prefill / extend dequantises the NVFP4 prefix into one FP8 workspace
reused by every layer ("nvfp4-kv-cache-memory-wall", section 3, item 2).
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import dev, gpu_append, gpu_cache, status_word

pytestmark = pytest.mark.gpu

CANARY = 0xA5


def _prefix_caches(wl, layer, gk=1.0, gv=1.0):
    g = gpu_cache(wl.num_pages, wl.num_kv_heads, gk, gv)
    o = oracle.Cache(wl.num_pages, wl.num_kv_heads, 128, 16, gk, gv)
    for b in range(wl.batch):
        k, v = wl.prefix_kv(layer, b)
        slots = wl.slots(b, 0, wl.prefix_len)
        gpu_append(g, k, v, slots)
        assert oracle.quantize_append(o, k, v, slots) == 0
    return g, o


def _run(wl, g, sk=1.0, sv=1.0, ws=None, status=None, page_table=None):
    rows = wl.total_rows
    if ws is None:
        ws = (torch.full((rows, wl.num_kv_heads, 128), CANARY, dtype=torch.uint8, device="cuda"),
              torch.full((rows, wl.num_kv_heads, 128), CANARY, dtype=torch.uint8, device="cuda"))
    pt = wl.page_table if page_table is None else page_table
    kv.nvfp4kv_dequant_to_fp8_workspace(g, dev(pt), dev(wl.prefix_lens), dev(wl.cu_prefix), ws[0], ws[1],
                                        sk, sv, device_status=status)
    return ws


def _expect(wl, o, sk=1.0, sv=1.0, page_table=None):
    pt = wl.page_table if page_table is None else page_table
    ek, ev, st = oracle.dequant_to_fp8_workspace(o, pt, wl.prefix_lens, wl.cu_prefix, wl.total_rows, sk, sv)
    # rows the call must not touch keep the canary
    mask = np.ones(wl.total_rows, bool)
    for b in range(wl.batch):
        mask[wl.cu_prefix[b]:wl.cu_prefix[b] + wl.prefix_lens[b]] = False
    ek[mask] = CANARY
    ev[mask] = CANARY
    return ek, ev, st


@pytest.mark.parametrize("sk,sv,gk,gv", [(1.0, 1.0, 1.0, 1.0), (6.0, 0.25, 1.0, 1.0),
                                         (1.0, 1.0, 0.37, 2.5), (6e-3, 2.4e-2, 1e-3, 4e-3)])
def test_scaled_extend_bit_exact(cuda_lib, sk, sv, gk, gv):
    wl = inputs.extend_config(scale=1 / 16, num_layers=1)
    g, o = _prefix_caches(wl, 0, gk, gv)
    ws = _run(wl, g, sk, sv)
    ek, ev, st = _expect(wl, o, sk, sv)
    assert st == 0
    np.testing.assert_array_equal(ws[0].cpu().numpy(), ek)
    np.testing.assert_array_equal(ws[1].cpu().numpy(), ev)


def test_workspace_reused_across_layers(cuda_lib):
    wl = inputs.extend_config(scale=1 / 32, num_layers=3)
    ws = None
    for layer in range(3):
        g, o = _prefix_caches(wl, layer)
        ws = _run(wl, g, ws=ws)
        ek, ev, _ = _expect(wl, o)
        np.testing.assert_array_equal(ws[0].cpu().numpy(), ek)
        np.testing.assert_array_equal(ws[1].cpu().numpy(), ev)


def test_bad_page_writes_zeros_and_flags(cuda_lib):
    wl = inputs.extend_config(scale=1 / 64, num_layers=1)
    g, o = _prefix_caches(wl, 0)
    pt = wl.page_table.copy()
    pt[1, 3] = -7
    st = status_word()
    ws = _run(wl, g, status=st, page_table=pt)
    torch.cuda.synchronize()
    assert int(st.item()) & kv.NVFP4KV_DEVERR_PAGE
    ek, ev, rs = _expect(wl, o, page_table=pt)
    assert rs == 1
    np.testing.assert_array_equal(ws[0].cpu().numpy(), ek)
    np.testing.assert_array_equal(ws[1].cpu().numpy(), ev)


def test_full_size_layer_sampled_rows(cuda_lib):
    # one full layer of the extend workload (16 x 16384-token prefixes, 8 KV heads)
    wl = inputs.extend_config(num_layers=1)
    g = gpu_cache(wl.num_pages, wl.num_kv_heads)
    prefixes = [wl.prefix_kv(0, b) for b in range(wl.batch)]
    for b, (k, v) in enumerate(prefixes):
        gpu_append(g, k, v, wl.slots(b, 0, wl.prefix_len))
    ws = _run(wl, g)
    wk, wv = ws[0].cpu().numpy(), ws[1].cpu().numpy()
    for b in (0, 9, 15):
        # oracle over this sequence only: a one-sequence cache with a compact page table
        k, v = prefixes[b]
        npg = (wl.prefix_len + 15) // 16
        o = oracle.Cache(npg, wl.num_kv_heads)
        assert oracle.quantize_append(o, k, v, np.arange(wl.prefix_len, dtype=np.int64)) == 0
        ek, ev, st = oracle.dequant_to_fp8_workspace(
            o, np.arange(npg, dtype=np.int32)[None], np.array([wl.prefix_len], np.int32),
            np.array([0, wl.prefix_len], np.int64), wl.prefix_len)
        assert st == 0
        r0 = int(wl.cu_prefix[b])
        np.testing.assert_array_equal(wk[r0:r0 + wl.prefix_len], ek)
        np.testing.assert_array_equal(wv[r0:r0 + wl.prefix_len], ev)
        assert np.all(wk[r0 + wl.prefix_len:int(wl.cu_prefix[b + 1])] == CANARY)


@pytest.mark.parametrize("gk,gv,sk,sv", [(1.0, 1.0, 1.0, 1.0), (0.37, 2.5, 6.0, 1e-3), (1e30, 1e-20, 1e-10, 1e31),
                                         (1.0, 3.0, 1e-35, 1e35), (1 / 2688, 2.9e-3, 6 / 2688, 6 * 2.9e-3),
                                         # workspace scales inside [2^-100, 2^100] whose quotients overflow
                                         # (saturate to 448) or pass 2^64
                                         (1e10, 1.0, 1e-29, 2.0 ** -99)])
def test_every_code_and_scale_bit_exact(cuda_lib, gk, gv, sk, sv):
    # One KV head, two pages: block j of row r holds scale byte 8 r + j (every
    # non-negative, non-NaN E4M3 byte once per page) and the 16 E2M1 codes
    # 0..15, in order for K and reversed for V.  Workspace scales inside and
    # outside [2^-100, 2^100] take the kernel's reciprocal path and its
    # IEEE-division fallback; (1, 1) takes the unit-scale path.
    sc = np.zeros((2, 16, 8), np.uint8)
    sc[:] = np.minimum(np.arange(128, dtype=np.uint8), 0x7E).reshape(16, 8)
    sc[1] = sc[1][::-1]
    fwd = np.array([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE], np.uint8)
    rev = np.array([0xEF, 0xCD, 0xAB, 0x89, 0x67, 0x45, 0x23, 0x01], np.uint8)
    kd = np.tile(fwd, (2, 16, 8))
    vd = np.tile(rev, (2, 16, 8))
    g = gpu_cache(2, 1, gk, gv)
    g.k_data.copy_(torch.from_numpy(kd.reshape(2, 1, 16, 64)))
    g.set_v_data(torch.from_numpy(vd.reshape(2, 1, 16, 64)).cuda())
    g.k_scale.copy_(torch.from_numpy(sc.reshape(2, 1, 16, 8)))
    g.v_scale.copy_(torch.from_numpy(sc[::-1].copy().reshape(2, 1, 16, 8)))
    o = oracle.Cache(2, 1, 128, 16, gk, gv, arrays=(kd, vd, sc, sc[::-1].copy()))
    pt = np.array([[1, 0]], np.int32)
    pl = np.array([32], np.int32)
    cu = np.array([0, 32], np.int64)
    ws = (torch.full((32, 1, 128), CANARY, dtype=torch.uint8, device="cuda"),
          torch.full((32, 1, 128), CANARY, dtype=torch.uint8, device="cuda"))
    kv.nvfp4kv_dequant_to_fp8_workspace(g, dev(pt), dev(pl), dev(cu), ws[0], ws[1], sk, sv)
    ek, ev, st = oracle.dequant_to_fp8_workspace(o, pt, pl, cu, 32, sk, sv)
    assert st == 0
    np.testing.assert_array_equal(ws[0].cpu().numpy(), ek)
    np.testing.assert_array_equal(ws[1].cpu().numpy(), ev)
