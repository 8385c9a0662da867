"""The C-ABI library builds, loads and exports every symbol the header declares.

No compute call is made here (these run without a GPU): only size queries and
the host-side argument checks that return before anything touches CUDA.
"""
import ctypes
import os
import re

import pytest

import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import build as kvbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "nvfp4kv.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4kv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)

    return kv.load()


def test_library_builds_in_tree():
    path = kvbuild.build()
    assert os.path.exists(path)
    assert os.path.dirname(path).startswith(os.path.dirname(kv.__file__))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert set(names) >= {"nvfp4kv_quantize_append", "nvfp4kv_decode_attention",
                          "nvfp4kv_dequant_to_fp8_workspace", "nvfp4kv_decode_workspace_size",
                          "nvfp4kv_cache_bytes", "nvfp4kv_status_string"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, 12345):
        assert kv.nvfp4kv_status_string(code)
    assert kv.nvfp4kv_status_string(-4).startswith("workspace")


def test_cache_bytes_nine_sixteenths(lib):
    n = kv.nvfp4kv_cache_bytes(10, 8)
    values = 10 * 8 * 16 * 128                    # of K, and as many of V
    assert n == 2 * values * 9 // 16
    assert n == 10 * 8 * kv.NVFP4KV_PAGE_HEAD_BYTES  # one 2304-byte page-head per (page, KV head)
    with pytest.raises(kv.Nvfp4kvError):
        kv.nvfp4kv_cache_bytes(0, 8)
    with pytest.raises(kv.Nvfp4kvError):
        kv.nvfp4kv_cache_bytes(1 << 62, 8)        # overflows size_t arithmetic


def test_page_head_views_cover_the_pool_once(lib):
    import torch

    for mx in (False, True):
        c = kv.Cache.empty(3, 2, device="cpu", zero=True, mxfp4=mx)
        for i, part in enumerate((c.k_data, c.k_scale, c.v_pairs, c.v_scale)):
            part.fill_(i + 1)
        # every byte of the pool belongs to exactly one of the four views
        counts = torch.bincount(c.pages.reshape(-1).long(), minlength=5)
        sc = 4 if mx else 8
        assert counts[0] == 0
        assert counts[1] == counts[3] == 3 * 2 * 16 * 64
        assert counts[2] == counts[4] == 3 * 2 * 16 * sc
        # the order within a page-head: K data, K scales, V data, V scales
        ph = c.pages[1, 1].tolist()
        assert ph == [1] * 1024 + [2] * 16 * sc + [3] * 1024 + [4] * 16 * sc
        # K scales token-major, V scales block-major
        c.pages.zero_()
        c.k_scale[0, 0, 3, 1] = 7
        c.v_scale[0, 0, 3, 1] = 9
        ph = c.pages[0, 0]
        assert ph[1024 + 3 * sc + 1] == 7
        assert ph[2048 + 16 * sc + 16 * 1 + 3] == 9
        # V data by token pair: dimension d of tokens 2p (low nibble) and 2p + 1 (high)
        rows = torch.zeros((3, 2, 16, 64), dtype=torch.uint8)
        rows[2, 1, 5, 3] = 0xA0                     # token 5, dimension 7 = 0xA (high nibble of byte 3)
        rows[2, 1, 4, 3] = 0x0B                     # token 4, dimension 6 = 0xB
        c.set_v_data(rows)
        pr = c.pages[2, 1, 1024 + 16 * sc: 2048 + 16 * sc].reshape(8, 128)
        assert pr[2, 7] == 0xA0 and pr[2, 6] == 0x0B and int(pr.sum()) == 0xA0 + 0x0B
        assert torch.equal(c.v_data, rows)


def test_decode_workspace_bytes_from_the_batch_shape(lib):
    # the call the scope table names: sized from (batch, q heads, max length, SMs)
    f = kv.nvfp4kv_decode_workspace_bytes
    assert f(-1, 8, 100, 152) == 0 and f(4, 0, 100, 152) == 0 and f(4, 8, 100, 0) == 0
    a = f(32, 64, 8193, 152)
    assert a > 0
    assert f(32, 64, 131072, 152) == a           # no length sizes the split-K scratch
    records = 2 * (152 * 3 * 4) * (8 * 128 + 16) * 4   # two per warp of the launch
    assert a == records + 33 * 4                 # and each sequence's page prefix
    assert f(33, 8, 8193, 152) == a + 4          # neither the query nor the KV heads count
    assert f(32, 64, 8193, 160) > a              # split records per CTA of the launch
    assert f(0, 64, 0, 152) == records + 4       # the records of the launch even for no sequences


def _fake_cache(**kw):
    # aligned fake addresses: these calls are rejected before any device access
    c = kv.Cache(0x10000, 4, 2)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _raw(lib, fn, *args):
    return getattr(lib, fn)(*args)


def test_host_validation_codes(lib):
    c = _fake_cache()
    cs = c.c_struct()
    P = ctypes.byref
    # null cache
    assert lib.nvfp4kv_quantize_append(None, 16, 16, 8, 1, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    # unsupported head_dim / page size
    bad = _fake_cache(head_dim=64).c_struct()
    assert lib.nvfp4kv_quantize_append(P(bad), 16, 16, 8, 1, None, None) == kv.NVFP4KV_ERR_UNSUPPORTED
    bad = _fake_cache(page_size=32).c_struct()
    assert lib.nvfp4kv_decode_attention(P(bad), 16, 16, 4, 1, 4, 1, 2, 0.1, 256, 1 << 20, None,
                                        None) == kv.NVFP4KV_ERR_UNSUPPORTED
    # misaligned pool, bad global scale
    bad = _fake_cache(pages=0x10001).c_struct()
    assert lib.nvfp4kv_quantize_append(P(bad), 16, 16, 8, 1, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    bad = _fake_cache(k_global_scale=float("nan")).c_struct()
    assert lib.nvfp4kv_quantize_append(P(bad), 16, 16, 8, 1, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    bad = _fake_cache(v_global_scale=0.0).c_struct()
    assert lib.nvfp4kv_quantize_append(P(bad), 16, 16, 8, 1, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    # zero tokens is a no-op; negative is an error
    assert lib.nvfp4kv_quantize_append(P(cs), None, None, None, 0, None, None) == kv.NVFP4KV_OK
    assert lib.nvfp4kv_quantize_append(P(cs), 16, 16, 8, -1, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    # misaligned k
    assert lib.nvfp4kv_quantize_append(P(cs), 18, 16, 8, 1, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    # decode: group not dividing, group > 8, bad softmax scale, empty batch
    assert lib.nvfp4kv_decode_attention(P(cs), 16, 16, 4, 1, 4, 1, 3, 0.1, 256, 1 << 20, None,
                                        None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert lib.nvfp4kv_decode_attention(P(cs), 16, 16, 4, 1, 4, 1, 18, 0.1, 256, 1 << 20, None,
                                        None) == kv.NVFP4KV_ERR_UNSUPPORTED
    assert lib.nvfp4kv_decode_attention(P(cs), 16, 16, 4, 1, 4, 1, 8, -1.0, 256, 1 << 20, None,
                                        None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert lib.nvfp4kv_decode_attention(P(cs), 16, 16, 4, 1, 4, 0, 8, 0.1, 256, 1 << 20, None,
                                        None) == kv.NVFP4KV_OK
    # dequant: bad workspace scale, misaligned workspace, nothing to do
    assert lib.nvfp4kv_dequant_to_fp8_workspace(P(cs), 4, 1, 4, 8, 1, 16, 0.0, 1.0, 16, 16, None,
                                                None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert lib.nvfp4kv_dequant_to_fp8_workspace(P(cs), 4, 1, 4, 8, 1, 16, 1.0, 1.0, 17, 16, None,
                                                None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert lib.nvfp4kv_dequant_to_fp8_workspace(P(cs), 4, 1, 4, 8, 1, 0, 1.0, 1.0, 16, 16, None,
                                                None) == kv.NVFP4KV_OK


def test_fused_step_checks_both_calls_before_enqueueing(lib):
    cs = _fake_cache().c_struct()
    P = ctypes.byref
    f = lib.nvfp4kv_append_decode_attention
    # a bad append argument (misaligned k) or a bad decode argument (group 3)
    # is reported; with nothing to append and an empty batch nothing happens
    assert f(P(cs), 18, 16, 8, 1, 16, 16, 4, 1, 4, 0, 8, 0.1, 256, 1 << 20, None, None) == \
        kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(P(cs), 16, 16, 8, 1, 16, 16, 4, 1, 4, 1, 3, 0.1, 256, 1 << 20, None, None) == \
        kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(P(cs), 16, 16, 8, 1, 16, 16, 4, 1, 4, 1, 8, float("inf"), 256, 1 << 20, None, None) == \
        kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(P(cs), None, None, None, 0, 16, 16, 4, 1, 4, 0, 8, 0.1, 256, 1 << 20, None, None) == kv.NVFP4KV_OK


def test_calibration_host_checks_and_scale(lib):
    from oracle import calibrated_global_scale

    import numpy as np

    # amax: negative size, misaligned input or output are refused before CUDA
    f = lib.nvfp4kv_tensor_amax
    assert f(16, -1, 16, 0, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(18, 8, 16, 0, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(16, 8, 18, 1, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(None, 8, 16, 0, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(16, 8, None, 1, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    # the global scale is host arithmetic: equal to the oracle's, bit for bit
    for bad in (-1.0, float("nan"), float("inf"), -0.5e-40):
        with pytest.raises(kv.Nvfp4kvError):
            kv.nvfp4kv_calibrated_global_scale(bad)
    rng = np.random.default_rng(7)
    amaxes = [0.0, -0.0, 1e-45, 1.0, 2688.0, 448.0, 6.0, 3.3895314e38] + \
        list(np.exp(rng.uniform(-100, 88, 200)).astype(np.float32))
    for a in amaxes:
        got = np.float32(kv.nvfp4kv_calibrated_global_scale(float(a)))
        want = np.float32(calibrated_global_scale(float(a)))
        assert got.tobytes() == want.tobytes(), a


def test_extend_host_checks(lib):
    f = lib.nvfp4kv_extend_attention
    # (q, cu_q, max_q_len, ws_k, ws_v, cu_prefix, prefix_lens, batch, total_rows, hq, hkv, d, sk, sv, scale, out, st, stream)
    ok = [16, 8, 4, 16, 16, 8, 4, 2, 100, 8, 2, 128, 1.0, 1.0, 0.1, 16, None, None]
    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a9=6) == kv.NVFP4KV_ERR_UNSUPPORTED           # group 3: not a power of two
    assert call(a9=7) == kv.NVFP4KV_ERR_INVALID_ARGUMENT      # 7 % 2 != 0
    assert call(a11=64) == kv.NVFP4KV_ERR_UNSUPPORTED         # head_dim
    assert call(a12=0.0) == kv.NVFP4KV_ERR_INVALID_ARGUMENT   # workspace scale
    assert call(a14=float("nan")) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert call(a0=18) == kv.NVFP4KV_ERR_INVALID_ARGUMENT     # misaligned q
    assert call(a5=12) == kv.NVFP4KV_ERR_INVALID_ARGUMENT     # misaligned cu_prefix
    assert call(a7=-1) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert call(a7=0) == kv.NVFP4KV_OK and call(a2=0) == kv.NVFP4KV_OK   # nothing to do
    g = lib.nvfp4kv_bf16_to_fp8_workspace
    assert g(16, 16, 8, 4, 2, 64, 10, 1.0, 1.0, 16, 16, None, None) == kv.NVFP4KV_ERR_UNSUPPORTED
    assert g(16, 16, 8, 4, 2, 128, 10, -1.0, 1.0, 16, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert g(16, 16, 12, 4, 2, 128, 10, 1.0, 1.0, 16, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert g(None, None, None, 0, 2, 128, 10, 1.0, 1.0, None, None, None, None) == kv.NVFP4KV_OK


def test_fused_write_host_checks(lib):
    cs = _fake_cache().c_struct()
    f = lib.nvfp4kv_quantize_append_fp8
    P = ctypes.byref
    # (cache, k, v, slots, n, ws_rows, total_rows, sk, sv, ws_k, ws_v, status, stream)
    assert f(P(cs), 16, 16, 8, 4, 8, 10, 0.0, 1.0, 16, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(P(cs), 16, 16, 8, 4, 12, 10, 1.0, 1.0, 16, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(P(cs), 18, 16, 8, 4, 8, 10, 1.0, 1.0, 16, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(P(cs), None, None, None, 0, None, 10, 1.0, 1.0, None, None, None, None) == kv.NVFP4KV_OK


def test_variant_append_host_checks(lib):
    cs = _fake_cache().c_struct()
    f = lib.nvfp4kv_quantize_append_variant
    P = ctypes.byref
    # (variant, cache, k, v, slots, n, rand_k, rand_v, status, stream)
    assert f(0, P(cs), 16, 16, 8, 4, 16, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT   # unknown variant
    assert f(4, P(cs), 16, 16, 8, 4, 16, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(kv.NVFP4KV_VARIANT_SR, P(cs), 16, 16, 8, 4, None, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(kv.NVFP4KV_VARIANT_SR, P(cs), 16, 16, 8, 4, 24, 16, None, None) == kv.NVFP4KV_ERR_INVALID_ARGUMENT
    assert f(kv.NVFP4KV_VARIANT_MXFP4, P(cs), 18, 16, 8, 4, None, None, None, None) == \
        kv.NVFP4KV_ERR_INVALID_ARGUMENT                                                      # misaligned k
    assert f(kv.NVFP4KV_VARIANT_HADAMARD, P(cs), None, None, None, 0, None, None, None, None) == kv.NVFP4KV_OK
