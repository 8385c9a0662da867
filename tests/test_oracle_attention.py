"""Pins of the oracle's fp64 decode attention over the paged NVFP4 cache.

Decode ("nvfp4-kv-cache-memory-wall", section 3, item 3): one query token per
sequence attends over every cached token, with the dequantisation folded into
the attention.  Pinned by closed forms (q = 0, one token, two tokens), by
torch's scaled_dot_product_attention in float64 over an independently
dequantised dense cache, and by page-table permutation invariance.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from nvfp4_quantized_paged_quantize_gb300 import inputs


def _fill(cache, kv_pairs, page_table):
    """Quantise each sequence's K/V into the cache through the oracle."""
    for b, (k, v) in enumerate(kv_pairs):
        n = k.shape[0]
        t = np.arange(n)
        slots = page_table[b, t // 16].astype(np.int64) * 16 + t % 16
        assert oracle.quantize_append(cache, k, v, slots) == 0


def _dense_dequant(cache, page_table, lens, which):
    """[B][Hkv][L][d] float64, decoded with ml_dtypes' own E2M1/E4M3 tables."""
    mld = pytest.importorskip("ml_dtypes")
    data = cache.k_data if which == "k" else cache.v_data
    scl = cache.k_scale if which == "k" else cache.v_scale
    g = np.float64(np.float32(cache.k_global_scale if which == "k" else cache.v_global_scale))
    H = cache.num_kv_heads
    out = []
    for b, L in enumerate(lens):
        t = np.arange(L)
        pages = page_table[b, t // 16]
        per_head = []
        for h in range(H):
            rows = (pages * H + h) * 16 + t % 16
            d = data[rows]
            codes = np.stack([d & 0xF, d >> 4], -1).reshape(L, -1).astype(np.uint8)
            vals = codes.view(mld.float4_e2m1fn).astype(np.float64)
            s = scl[rows].view(mld.float8_e4m3fn).astype(np.float64)
            per_head.append(vals * np.repeat(s, 16, axis=1) * g)
        out.append(np.stack(per_head))
    return out


def _case(B=3, H=2, G=4, lens=(5, 40, 33), gk=1.0, gv=1.0, seed=0, q_scale=1.0):
    rng = np.random.default_rng(seed)
    maxp = max((L + 15) // 16 for L in lens)
    num_pages = sum((L + 15) // 16 for L in lens) + 3
    perm = rng.permutation(num_pages).astype(np.int32)
    pt = np.full((B, maxp), -1, np.int32)
    pos = 0
    for b, L in enumerate(lens):
        n = (L + 15) // 16
        pt[b, :n] = perm[pos:pos + n]
        pos += n
    cache = oracle.Cache(num_pages, H, 128, 16, gk, gv)
    kv = [(inputs.bf16_bits(rng.normal(0, 1, (L, H, 128)).astype(np.float32)),
           inputs.bf16_bits(rng.normal(0, 1, (L, H, 128)).astype(np.float32))) for L in lens]
    _fill(cache, kv, pt)
    q = inputs.bf16_bits((rng.normal(0, 1, (B, H * G, 128)) * q_scale).astype(np.float32))
    return cache, pt, np.array(lens, np.int32), q


def test_matches_torch_sdpa_float64():
    cache, pt, lens, q = _case(gk=0.7, gv=1.9)
    scale = 1 / math.sqrt(128)
    out, st = oracle.decode_attention(cache, q, pt, lens, scale)
    assert st == 0
    K = _dense_dequant(cache, pt, lens, "k")
    V = _dense_dequant(cache, pt, lens, "v")
    qf = inputs.bf16_bits_to_f32(q).astype(np.float64)
    H = cache.num_kv_heads
    G = q.shape[1] // H
    for b in range(len(lens)):
        qt = torch.from_numpy(qf[b]).unsqueeze(1)                       # [Hq, 1, d]
        kt = torch.from_numpy(K[b]).repeat_interleave(G, dim=0)         # [Hq, L, d]
        vt = torch.from_numpy(V[b]).repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        np.testing.assert_allclose(out[b], ref[:, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_closed_forms_zero_query_single_token():
    cache, pt, lens, q = _case(lens=(1, 37, 16), gv=0.3)
    q0 = np.zeros_like(q)
    out, st = oracle.decode_attention(cache, q0, pt, lens, 1 / math.sqrt(128))
    assert st == 0
    V = _dense_dequant(cache, pt, lens, "v")
    G = q.shape[1] // cache.num_kv_heads
    for b, L in enumerate(lens):
        for hq in range(q.shape[1]):
            # q = 0: every score is 0 and the output is the plain mean of V
            np.testing.assert_allclose(out[b, hq], V[b][hq // G].mean(axis=0), rtol=1e-13,
                                       atol=1e-15)
    out1, _ = oracle.decode_attention(cache, q, pt, lens, 1 / math.sqrt(128))
    for hq in range(q.shape[1]):
        # a single cached token: the output is that token's V
        np.testing.assert_array_equal(out1[0, hq], V[0][hq // G][0])


def test_two_tokens_sigmoid_weighting():
    # K rows chosen on the E2M1 grid so the dequantised scores are known exactly
    H, G = 1, 1
    cache = oracle.Cache(2, H, 128, 16, 1.0, 1.0)
    k = np.zeros((2, 1, 128), np.float32)
    k[0, 0, :16] = 6.0
    k[1, 0, :16] = 3.0
    v = np.zeros((2, 1, 128), np.float32)
    v[0, 0, :] = 6.0          # on the grid: block scale 1.0 exactly
    v[1, 0, :] = -3.0         # on the grid: block scale 0.5 exactly
    pt = np.array([[1]], np.int32)
    oracle.quantize_append(cache, inputs.bf16_bits(k), inputs.bf16_bits(v), np.array([16, 17]))
    q = np.zeros((1, 1, 128), np.float32)
    q[0, 0, 0] = 0.5
    scale = 0.25
    out, _ = oracle.decode_attention(cache, inputs.bf16_bits(q), pt, np.array([2], np.int32), scale)
    gap = scale * 0.5 * (6.0 - 3.0)
    w0 = 1 / (1 + math.exp(-gap))
    np.testing.assert_allclose(out[0, 0], w0 * 6.0 + (1 - w0) * -3.0, rtol=1e-14)


def test_page_permutation_invariance_and_empty_sequence():
    cache, pt, lens, q = _case(lens=(0, 50, 17), seed=3)
    out, st = oracle.decode_attention(cache, q, pt, lens, 1 / math.sqrt(128))
    assert st == 0
    assert not out[0].any()                          # empty sequence -> zeros
    # move every physical page to a new id and rewrite the table accordingly
    rng = np.random.default_rng(5)
    perm = rng.permutation(cache.num_pages)
    H = cache.num_kv_heads
    moved = oracle.Cache(cache.num_pages, H, 128, 16, cache.k_global_scale, cache.v_global_scale)
    for old in range(cache.num_pages):
        new = perm[old]
        for arr_new, arr_old in ((moved.k_data, cache.k_data), (moved.v_data, cache.v_data),
                                 (moved.k_scale, cache.k_scale), (moved.v_scale, cache.v_scale)):
            arr_new[new * H * 16:(new + 1) * H * 16] = arr_old[old * H * 16:(old + 1) * H * 16]
    pt2 = np.where(pt >= 0, perm[np.maximum(pt, 0)], -1).astype(np.int32)
    out2, _ = oracle.decode_attention(moved, q, pt2, lens, 1 / math.sqrt(128))
    np.testing.assert_array_equal(out, out2)


def test_out_of_range_page_is_flagged():
    cache, pt, lens, q = _case(lens=(20,), B=1)
    bad = pt.copy()
    bad[0, 1] = cache.num_pages + 7
    _, st = oracle.decode_attention(cache, q, bad, lens, 0.1)
    assert st == 1
