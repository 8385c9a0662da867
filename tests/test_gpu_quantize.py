"""GPU quantize-append vs the oracle: packed nibbles and scale bytes bit-exact.

Two-level scaling ("nvfp4-kv-cache-memory-wall", section 2) applied on the way
into the paged cache (same page, section 3).
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import (bf16_dev, dev, fill_workload_gpu, fill_workload_oracle, gpu_append, gpu_cache,
                      pool_host, status_word)

pytestmark = pytest.mark.gpu


def _assert_pool_equal(gpu_cache_, orc):
    kd, vd, ks, vs = pool_host(gpu_cache_)
    np.testing.assert_array_equal(ks, orc.k_scale)
    np.testing.assert_array_equal(vs, orc.v_scale)
    np.testing.assert_array_equal(kd, orc.k_data)
    np.testing.assert_array_equal(vd, orc.v_data)


def test_tiny_workload_pool_bit_exact(cuda_lib):
    wl = inputs.decode_config(1)
    prompts = wl.all_prompt_kv()
    new = wl.new_kv()
    st = status_word()
    g = fill_workload_gpu(wl, prompts, new, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _assert_pool_equal(g, fill_workload_oracle(wl, prompts, new))


@pytest.mark.parametrize("index", [2, 3, 4])
def test_scaled_workloads_pool_bit_exact(cuda_lib, index):
    wl = inputs.decode_config(index, scale=1 / 64)
    prompts = wl.all_prompt_kv()
    new = wl.new_kv() if wl.append else None
    g = fill_workload_gpu(wl, prompts, new)
    _assert_pool_equal(g, fill_workload_oracle(wl, prompts, new))


def _edge_blocks():
    """Blocks that walk every E4M3 scale rounding boundary and every E2M1 midpoint."""
    rng = np.random.default_rng(7)
    blocks = []
    e4 = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (e4[:-1] + e4[1:]) / 2
    for m in mids:  # amax / 6 lands on, just below and just above each scale midpoint
        for f in (1.0, 1.0 - 2 ** -7, 1.0 + 2 ** -7):
            x = rng.normal(0, 1, 16) * m
            x[3] = 6 * m * f
            blocks.append(x)
    for s in e4[1:]:  # E2M1 midpoints at an exact scale (amax = 6 * scale)
        x = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, 0.1])
        blocks.append(x * s)
    blocks.append(np.zeros(16))
    blocks.append(-np.zeros(16))
    blocks.append(np.full(16, 1e-6))                         # scale rounds to 0 -> signed zeros
    blocks.append(np.array([3e38] + [1.0] * 15))            # saturated scale
    blocks.append(rng.normal(0, 1e-30, 16))                 # bf16 subnormal range
    return np.stack(blocks).astype(np.float32)


@pytest.mark.parametrize("gk,gv", [(1.0, 1.0), (0.37, 5.5), (1.0 / 2688, 3e-3), (1e3, 1e-5)])
def test_edge_blocks_bit_exact(cuda_lib, gk, gv):
    blocks = _edge_blocks()
    n = (blocks.shape[0] + 7) // 8
    flat = np.zeros((n * 8, 16), np.float32)
    flat[:blocks.shape[0]] = blocks
    x = flat.reshape(n, 1, 128)
    kb = inputs.bf16_bits(x)
    vb = inputs.bf16_bits(-x[::-1].copy())
    slots = np.random.default_rng(1).permutation(n + 5)[:n].astype(np.int64)
    pages = (n + 5 + 15) // 16
    g = gpu_cache(pages, 1, gk, gv)
    gpu_append(g, kb, vb, slots)
    o = oracle.Cache(pages, 1, 128, 16, gk, gv)
    oracle.quantize_append(o, kb, vb, slots)
    _assert_pool_equal(g, o)


def test_every_bf16_value_at_every_scale_bit_exact(cuda_lib):
    # g = 1: for each non-zero E4M3 scale s, blocks whose amax is exactly 6 s
    # followed by 15 bf16 values swept over every bf16 magnitude below 6 s
    allbits = np.arange(0x8000, dtype=np.uint16)                    # non-negative bf16 patterns
    vals = inputs.bf16_bits_to_f32(allbits)
    vals = vals[np.isfinite(vals)]
    rows = []
    for sb in range(1, 0x7F):
        s = oracle.e4m3_value(sb)
        v = vals[vals <= 6 * s]
        v = np.concatenate([v, -v])
        pad = (-v.size) % 15
        v = np.concatenate([v, np.zeros(pad, np.float32)]).reshape(-1, 15)
        blk = np.concatenate([np.full((v.shape[0], 1), 6 * s, np.float32), v], axis=1)
        rows.append(blk)
    blocks = np.concatenate(rows).astype(np.float32)
    n = (blocks.shape[0] + 7) // 8
    flat = np.zeros((n * 8, 16), np.float32)
    flat[:blocks.shape[0]] = blocks
    x = inputs.bf16_bits(flat.reshape(n, 1, 128))
    slots = np.arange(n, dtype=np.int64)
    pages = (n + 15) // 16
    g = gpu_cache(pages, 1)
    gpu_append(g, x, x, slots)
    o = oracle.Cache(pages, 1)
    oracle.quantize_append(o, x, x, slots)
    _assert_pool_equal(g, o)


def test_padding_and_out_of_range_slots(cuda_lib):
    rng = np.random.default_rng(3)
    x = inputs.bf16_bits(rng.normal(0, 1, (6, 2, 128)).astype(np.float32))
    slots = np.array([5, -1, 40, 63, 64, 1 << 40], np.int64)   # pool holds 64 slots
    g = gpu_cache(4, 2)
    st = status_word()
    gpu_append(g, x, x, slots, st)
    torch.cuda.synchronize()
    assert int(st.item()) & kv.NVFP4KV_DEVERR_SLOT
    o = oracle.Cache(4, 2)
    assert oracle.quantize_append(o, x, x, slots) == 1
    _assert_pool_equal(g, o)


@pytest.mark.parametrize("variant", [None, "sr", "hadamard", "mxfp4"])
def test_v_token_pairs_any_slot_order(cuda_lib, variant):
    # V data is stored by token pair (slots 2m, 2m + 1 share bytes): a call's two
    # tokens of a step fill a pair row whole only when their slots are 2m, 2m + 1;
    # every other case merges nibbles.  Cover: consecutive slots from an even
    # and from an odd start, a shuffled order, a pair split between two calls
    # (in both orders), pairs whose partner is padding, and the last token of an
    # odd count; the final pool must equal the oracle's after the same calls.
    from variant_util import MXFP4, SR, HADAMARD, oracle_variant_pools

    rng = np.random.default_rng(17)
    H, pages = 3, 12                                          # 192 slots
    calls = []
    calls.append(np.arange(10, 10 + 21, dtype=np.int64))      # even start, odd count
    calls.append(np.arange(35, 35 + 20, dtype=np.int64))      # odd start: every step straddles two pair rows
    calls.append(rng.permutation(np.arange(60, 100, dtype=np.int64)))  # shuffled
    calls.append(np.array([101, 130, 103, 102, -1, 100, 131], np.int64))  # mixed, partners in this call or none
    calls.append(np.array([104, 150, 107], np.int64))         # halves of pairs (104, 105), (106, 107), (150, 151)
    calls.append(np.array([105, 106, 151, -1, 152], np.int64))  # ... completed later, in the other order
    xs = [inputs.bf16_bits(rng.normal(0, 1, (len(c), H, 128)).astype(np.float32)) for c in calls]
    vs = [inputs.bf16_bits(rng.standard_t(4, (len(c), H, 128)).astype(np.float32)) for c in calls]
    if variant is None:
        g = gpu_cache(pages, H)
        o = oracle.Cache(pages, H)
        for c, x, v in zip(calls, xs, vs):
            gpu_append(g, x, v, c)
            assert oracle.quantize_append(o, x, v, c) == 0
        _assert_pool_equal(g, o)
        return
    var = {"sr": SR, "hadamard": HADAMARD, "mxfp4": MXFP4}[variant]
    g = kv.Cache.empty(pages, H, zero=True, mxfp4=variant == "mxfp4")
    rk = [rng.integers(0, 256, x.shape, dtype=np.uint8) for x in xs]
    rv = [rng.integers(0, 256, x.shape, dtype=np.uint8) for x in xs]
    for c, x, v, a, b in zip(calls, xs, vs, rk, rv):
        kv.nvfp4kv_quantize_append_variant(var, g, bf16_dev(x), bf16_dev(v), dev(c), dev(a), dev(b))
    # the oracle's pools after the same calls, one by one
    want = oracle_variant_pools(var, np.concatenate(xs), np.concatenate(vs), np.concatenate(calls), pages, H,
                                1.0, 1.0, np.concatenate(rk), np.concatenate(rv))
    rows = pages * H * 16
    for name, (data, scale) in want.items():
        gd = (g.k_data if name == "k" else g.v_data).reshape(rows, -1).cpu().numpy()
        gs = (g.k_scale if name == "k" else g.v_scale).reshape(rows, -1).cpu().numpy()
        assert np.array_equal(gd, data), f"{name} data"
        assert np.array_equal(gs, scale), f"{name} scales"


def test_extend_chunk_full_size_bit_exact(cuda_lib):
    # one layer of the extend workload: 16 sequences x 2048 new tokens x 8 KV heads
    wl = inputs.extend_config()
    ks, vs = zip(*[wl.chunk_kv(0, b) for b in range(wl.batch)])
    k = np.concatenate(ks)
    v = np.concatenate(vs)
    slots = wl.chunk_slots()
    g = gpu_cache(wl.num_pages, wl.num_kv_heads)
    kv.nvfp4kv_quantize_append(g, bf16_dev(k), bf16_dev(v), dev(slots))
    o = oracle.Cache(wl.num_pages, wl.num_kv_heads)
    assert oracle.quantize_append(o, k, v, slots) == 0
    _assert_pool_equal(g, o)


def test_random_blocks_wide_scale_range_bit_exact(cuda_lib):
    # 2^20 blocks: magnitudes over 60 binades, global scales over 40 binades
    rng = np.random.default_rng(21)
    for trial, (lo, hi) in enumerate([(-30, 30), (-6, 6)]):
        n = 1 << 13                                          # tokens of one head: 8 blocks each
        mag = 2.0 ** rng.uniform(lo, hi, (n, 1, 8, 1))
        x = (rng.standard_normal((n, 1, 8, 16)) * mag).astype(np.float32).reshape(n, 1, 128)
        x[rng.random(x.shape) < 0.01] *= -1e3
        kb = inputs.bf16_bits(x)
        vb = inputs.bf16_bits(rng.standard_t(3, x.shape).astype(np.float32) * np.float32(2.0 ** rng.uniform(-8, 8)))
        for gk, gv in [(float(2.0 ** rng.uniform(-20, 20)), float(2.0 ** rng.uniform(-20, 20))) for _ in range(3)]:
            gk, gv = float(np.float32(gk)), float(np.float32(gv))
            pages = n // 16
            slots = rng.permutation(n).astype(np.int64)
            g = gpu_cache(pages, 1, gk, gv)
            gpu_append(g, kb, vb, slots)
            o = oracle.Cache(pages, 1, 128, 16, gk, gv)
            assert oracle.quantize_append(o, kb, vb, slots) == 0
            _assert_pool_equal(g, o)


@pytest.mark.parametrize("gk,gv", [(1.0, 0.37), (1 / 2688, 2.9e-3), (5e-31, 1e25), (1e-35, 1e35)])
def test_every_bf16_block_amax_bit_exact(cuda_lib, gk, gv):
    # The block scale is E4M3(amax / (6 g)): every finite positive bf16 value
    # is the amax of one block, once for K and once for V, at global scales
    # whose 6 g lies inside and outside [2^-100, 2^100] (the kernel's fast
    # reciprocal path and its IEEE-division fallback).  The other 15 values of
    # a block are drawn at or below the amax, with random signs.
    rng = np.random.default_rng(17)
    amax = inputs.bf16_bits_to_f32(np.arange(1, 0x7F80, dtype=np.uint16))
    frac = rng.random((amax.size, 15)).astype(np.float32)
    sign = np.where(rng.random((amax.size, 15)) < 0.5, -1.0, 1.0).astype(np.float32)
    blocks = np.concatenate([amax[:, None], amax[:, None] * frac * sign], axis=1)
    n = (blocks.shape[0] + 7) // 8
    flat = np.zeros((n * 8, 16), np.float32)
    flat[:blocks.shape[0]] = blocks
    kb = inputs.bf16_bits(flat.reshape(n, 1, 128))
    vb = inputs.bf16_bits(flat[::-1].copy().reshape(n, 1, 128))
    slots = np.arange(n, dtype=np.int64)
    pages = (n + 15) // 16
    g = gpu_cache(pages, 1, gk, gv)
    gpu_append(g, kb, vb, slots)
    o = oracle.Cache(pages, 1, 128, 16, gk, gv)
    oracle.quantize_append(o, kb, vb, slots)
    _assert_pool_equal(g, o)
