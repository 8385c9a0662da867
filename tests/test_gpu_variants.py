"""The format variants on the GPU against the oracle: their quantize-append bit
for bit, and decode attention over their caches within the attention tolerance.

"NVFP4: breaking the memory wall" (cloud.tencent.com): stochastic rounding and
a Hadamard rotation before quantisation; MXFP4's blocks of 32 ("NVIDIA NVFP4:
LLM memory doubled, inference 3x" (nmedialink), figure 6).  The oracle side
applies the oracle's per-block functions to every row at its slot, and its
fp64 decode over each format (oracle.decode_attention_format) is the
attention reference.
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import bf16_dev, check_rows, dev, status_word
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


# ---------------------------------------------------------------------------
# decode over each variant's cache
# ---------------------------------------------------------------------------

def _variant_decode_workload(which):
    if which == "tiny":
        return inputs.decode_config(1)                     # B = 2, lengths {101, 258}, 8 q / 2 KV heads
    if which == "8k_scaled":
        return inputs.decode_config(2, 1 / 64)             # 32 x 129 tokens, 64 q / 8 KV heads
    if which == "gqa4_ragged":                             # G = 4, ragged tails and one-token sequences
        return inputs.DecodeWorkload("custom", 31, np.array([1, 15, 16, 17, 200, 64], np.int64), True, 16, 4,
                                     inputs.KVDist("student_t", 0.05, nu=4.0), pool_factor=1.2)
    return inputs.DecodeWorkload("custom", 32, np.array([40, 300, 33], np.int64), True, 16, 2,
                                 inputs.KVDist("channel", lo=0.1, hi=10.0))   # blocks of very different sizes


def _variant_decode_caches(wl, variant):
    """The workload's cache written twice: by the library's variant append (on
    the GPU) and by the oracle's block functions; the same random bytes serve
    stochastic rounding on both sides."""
    prompts = wl.all_prompt_kv()
    nk, nv = wl.new_kv()
    ks, vs, ss = [], [], []
    for b, (k, v) in enumerate(prompts):
        ks += [k, nk[b:b + 1]]
        vs += [v, nv[b:b + 1]]
        ss += [wl.slots(b, 0, k.shape[0]), wl.append_slots()[b:b + 1]]
    k, v, slots = np.concatenate(ks), np.concatenate(vs), np.concatenate(ss)
    n, H = k.shape[0], wl.num_kv_heads
    rk = inputs.rounding_bytes(12, n * H * 128).reshape(n, H, 128)
    rv = inputs.rounding_bytes(13, n * H * 128).reshape(n, H, 128)
    cache = kv.Cache.empty(wl.num_pages, H, zero=True, mxfp4=variant == kv.NVFP4KV_VARIANT_MXFP4)
    kv.nvfp4kv_quantize_append_variant(variant, cache, bf16_dev(k), bf16_dev(v), dev(slots), dev(rk), dev(rv))
    pools = oracle_variant_pools(variant, k, v, slots, wl.num_pages, H, 1.0, 1.0, rk, rv)
    oc = oracle.Cache(wl.num_pages, H, 128, 16,
                      arrays=(pools["k"][0], pools["v"][0], pools["k"][1], pools["v"][1]))
    return cache, oc


@pytest.mark.parametrize("variant", [kv.NVFP4KV_VARIANT_SR, kv.NVFP4KV_VARIANT_HADAMARD, kv.NVFP4KV_VARIANT_MXFP4])
@pytest.mark.parametrize("which", ["tiny", "8k_scaled", "gqa4_ragged", "wide_range"])
def test_variant_decode_matches_oracle(cuda_lib, variant, which):
    wl = _variant_decode_workload(which)
    cache, oc = _variant_decode_caches(wl, variant)
    fmt = {kv.NVFP4KV_VARIANT_SR: oracle.FORMAT_NVFP4, kv.NVFP4KV_VARIANT_HADAMARD: oracle.FORMAT_NVFP4_HADAMARD,
           kv.NVFP4KV_VARIANT_MXFP4: oracle.FORMAT_MXFP4}[variant]
    q = wl.q()
    ref, rs = oracle.decode_attention_format(oc, fmt, q, wl.page_table, wl.seq_lens, wl.softmax_scale)
    assert rs == 0
    ws = torch.zeros(kv.nvfp4kv_decode_workspace_size(cache, wl.batch, wl.num_q_heads), dtype=torch.uint8,
                     device="cuda")
    out = torch.full((wl.batch, wl.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = status_word()
    kv.nvfp4kv_decode_attention_variant(variant, cache, bf16_dev(q), out, dev(wl.page_table),
                                        dev(wl.seq_lens.astype(np.int32)), wl.softmax_scale, ws, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_rows(out.cpu().numpy(), ref)
    if variant == kv.NVFP4KV_VARIANT_SR:
        # stochastic rounding writes plain NVFP4: the ordinary decode reads it the same way
        out2 = torch.empty_like(out)
        kv.nvfp4kv_decode_attention(cache, bf16_dev(q), out2, dev(wl.page_table), dev(wl.seq_lens.astype(np.int32)),
                                    wl.softmax_scale, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, out2)


def test_variant_decode_argument_checks(cuda_lib):
    cache = kv.Cache.empty(2, 1, zero=True)
    q = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda")
    ws = torch.zeros(kv.nvfp4kv_decode_workspace_size(cache, 1, 1), dtype=torch.uint8, device="cuda")
    pt, sl = dev(np.zeros((1, 2), np.int32)), dev(np.array([3], np.int32))
    with pytest.raises(kv.Nvfp4kvError):
        kv.nvfp4kv_decode_attention_variant(7, cache, q, out, pt, sl, 0.1, ws)
    with pytest.raises(kv.Nvfp4kvError):                   # workspace too small
        kv.nvfp4kv_decode_attention_variant(kv.NVFP4KV_VARIANT_MXFP4, cache, q, out, pt, sl, 0.1, ws[:16])
