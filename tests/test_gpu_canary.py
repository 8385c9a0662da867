"""Guard-band canaries around every output of the library.

Each output (cache pools, FP8 workspaces, attention outputs, split-K scratch,
the amax word) is a view into the middle of a larger allocation whose two
64 KB guard bands hold a sentinel byte.  After the calls, the bands must be
untouched: a write past either end of an output shows here, where the
element-wise comparisons with the oracle (which look only inside the outputs)
cannot see it.
"""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import bf16_dev, dev, gpu_append

pytestmark = pytest.mark.gpu

GUARD = 1 << 16  # bytes on each side: a multiple of 16, so every view stays 16-byte aligned
SENTINEL = 0xA7


class Guarded:
    """A tensor of the given shape and dtype between two sentinel bands."""

    def __init__(self, shape, dtype):
        itemsize = torch.empty(0, dtype=dtype).element_size()
        nbytes = int(np.prod(shape)) * itemsize
        self.raw = torch.full((GUARD + nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        r = self.raw.cpu().numpy()
        return bool((r[:GUARD] == SENTINEL).all() and (r[-GUARD:] == SENTINEL).all())


def _guarded_cache(pages, H, scale_bytes=8, gk=1.0, gv=1.0):
    mx = scale_bytes == 4
    phb = kv.NVFP4KV_MXFP4_PAGE_HEAD_BYTES if mx else kv.NVFP4KV_PAGE_HEAD_BYTES
    pool = Guarded((pages, H, phb), torch.uint8)
    return kv.Cache(pool.t, pages, H, gk, gv, mxfp4=mx), [pool]


def test_decode_paths_stay_inside_their_outputs(cuda_lib):
    wl = inputs.decode_config(1)                           # B = 2, lengths {101, 258}, 8 q / 2 KV heads
    prompts = wl.all_prompt_kv()
    new = wl.new_kv()
    cache, pools = _guarded_cache(wl.num_pages, wl.num_kv_heads)
    for b, (k, v) in enumerate(prompts):
        gpu_append(cache, k, v, wl.slots(b, 0, k.shape[0]))
    B, Hq = wl.batch, wl.num_q_heads
    n = kv.nvfp4kv_decode_workspace_size(cache, B, Hq)
    ws = Guarded((n,), torch.uint8)
    out = Guarded((B, Hq, 128), torch.float32)
    q, pt, lens = bf16_dev(wl.q()), dev(wl.page_table), dev(wl.seq_lens.astype(np.int32))
    # the fused step (append of the new tokens + decode), then the plain decode
    kv.nvfp4kv_append_decode_attention(cache, bf16_dev(new[0]), bf16_dev(new[1]), dev(wl.append_slots()), q, out.t,
                                       pt, lens, wl.softmax_scale, ws.t)
    kv.nvfp4kv_decode_attention(cache, q, out.t, pt, lens, wl.softmax_scale, ws.t)
    torch.cuda.synchronize()
    assert np.isfinite(out.t.cpu().numpy()).all()
    for g in pools + [ws, out]:
        assert g.intact()


def test_extend_paths_stay_inside_their_outputs(cuda_lib):
    ew = inputs.extend_config(scale=1 / 32, num_layers=1)  # 16 x (512 prefix + 64 chunk), 64 q / 8 KV heads
    H = ew.num_kv_heads
    cache, pools = _guarded_cache(ew.num_pages, H)
    for b in range(ew.batch):
        k, v = ew.prefix_kv(0, b)
        gpu_append(cache, k, v, ew.slots(b, 0, ew.prefix_len))
    ks, vs = zip(*[ew.chunk_kv(0, b) for b in range(ew.batch)])
    kc, vc = bf16_dev(np.concatenate(ks)), bf16_dev(np.concatenate(vs))
    wk, wv = Guarded((ew.total_rows, H, 128), torch.uint8), Guarded((ew.total_rows, H, 128), torch.uint8)
    pt, pl, cu = dev(ew.page_table), dev(ew.prefix_lens), dev(ew.cu_prefix)
    rows, slots = dev(ew.chunk_ws_rows()), dev(ew.chunk_slots())
    kv.nvfp4kv_dequant_to_fp8_workspace(cache, pt, pl, cu, wk.t, wv.t)
    kv.nvfp4kv_bf16_to_fp8_workspace(kc, vc, rows, wk.t, wv.t)
    kv.nvfp4kv_quantize_append_fp8(cache, kc, vc, slots, rows, wk.t, wv.t)
    q = ew.q(0)
    out = Guarded((q.shape[0], ew.num_q_heads, 128), torch.float32)
    kv.nvfp4kv_extend_attention(bf16_dev(q), dev(ew.cu_q), ew.chunk_len, wk.t, wv.t, cu, pl, out.t, ew.softmax_scale)
    torch.cuda.synchronize()
    assert np.isfinite(out.t.cpu().numpy()).all()
    for g in pools + [wk, wv, out]:
        assert g.intact()


def test_calibration_and_variant_appends_stay_inside_their_outputs(cuda_lib):
    rng = np.random.default_rng(12)
    n, H, pages = 45, 2, 4
    k = inputs.bf16_bits(rng.standard_normal((n, H, 128)).astype(np.float32))
    v = inputs.bf16_bits(rng.standard_normal((n, H, 128)).astype(np.float32))
    slots = dev(rng.permutation(pages * 16)[:n].astype(np.int64))
    amax = Guarded((1,), torch.float32)
    kv.nvfp4kv_tensor_amax(bf16_dev(k).reshape(-1), amax.t)
    guards = [amax]
    rk = dev(inputs.rounding_bytes(4, n * H * 128).reshape(n, H, 128))
    for variant in (kv.NVFP4KV_VARIANT_SR, kv.NVFP4KV_VARIANT_HADAMARD, kv.NVFP4KV_VARIANT_MXFP4):
        cache, pools = _guarded_cache(pages, H, 4 if variant == kv.NVFP4KV_VARIANT_MXFP4 else 8)
        kv.nvfp4kv_quantize_append_variant(variant, cache, bf16_dev(k), bf16_dev(v), slots, rk, rk)
        guards += pools
    torch.cuda.synchronize()
    assert amax.t.item() == float(np.abs(inputs.bf16_bits_to_f32(k)).max())
    for g in guards:
        assert g.intact()
