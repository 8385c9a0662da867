"""Glue shared by the GPU parity tests: move seeded inputs to the device, run
the CUDA library through its C ABI, and build the matching oracle state from
the same inputs.  Nothing here computes any of the method's arithmetic."""
import math

import numpy as np
import torch

import oracle
import nvfp4_quantized_paged_quantize_gb300 as kv

# max-abs error of each output row relative to that row's L2 norm
ATTN_TOL = 2e-3


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(bits):
    return dev(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16), torch.bfloat16)


def gpu_cache(num_pages, hkv, gk=1.0, gv=1.0):
    return kv.Cache.empty(num_pages, hkv, k_global_scale=gk, v_global_scale=gv, zero=True)


def status_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def gpu_append(cache, k_bits, v_bits, slots, status=None, chunk=1 << 16):
    """Quantise tokens into the GPU cache in chunks of `chunk` tokens."""
    n = k_bits.shape[0]
    for i in range(0, n, chunk):
        kv.nvfp4kv_quantize_append(cache, bf16_dev(k_bits[i:i + chunk]), bf16_dev(v_bits[i:i + chunk]),
                                   dev(np.asarray(slots[i:i + chunk], np.int64)), device_status=status)


def pool_host(cache):
    """The GPU pool as the oracle's flat row arrays (rows = page*Hkv*16 + h*16 + off)."""
    rows = cache.num_pages * cache.num_kv_heads * 16
    return tuple(t.reshape(rows, -1).cpu().numpy() for t in (cache.k_data, cache.v_data, cache.k_scale,
                                                               cache.v_scale))


def oracle_global_scales(wl, prompts, new=None):
    """(k, v) global scales by the oracle: 1, or the calibration over every K
    (every V) tensor of the workload."""
    pairs = wl.calibration_tensors(prompts, new)
    if not pairs:
        return 1.0, 1.0
    return tuple(oracle.calibrated_global_scale(max(oracle.tensor_amax(p[i]) for p in pairs)) for i in range(2))


def gpu_global_scales(wl, prompts, new=None):
    """(k, v) global scales through the library: nvfp4kv_tensor_amax folded
    over every K (every V) tensor on the device, then
    nvfp4kv_calibrated_global_scale of the two maxima."""
    pairs = wl.calibration_tensors(prompts, new)
    if not pairs:
        return 1.0, 1.0
    amax = torch.zeros(2, dtype=torch.float32, device="cuda")
    for p in pairs:
        for i in range(2):
            kv.nvfp4kv_tensor_amax(bf16_dev(p[i]).reshape(-1), amax[i:i + 1], accumulate=True)
    a = amax.cpu().tolist()
    return kv.nvfp4kv_calibrated_global_scale(a[0]), kv.nvfp4kv_calibrated_global_scale(a[1])


def fill_workload_gpu(wl, prompts, new=None, status=None):
    """GPU cache holding every sequence's prompt (and the appended token)."""
    gk, gv = gpu_global_scales(wl, prompts, new)
    cache = gpu_cache(wl.num_pages, wl.num_kv_heads, gk, gv)
    for b in range(wl.batch):
        k, v = prompts[b]
        if k.shape[0]:
            gpu_append(cache, k, v, wl.slots(b, 0, k.shape[0]), status)
    if wl.append:
        new = new if new is not None else wl.new_kv()
        gpu_append(cache, new[0], new[1], wl.append_slots(), status)
    return cache


def fill_workload_oracle(wl, prompts, new=None):
    gk, gv = oracle_global_scales(wl, prompts, new)
    c = oracle.Cache(wl.num_pages, wl.num_kv_heads, 128, 16, gk, gv)
    for b in range(wl.batch):
        k, v = prompts[b]
        if k.shape[0]:
            assert oracle.quantize_append(c, k, v, wl.slots(b, 0, k.shape[0])) == 0
    if wl.append:
        new = new if new is not None else wl.new_kv()
        assert oracle.quantize_append(c, new[0], new[1], wl.append_slots()) == 0
    return c


def oracle_pair(wl, b, h, k_seq, v_seq, q_bits, gk, gv):
    """Oracle decode of one (sequence, KV head): a one-head oracle cache with a
    compact page table, filled from the same bf16 inputs.

    k_seq, v_seq: [L, Hkv, d] bits of the whole sequence (prompt + appended).
    Returns (out [G, d] float64, oracle cache, np pages)."""
    L = k_seq.shape[0]
    npg = (L + 15) // 16
    c = oracle.Cache(max(npg, 1), 1, 128, 16, gk, gv)
    t = np.arange(L, dtype=np.int64)
    assert oracle.quantize_append(c, np.ascontiguousarray(k_seq[:, h:h + 1]),
                                  np.ascontiguousarray(v_seq[:, h:h + 1]), t) == 0
    G = wl.num_q_heads // wl.num_kv_heads
    q = np.ascontiguousarray(q_bits[b:b + 1, h * G:(h + 1) * G])
    pt = np.arange(max(npg, 1), dtype=np.int32)[None, :]
    out, st = oracle.decode_attention(c, q, pt, np.array([L], np.int32), wl.softmax_scale)
    assert st == 0
    return out[0], c, npg


def check_rows(got, ref, tol=ATTN_TOL):
    """Per-row max |got - ref| <= tol * ||ref||_2; returns the worst ratio."""
    got = np.asarray(got, np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, ref.shape[-1])
    err = np.abs(got - ref).max(axis=1)
    norm = np.linalg.norm(ref, axis=1)
    ratio = np.where(norm > 0, err / np.where(norm > 0, norm, 1), err)
    worst = float(ratio.max()) if ratio.size else 0.0
    assert np.all(np.isfinite(got)), "non-finite output"
    assert worst <= tol, f"worst row error {worst:.3e} > {tol}"
    return worst


def decode_gpu(wl, cache, q_bits, status=None, workspace=None, out=None):
    B, Hq = wl.batch, wl.num_q_heads
    if workspace is None:
        n = kv.nvfp4kv_decode_workspace_size(cache, B, Hq)
        workspace = torch.zeros(n, dtype=torch.uint8, device="cuda")
    if out is None:
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    kv.nvfp4kv_decode_attention(cache, bf16_dev(q_bits), out, dev(wl.page_table),
                                dev(wl.seq_lens.astype(np.int32)), wl.softmax_scale, workspace,
                                device_status=status)
    return out, workspace


def softmax_scale(d=128):
    return 1.0 / math.sqrt(d)
