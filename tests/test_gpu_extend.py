"""Extend over the FP8 workspace on the GPU against the oracle.

"nvfp4-kv-cache-memory-wall", section 3, item 2 and the data-flow figure.
The chunk -> workspace conversion must match the oracle bit for bit; the
attention output row by row within ATTN_TOL of the row's L2 norm (f16
operands that hold the E4M3 values exactly, f16 probabilities, f32
accumulation; q rounded to f16 -- exact for the workloads' magnitudes).
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_quantized_paged_quantize_gb300 as kv
from nvfp4_quantized_paged_quantize_gb300 import inputs
from gpu_util import bf16_dev, check_rows, dev, gpu_append, gpu_cache, pool_host, status_word

pytestmark = pytest.mark.gpu


def _u8(a):
    return dev(np.ascontiguousarray(a, np.uint8))


def _extend_gpu(case_like, wk, wv, q_bits, max_q_len=None, sk=1.0, sv=1.0, status=None, cu_prefix=None):
    total_q, hq = q_bits.shape[0], q_bits.shape[1]
    out = torch.full((total_q, hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    cu_p = case_like.cu_prefix if cu_prefix is None else cu_prefix
    mq = int(np.diff(case_like.cu_q).max()) if max_q_len is None else max_q_len
    kv.nvfp4kv_extend_attention(bf16_dev(q_bits), dev(np.asarray(case_like.cu_q, np.int64)), mq, wk, wv,
                                dev(np.asarray(cu_p, np.int64)), dev(np.asarray(case_like.prefix_lens, np.int32)),
                                out, case_like.softmax_scale, sk, sv, device_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy()


# --------------------------------------------------------------------------
# chunk rows -> workspace
# --------------------------------------------------------------------------

@pytest.mark.parametrize("sk,sv", [(1.0, 1.0), (0.37, 5.5), (1e-3, 2.0 ** -20), (3e30, 1e-30)])
def test_chunk_rows_bit_exact(cuda_lib, sk, sv):
    rng = np.random.default_rng(17)
    n, H, rows = 301, 8, 700
    x = (rng.standard_normal((n, H, 128)) * 2.0 ** rng.integers(-30, 30, (n, H, 128))).astype(np.float32)
    k, v = inputs.bf16_bits(x), inputs.bf16_bits(x[::-1].copy() * 3)
    k[5, 3, :8] = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x0001, 0x8001, 0x7F7F, 0x3F80], np.uint16)  # +-0, +-inf, subnormals, max
    ws_rows = rng.permutation(rows)[:n].astype(np.int64)
    ws_rows[::37] = -1                                                 # padding tokens
    ok, ov = (np.full((rows, H, 128), 0x5A, np.uint8) for _ in range(2))
    assert oracle.bf16_to_fp8_workspace(k, v, ws_rows, ok, ov, sk, sv) == 0
    gk, gv = _u8(np.full((rows, H, 128), 0x5A)), _u8(np.full((rows, H, 128), 0x5A))
    st = status_word()
    kv.nvfp4kv_bf16_to_fp8_workspace(bf16_dev(k), bf16_dev(v), dev(ws_rows), gk, gv, sk, sv, device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(gk.cpu().numpy(), ok) and np.array_equal(gv.cpu().numpy(), ov)


def test_chunk_row_outside_workspace_flagged(cuda_lib):
    k = inputs.bf16_bits(np.ones((3, 2, 128), np.float32))
    wk, wv = _u8(np.zeros((4, 2, 128))), _u8(np.zeros((4, 2, 128)))
    st = status_word()
    kv.nvfp4kv_bf16_to_fp8_workspace(bf16_dev(k), bf16_dev(k), dev(np.array([0, 4, 3], np.int64)), wk, wv,
                                     device_status=st)
    torch.cuda.synchronize()
    assert st.item() & kv.NVFP4KV_DEVERR_ROW
    got = wk.cpu().numpy()
    assert (got[0] == 0x38).all() and (got[3] == 0x38).all() and not got[1:3].any()   # 1.0 = 0x38


# --------------------------------------------------------------------------
# extend attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("index", [1, 2, 3, 4])
def test_extend_attention_matches_oracle(cuda_lib, index):
    case = inputs.extend_attn_case(index)
    wk, wv = case.workspace()
    q = case.q()
    ref, st = oracle.extend_attention(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale)
    assert st == 0
    status = status_word()
    got = _extend_gpu(case, _u8(wk), _u8(wv), q, status=status)
    assert status.item() == 0
    check_rows(got, ref)


def test_extend_attention_workspace_scales(cuda_lib):
    case = inputs.extend_attn_case(2)
    wk, wv = case.workspace()
    q = case.q()
    ref, _ = oracle.extend_attention(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale,
                                     k_ws_scale=0.37, v_ws_scale=5.5)
    check_rows(_extend_gpu(case, _u8(wk), _u8(wv), q, sk=0.37, sv=5.5), ref)


def test_extend_attention_sharp_scores_and_empty_chunks(cuda_lib):
    # large K magnitudes (scores of hundreds: the lazy running max must move), a
    # sequence with no new tokens and one whose only token has no prefix
    case = inputs.ExtendAttnCase("extend_attn_sharp", inputs.BASE_SEED + 150, np.array([300, 64, 0], np.int32),
                                 np.array([40, 0, 1], np.int32), 16, 2, k_exp=(6, 13), v_exp=(3, 9))
    wk, wv = case.workspace()
    q = case.q()
    ref, _ = oracle.extend_attention(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale)
    got = _extend_gpu(case, _u8(wk), _u8(wv), q, max_q_len=200)   # a generous max_q_len: extra tiles leave
    check_rows(got, ref)


def test_extend_attention_rows_outside_workspace_flagged(cuda_lib):
    case = inputs.extend_attn_case(1)
    wk, wv = case.workspace()
    cu = case.cu_prefix.copy()
    cu[2] = case.total_rows - 10                      # sequence 2 runs past the end
    st = status_word()
    got = _extend_gpu(case, _u8(wk), _u8(wv), case.q(), status=st, cu_prefix=cu)
    assert st.item() & kv.NVFP4KV_DEVERR_ROW
    assert np.isfinite(got[: case.cu_q[2]]).all()   # the other sequences are still computed


def _pipeline(ew, layer, pairs_per_seq, rng):
    """One extend layer through the library (quantize the prefix, dequantize it
    into the workspace, add the chunk rows, attend) and through the oracle;
    returns (workspace bytes equal, worst row error on sampled rows)."""
    H = ew.num_kv_heads
    g = gpu_cache(ew.num_pages, H)
    o = oracle.Cache(ew.num_pages, H, 128, 16)
    for b in range(ew.batch):
        k, v = ew.prefix_kv(layer, b)
        gpu_append(g, k, v, ew.slots(b, 0, ew.prefix_len))
        assert oracle.quantize_append(o, k, v, ew.slots(b, 0, ew.prefix_len)) == 0
    ks, vs = zip(*[ew.chunk_kv(layer, b) for b in range(ew.batch)])
    kc, vc = np.concatenate(ks), np.concatenate(vs)
    rows = ew.chunk_ws_rows()
    wk = torch.zeros((ew.total_rows, H, 128), dtype=torch.uint8, device="cuda")
    wv = torch.zeros_like(wk)
    pt, pl, cu = dev(ew.page_table), dev(ew.prefix_lens), dev(ew.cu_prefix)
    kv.nvfp4kv_dequant_to_fp8_workspace(g, pt, pl, cu, wk, wv)
    kv.nvfp4kv_bf16_to_fp8_workspace(bf16_dev(kc), bf16_dev(vc), dev(rows), wk, wv)
    q = ew.q(layer)
    out = torch.empty((q.shape[0], ew.num_q_heads, 128), dtype=torch.float32, device="cuda")
    st = status_word()
    kv.nvfp4kv_extend_attention(bf16_dev(q), dev(ew.cu_q), ew.chunk_len, wk, wv, cu, pl, out, ew.softmax_scale,
                                device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    owk, owv, ost = oracle.dequant_to_fp8_workspace(o, ew.page_table, ew.prefix_lens, ew.cu_prefix, ew.total_rows)
    assert ost == 0
    assert oracle.bf16_to_fp8_workspace(kc, vc, rows, owk, owv) == 0
    same = np.array_equal(wk.cpu().numpy(), owk) and np.array_equal(wv.cpu().numpy(), owv)
    # sampled rows: every sequence, its first and last token and random ones, random heads
    pairs = []
    for b in range(ew.batch):
        ts = {0, ew.chunk_len - 1} | set(rng.integers(0, ew.chunk_len, pairs_per_seq).tolist())
        pairs += [(int(ew.cu_q[b] + t), int(rng.integers(0, ew.num_q_heads))) for t in sorted(ts)]
    ref, rst = oracle.extend_attention_rows(owk, owv, q, ew.cu_q, ew.cu_prefix, ew.prefix_lens, ew.softmax_scale,
                                            pairs)
    assert rst == 0
    got = out.cpu().numpy()[[p[0] for p in pairs], [p[1] for p in pairs]]
    return same, check_rows(got, ref)


def test_extend_layer_pipeline_small(cuda_lib):
    # the extend workload at 1/16 of its lengths (prefix 1024, chunk 128)
    same, _ = _pipeline(inputs.extend_config(scale=1 / 16, num_layers=2), 1, 6, np.random.default_rng(1))
    assert same


def test_extend_layer_full_size_sampled(cuda_lib):
    # one layer at full size (16 x (16384 prefix + 2048 chunk), 64 / 8 heads), as the bench times it
    same, _ = _pipeline(inputs.extend_config(num_layers=1), 0, 3, np.random.default_rng(2))
    assert same


# --------------------------------------------------------------------------
# the fused write: NVFP4 cache rows and FP8 workspace rows in one pass
# --------------------------------------------------------------------------

@pytest.mark.parametrize("sk,sv", [(1.0, 1.0), (0.37, 5.5)])
def test_fused_write_matches_oracle(cuda_lib, sk, sv):
    rng = np.random.default_rng(23)
    n, H, pages, rows = 333, 4, 40, 500
    x = (rng.standard_normal((n, H, 128)) * 2.0 ** rng.integers(-8, 8, (n, H, 128))).astype(np.float32)
    k, v = inputs.bf16_bits(x), inputs.bf16_bits(x[::-1].copy() * 0.5)
    slots = rng.permutation(pages * 16)[:n].astype(np.int64)
    slots[::41] = -1                                      # padding tokens
    slots[7] = pages * 16 + 3                             # outside the pool
    ws_rows = rng.permutation(rows)[:n].astype(np.int64)
    ws_rows[::29] = -1
    ws_rows[11] = rows                                    # outside the workspace
    g = gpu_cache(pages, H, 0.37, 2.5)
    wk, wv = _u8(np.full((rows, H, 128), 0x5A)), _u8(np.full((rows, H, 128), 0x5A))
    st = status_word()
    kv.nvfp4kv_quantize_append_fp8(g, bf16_dev(k), bf16_dev(v), dev(slots), dev(ws_rows), wk, wv, sk, sv,
                                   device_status=st)
    torch.cuda.synchronize()
    assert st.item() & kv.NVFP4KV_DEVERR_SLOT and st.item() & kv.NVFP4KV_DEVERR_ROW
    o = oracle.Cache(pages, H, 128, 16, 0.37, 2.5)
    assert oracle.quantize_append(o, k, v, slots) != 0   # the out-of-pool slot is reported
    owk, owv = (np.full((rows, H, 128), 0x5A, np.uint8) for _ in range(2))
    assert oracle.bf16_to_fp8_workspace(k, v, ws_rows, owk, owv, sk, sv) != 0
    for got, want in zip(pool_host(g), (o.k_data, o.v_data, o.k_scale, o.v_scale)):
        assert np.array_equal(got, want)
    assert np.array_equal(wk.cpu().numpy(), owk) and np.array_equal(wv.cpu().numpy(), owv)


def test_initial_prefill_through_the_fused_write(cuda_lib):
    # prompts {1, 77, 300}: one pass writes the NVFP4 cache and the FP8 rows,
    # then the extend attention runs with empty prefixes
    case = inputs.ExtendAttnCase("prefill", inputs.BASE_SEED + 160, np.zeros(3, np.int32),
                                 np.array([1, 77, 300], np.int32), 16, 2, gap=0)
    rng = np.random.default_rng(5)
    n, H = case.total_q, case.num_kv_heads
    k = inputs.bf16_bits((rng.standard_normal((n, H, 128)) * 0.5).astype(np.float32))
    v = inputs.bf16_bits(rng.standard_normal((n, H, 128)).astype(np.float32))
    q = case.q()
    pages = (n + 15) // 16 + 3
    slots = rng.permutation(pages * 16)[:n].astype(np.int64)
    ws_rows = np.arange(n, dtype=np.int64)                # cu_prefix == cu_q: each prompt's rows in order
    g = gpu_cache(pages, H)
    wk = torch.zeros((case.total_rows, H, 128), dtype=torch.uint8, device="cuda")
    wv = torch.zeros_like(wk)
    kv.nvfp4kv_quantize_append_fp8(g, bf16_dev(k), bf16_dev(v), dev(slots), dev(ws_rows), wk, wv)
    got = _extend_gpu(case, wk, wv, q)
    o = oracle.Cache(pages, H, 128, 16)
    assert oracle.quantize_append(o, k, v, slots) == 0
    owk, owv = (np.zeros((case.total_rows, H, 128), np.uint8) for _ in range(2))
    assert oracle.bf16_to_fp8_workspace(k, v, ws_rows, owk, owv) == 0
    for gg, want in zip(pool_host(g), (o.k_data, o.v_data, o.k_scale, o.v_scale)):
        assert np.array_equal(gg, want)
    assert np.array_equal(wk.cpu().numpy(), owk)
    ref, st = oracle.extend_attention(owk, owv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale)
    assert st == 0
    check_rows(got, ref)


def test_extend_layer_79_pipeline(cuda_lib):
    # the last of the 80 layers (its own seeds), at 1/32 of the lengths
    same, _ = _pipeline(inputs.extend_config(scale=1 / 32, num_layers=80), 79, 4, np.random.default_rng(79))
    assert same
