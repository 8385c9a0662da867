"""Oracle extend (chunked prefill) over the FP8 workspace, pinned to library
routines, closed forms and invariants.

"nvfp4-kv-cache-memory-wall", section 3, item 2 and the data-flow figure: the
chunk attends over its cached prefix (dequantised into the FP8 workspace) and
over itself; the current tokens' own K/V take part as FP8.  Causal: chunk
token t of sequence b sees keys 0 .. prefix_lens[b] + t.
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_quantized_paged_quantize_gb300 import inputs


def _e4m3_f64(b):
    """E4M3 bytes -> float64 through torch's float8_e4m3fn dtype (independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _case_arrays(case):
    wk, wv = case.workspace()
    return wk, wv, case.q()


def _sdpa_reference(case, wk, wv, q, sk=1.0, sv=1.0):
    """torch scaled_dot_product_attention (float64) per sequence and KV head,
    with the causal-after-prefix mask written out as a boolean matrix."""
    G = case.num_q_heads // case.num_kv_heads
    out = np.zeros((case.total_q, case.num_q_heads, case.head_dim))
    kf, vf = _e4m3_f64(wk) * np.float32(sk), _e4m3_f64(wv) * np.float32(sv)
    qf = inputs.bf16_bits_to_f32(q).astype(np.float64)
    for b in range(case.batch):
        P, C = int(case.prefix_lens[b]), int(case.chunk_lens[b])
        r0, q0 = int(case.cu_prefix[b]), int(case.cu_q[b])
        keys = np.arange(P + C)
        mask = keys[None, :] <= (P + np.arange(C))[:, None]          # [C, P + C]
        for h in range(case.num_kv_heads):
            K = torch.from_numpy(kf[r0:r0 + P + C, h])[None]            # [1, L, d]
            V = torch.from_numpy(vf[r0:r0 + P + C, h])[None]
            Q = torch.from_numpy(qf[q0:q0 + C, h * G:(h + 1) * G]).permute(1, 0, 2)   # [G, C, d]
            o = torch.nn.functional.scaled_dot_product_attention(
                Q, K.expand(G, -1, -1), V.expand(G, -1, -1), attn_mask=torch.from_numpy(mask)[None],
                scale=case.softmax_scale)
            out[q0:q0 + C, h * G:(h + 1) * G] = o.permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("index", [1, 2, 3, 4])
def test_extend_attention_matches_sdpa(index):
    case = inputs.extend_attn_case(index)
    wk, wv, q = _case_arrays(case)
    got, st = oracle.extend_attention(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale)
    assert st == 0
    ref = _sdpa_reference(case, wk, wv, q)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_workspace_scales_multiply_keys_and_values():
    case = inputs.extend_attn_case(1)
    wk, wv, q = _case_arrays(case)
    got, st = oracle.extend_attention(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale,
                                      k_ws_scale=0.37, v_ws_scale=5.5)
    assert st == 0
    np.testing.assert_allclose(got, _sdpa_reference(case, wk, wv, q, 0.37, 5.5), rtol=1e-12, atol=1e-12)


def test_zero_query_is_mean_of_visible_values():
    # q = 0: uniform weights over exactly the P + t + 1 visible keys
    case = inputs.extend_attn_case(1)
    wk, wv, _ = _case_arrays(case)
    q = np.zeros((case.total_q, case.num_q_heads, case.head_dim), np.uint16)
    got, st = oracle.extend_attention(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale)
    assert st == 0
    vf = _e4m3_f64(wv)
    G = case.num_q_heads // case.num_kv_heads
    for b in range(case.batch):
        P, r0 = int(case.prefix_lens[b]), int(case.cu_prefix[b])
        for t in range(int(case.chunk_lens[b])):
            for h in range(case.num_q_heads):
                want = vf[r0:r0 + P + t + 1, h // G].mean(axis=0)
                np.testing.assert_allclose(got[case.cu_q[b] + t, h], want, rtol=1e-13, atol=1e-13)


def test_first_token_of_an_empty_prefix_returns_its_own_value():
    case = inputs.extend_attn_case(1)               # sequence 0 has no prefix
    wk, wv, q = _case_arrays(case)
    got, _ = oracle.extend_attention(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale)
    G = case.num_q_heads // case.num_kv_heads
    for h in range(case.num_q_heads):
        assert np.array_equal(got[0, h], _e4m3_f64(wv[0, h // G]))


def test_causal_extent():
    # changing key P + t changes token t's output; changing any later row does not
    case = inputs.extend_attn_case(1)
    wk, wv, q = _case_arrays(case)
    b, t = 2, 40
    P, r0, i = int(case.prefix_lens[b]), int(case.cu_prefix[b]), int(case.cu_q[b]) + t
    pairs = [(i, h) for h in range(case.num_q_heads)]
    base, _ = oracle.extend_attention_rows(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens,
                                           case.softmax_scale, pairs)
    for row, changes in ((r0 + P + t + 1, False), (case.total_rows - 1, False), (r0 + P + t, True), (r0, True)):
        k2, v2 = wk.copy(), wv.copy()
        k2[row] ^= 0x08                                 # flip one exponent bit of every value
        v2[row] ^= 0x08
        got, _ = oracle.extend_attention_rows(k2, v2, q, case.cu_q, case.cu_prefix, case.prefix_lens,
                                              case.softmax_scale, pairs)
        assert (not np.array_equal(got, base)) == changes, row


def test_prefix_order_does_not_matter():
    case = inputs.extend_attn_case(1)
    wk, wv, q = _case_arrays(case)
    base, _ = oracle.extend_attention(wk, wv, q, case.cu_q, case.cu_prefix, case.prefix_lens, case.softmax_scale)
    perm_k, perm_v = wk.copy(), wv.copy()
    for b in range(case.batch):
        r0, P = int(case.cu_prefix[b]), int(case.prefix_lens[b])
        p = np.random.default_rng(b).permutation(P)
        perm_k[r0:r0 + P] = wk[r0 + p]
        perm_v[r0:r0 + P] = wv[r0 + p]
    got, _ = oracle.extend_attention(perm_k, perm_v, q, case.cu_q, case.cu_prefix, case.prefix_lens,
                                     case.softmax_scale)
    np.testing.assert_allclose(got, base, rtol=1e-12, atol=1e-13)


def test_rows_outside_the_workspace_are_reported():
    case = inputs.extend_attn_case(1)
    wk, wv, q = _case_arrays(case)
    cu = case.cu_prefix.copy()
    cu[2] = case.total_rows - 10                        # sequence 2 runs past the end
    _, st = oracle.extend_attention(wk, wv, q, case.cu_q, cu, case.prefix_lens, case.softmax_scale)
    assert st == 1


# --------------------------------------------------------------------------
# the chunk's own K/V into the workspace: E4M3(fp32(x) / s_ws)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("s", [1.0, 0.37, 4.0, 1e-3])
def test_chunk_rows_are_the_e4m3_cast(s):
    # within E4M3's range the encoder equals torch's float8_e4m3fn cast of the
    # binary32 quotient (round to nearest even)
    rng = np.random.default_rng(4)
    n, H = 37, 2
    x = (rng.standard_normal((n, H, 128)) * 2.0 ** rng.integers(-12, 5, (n, H, 128))).astype(np.float32) * s
    k = inputs.bf16_bits(x)
    v = inputs.bf16_bits(-x)
    rows = np.arange(n, dtype=np.int64) * 2 + 1
    wk = np.zeros((2 * n + 1, H, 128), np.uint8)
    wv = np.zeros_like(wk)
    assert oracle.bf16_to_fp8_workspace(k, v, rows, wk, wv, s, s) == 0
    z = inputs.bf16_bits_to_f32(k) / np.float32(s)
    assert np.abs(z).max() < 448
    want = torch.from_numpy(z).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(wk[rows], want)
    want_v = torch.from_numpy(inputs.bf16_bits_to_f32(v) / np.float32(s)).to(torch.float8_e4m3fn)
    assert np.array_equal(wv[rows], want_v.view(torch.uint8).numpy())
    assert not wk[0::2].any() and not wv[0::2].any()    # rows not named stay untouched


def test_chunk_rows_saturate_keep_signs_and_skip_padding():
    vals = np.array([500.0, -1e6, 448.0, -0.0, -1e-5, 3e-3], np.float32)
    x = np.zeros((3, 1, 128), np.float32)
    x[:, 0, :6] = vals
    bits = inputs.bf16_bits(x)
    wk = np.full((3, 1, 128), 0xAA, np.uint8)
    wv = wk.copy()
    assert oracle.bf16_to_fp8_workspace(bits, bits, np.array([0, -1, 2]), wk, wv) == 0
    assert list(wk[0, 0, :6]) == [0x7E, 0xFE, 0x7E, 0x80, 0x80, 0x02]   # 448, -448, 448, -0, -0, 3 x 2^-9 (nearest)
    assert (wk[1] == 0xAA).all()                                       # padding row untouched
    assert oracle.bf16_to_fp8_workspace(bits, bits, np.array([0, 1, 3]), wk, wv) == 1   # row 3 is outside
