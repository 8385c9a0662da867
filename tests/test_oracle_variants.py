"""Oracle format variants the pages compare with NVFP4, pinned, and their RMSE.

- MXFP4: 32-value blocks with a power-of-two (E8M0) scale ("NVIDIA NVFP4: LLM
  memory doubled, inference 3x", figure 6; "NVFP4: breaking the memory wall",
  technical breakdown).
- Stochastic rounding of the E2M1 codes ("NVFP4: breaking the memory wall",
  quantisation techniques: 2.3 -> 2 with 70 %, -> 3 with 30 %).
- The orthonormal Walsh-Hadamard rotation before quantisation (same page).
"""
import math

import numpy as np
import pytest

import oracle
from conftest import read_golden
from nvfp4_quantized_paged_quantize_gb300 import inputs

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _nearest_e2m1(y):
    """Brute-force nearest E2M1 code (ties to the even code, saturating, sign kept)."""
    m = abs(y)
    if m >= 6.0:
        c = 7
    else:
        d = [abs(m - v) for v in E2M1]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        c = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
    return c | (8 if math.copysign(1.0, y) < 0 else 0)


# --------------------------------------------------------------------------
# MXFP4
# --------------------------------------------------------------------------

def test_e8m0_is_a_power_of_two():
    for code in (0, 1, 100, 127, 128, 254):
        assert oracle.e8m0_value(code) == 2.0 ** (code - 127)
    assert math.isnan(oracle.e8m0_value(0xFF))


def test_mxfp4_scale_and_elements_by_brute_force():
    rng = np.random.default_rng(31)
    for _ in range(300):
        x = (rng.standard_normal(32) * 2.0 ** rng.integers(-20, 20)).astype(np.float32)
        packed, sc = oracle.mxfp4_quantize_block(x)
        amax = float(np.abs(x).max())
        e = math.frexp(amax)[1] - 1 - 2                  # floor(log2 amax) - E2M1's largest exponent
        assert sc == e + 127
        codes = np.stack([packed & 0xF, packed >> 4], -1).reshape(-1)
        for xi, ci in zip(x, codes):
            assert ci == _nearest_e2m1(float(xi) / 2.0 ** e)
        assert 4.0 <= amax / 2.0 ** e < 8.0               # so the block's amax maps to 4 or 6


def test_mxfp4_zero_block_and_on_grid_round_trip():
    packed, sc = oracle.mxfp4_quantize_block(np.zeros(32, np.float32))
    assert sc == 0 and not packed.any()
    rng = np.random.default_rng(2)
    for k in (-10, 0, 7):
        vals = np.array(E2M1)[rng.integers(0, 8, 32)] * np.where(rng.random(32) < 0.5, -1, 1)
        vals[3] = 6.0                                     # amax 6 * 2^k: the scale is 2^k
        x = (vals * 2.0 ** k).astype(np.float32)
        packed, sc = oracle.mxfp4_quantize_block(x)
        assert sc == k + 127
        codes = np.stack([packed & 0xF, packed >> 4], -1).reshape(-1)
        got = [oracle.mxfp4_dequant_value(int(c), sc) for c in codes]
        assert np.array_equal(np.array(got), x.astype(np.float64))


# --------------------------------------------------------------------------
# stochastic rounding
# --------------------------------------------------------------------------

def test_sr_reproduces_the_pages_example():
    (row,) = read_golden("page_stochastic_rounding_example.txt")
    y, lo, hi, p_lo, p_hi = (float(v) for v in row)
    ups = sum(oracle.e2m1_value(oracle.e2m1_encode_sr(y, r)) == hi for r in range(256))
    downs = sum(oracle.e2m1_value(oracle.e2m1_encode_sr(y, r)) == lo for r in range(256))
    assert ups + downs == 256
    assert abs(ups / 256 - p_hi) <= 1 / 256 and abs(downs / 256 - p_lo) <= 1 / 256


def test_sr_is_unbiased_and_picks_a_neighbour():
    # over the 256 random bytes the mean equals y to within the byte's resolution
    rng = np.random.default_rng(9)
    ys = np.concatenate([rng.uniform(0, 6, 400), np.array(E2M1[:-1]) + 1e-3]).astype(np.float32)
    for y in ys:
        vals = np.array([oracle.e2m1_value(oracle.e2m1_encode_sr(float(y), r)) for r in range(256)])
        lo = max(v for v in E2M1 if v <= y)
        hi = min(v for v in E2M1 if v > y)
        assert set(vals) <= {lo, hi}
        assert abs(vals.mean() - float(y)) <= (hi - lo) / 512 + 1e-12


def test_sr_grid_values_signs_and_saturation():
    for c, v in enumerate(E2M1):
        for r in (0, 77, 255):
            assert oracle.e2m1_encode_sr(v, r) == c
            assert oracle.e2m1_encode_sr(-v, r) == c | 8
    for r in (0, 255):
        assert oracle.e2m1_encode_sr(6.5, r) == 7 and oracle.e2m1_encode_sr(-1e9, r) == 15
        assert oracle.e2m1_encode_sr(-0.1, r) in (8, 9)


def test_sr_block_keeps_the_scale_and_moves_codes_at_most_one_step():
    rng = np.random.default_rng(4)
    for _ in range(200):
        x = (rng.standard_normal(16) * 2.0 ** rng.integers(-6, 6)).astype(np.float32)
        g = float(np.float32(2.0 ** rng.uniform(-4, 4)))
        r = rng.integers(0, 256, 16).astype(np.uint8)
        p_rne, s_rne = oracle.quantize_block(x, g)
        p_sr, s_sr = oracle.quantize_block_sr(x, g, r)
        assert s_sr == s_rne
        c_rne = np.stack([p_rne & 0xF, p_rne >> 4], -1).reshape(-1).astype(int)
        c_sr = np.stack([p_sr & 0xF, p_sr >> 4], -1).reshape(-1).astype(int)
        assert np.all(np.abs((c_sr & 7) - (c_rne & 7)) <= 1)


# --------------------------------------------------------------------------
# Hadamard rotation
# --------------------------------------------------------------------------

def _hadamard_matrix(n):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    return scipy_linalg.hadamard(n).astype(np.float64) / math.sqrt(n)


@pytest.mark.parametrize("n", [2, 16, 128])
def test_hadamard_matches_the_matrix(n):
    rng = np.random.default_rng(n)
    H = _hadamard_matrix(n)
    for _ in range(20):
        x = (rng.standard_normal(n) * 2.0 ** rng.integers(-8, 8)).astype(np.float32)
        y = oracle.hadamard(x).astype(np.float64)
        ref = H @ x.astype(np.float64)
        # log2(n) binary32 passes and one scaling: a few ulps of the vector norm
        assert np.abs(y - ref).max() <= (math.log2(n) + 2) * 2.0 ** -23 * np.linalg.norm(x)


def test_hadamard_is_orthonormal_and_self_inverse():
    rng = np.random.default_rng(3)
    q = rng.standard_normal(128).astype(np.float32)
    k = rng.standard_normal(128).astype(np.float32)
    hq, hk = oracle.hadamard(q), oracle.hadamard(k)
    assert abs(float(np.linalg.norm(hq)) - float(np.linalg.norm(q))) <= 1e-5 * float(np.linalg.norm(q))
    assert abs(float(hq.astype(np.float64) @ hk) - float(q.astype(np.float64) @ k)) <= 1e-4
    np.testing.assert_allclose(oracle.hadamard(hq), q, rtol=0, atol=1e-5)


def test_hadamard_spreads_an_outlier():
    # the page's idea: one large value among small ones is spread over the
    # vector; with small values of random sign every entry carries the
    # outlier's share 5 / sqrt(128) = 0.44 (plus at most 0.1 * 127 / sqrt(128)
    # of the rest in the worst case, far less here) and the peak falls
    x = (0.1 * np.where(np.random.default_rng(6).random(128) < 0.5, -1, 1)).astype(np.float32)
    x[5] = 5.0
    y = np.abs(oracle.hadamard(x))
    assert y.max() < 5.0 / 4 and y.min() > 0.1


# --------------------------------------------------------------------------
# RMSE report: NVFP4 against its variants on the workloads' data
# --------------------------------------------------------------------------

def _workload_values(index, n):
    wl = inputs.decode_config(index, 1 / 64)
    k, _ = wl.prompt_kv(0)
    x = inputs.bf16_bits_to_f32(k).reshape(-1)
    return x[: n - n % 128]


@pytest.mark.parametrize("name,x", [
    ("8K workload K (N(0, 0.02) + 6.0 outliers)", lambda: _workload_values(2, 32768)),
    ("ragged workload K (Student-t(4) x 0.05)", lambda: _workload_values(4, 32768)),
    ("page demo (gauss 0.02 + 8 x 6.0)", lambda: np.array(inputs.page_demo_values(), np.float32)),
])
def test_rmse_report_variants(name, x, capsys):
    x = x()
    r = inputs.rounding_bytes(1, x.shape[0])
    rm = {v: float(np.sqrt(np.mean((oracle.fake_quant(x, v, rand=r) - x.astype(np.float64)) ** 2)))
          for v in ("nvfp4", "mxfp4", "nvfp4_sr", "nvfp4_hadamard")}
    bias = {v: float(np.mean(oracle.fake_quant(x, v, rand=r) - x.astype(np.float64))) for v in ("nvfp4", "nvfp4_sr")}
    with capsys.disabled():
        print(f"\n{name}: RMSE " + ", ".join(f"{k} {v:.4g}" for k, v in rm.items()) +
              f"; mean error nvfp4 {bias['nvfp4']:.2e}, nvfp4_sr {bias['nvfp4_sr']:.2e}")
    assert rm["mxfp4"] > rm["nvfp4"]                   # the pages: NVFP4's finer, E4M3-scaled blocks win
    assert rm["nvfp4_sr"] >= rm["nvfp4"]               # stochastic rounding trades RMSE for no bias


# --------------------------------------------------------------------------
# decode over a variant's cache
# --------------------------------------------------------------------------

from variant_util import HADAMARD, MXFP4, SR, oracle_variant_pools  # noqa: E402


def _variant_cache(wl, variant, b_count=None, rk=None, rv=None):
    """An oracle cache holding the first b_count sequences of a decode workload (prompt + new token)."""
    prompts = wl.all_prompt_kv()
    new_k, new_v = wl.new_kv()
    B = wl.batch if b_count is None else b_count
    ks, vs, ss = [], [], []
    for b in range(B):
        k, v = prompts[b]
        ks += [k, new_k[b:b + 1]]
        vs += [v, new_v[b:b + 1]]
        ss += [wl.slots(b, 0, k.shape[0]), wl.append_slots()[b:b + 1]]
    k, v, slots = np.concatenate(ks), np.concatenate(vs), np.concatenate(ss)
    pools = oracle_variant_pools(variant, k, v, slots, wl.num_pages, wl.num_kv_heads, 1.0, 1.0, rk, rv)
    c = oracle.Cache(wl.num_pages, wl.num_kv_heads, 128, 16,
                     arrays=(pools["k"][0], pools["v"][0], pools["k"][1], pools["v"][1]))
    return c, k, v, slots


def _sdpa(q, K, V, scale):
    import torch

    G = q.shape[0] // K.shape[0]
    out = np.zeros_like(q)
    for h in range(K.shape[0]):
        Q = torch.from_numpy(q[h * G:(h + 1) * G])[:, None, :]              # [G, 1, d]
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, torch.from_numpy(K[h])[None].expand(G, -1, -1), torch.from_numpy(V[h])[None].expand(G, -1, -1),
            scale=scale)
        out[h * G:(h + 1) * G] = o[:, 0, :].numpy()
    return out


def _dequant_rows(c, which, fmt):
    """Every pool row in fp64, decoded here without the oracle: E2M1 from the
    pages' value list, E4M3 through torch's float8_e4m3fn, E8M0 as 2^(s - 127)."""
    import torch

    vals = np.array(E2M1 + [-v for v in E2M1])
    data = c.k_data if which == "k" else c.v_data
    scl = c.k_scale if which == "k" else c.v_scale
    codes = np.stack([data & 0xF, data >> 4], -1).reshape(data.shape[0], -1)
    x = vals[codes]
    if fmt == oracle.FORMAT_MXFP4:
        return x * np.repeat(2.0 ** (scl.astype(np.float64) - 127), 32, axis=1)
    sc = torch.from_numpy(np.ascontiguousarray(scl)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    x = x * np.repeat(sc, 16, axis=1)
    if fmt == oracle.FORMAT_NVFP4_HADAMARD:
        x = x @ _hadamard_matrix(128)                                       # symmetric, its own inverse
    return x


@pytest.mark.parametrize("fmt,variant", [(oracle.FORMAT_NVFP4, None), (oracle.FORMAT_NVFP4_HADAMARD, HADAMARD),
                                         (oracle.FORMAT_MXFP4, MXFP4)])
def test_variant_decode_matches_sdpa(fmt, variant):
    wl = inputs.decode_config(1)                           # B = 2, lengths {101, 258}, 8 q / 2 KV heads
    if variant is None:
        c = oracle.Cache(wl.num_pages, wl.num_kv_heads)
        for b, (k, v) in enumerate(wl.all_prompt_kv()):
            oracle.quantize_append(c, k, v, wl.slots(b, 0, k.shape[0]))
        nk, nv = wl.new_kv()
        oracle.quantize_append(c, nk, nv, wl.append_slots())
    else:
        c, _, _, _ = _variant_cache(wl, variant)
    q = wl.q()
    got, st = oracle.decode_attention_format(c, fmt, q, wl.page_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    if fmt == oracle.FORMAT_NVFP4:
        same, _ = oracle.decode_attention(c, q, wl.page_table, wl.seq_lens, wl.softmax_scale)
        assert np.array_equal(got, same)
    Kr, Vr = _dequant_rows(c, "k", fmt), _dequant_rows(c, "v", fmt)
    qf = inputs.bf16_bits_to_f32(q).astype(np.float64)
    H = wl.num_kv_heads
    for b in range(wl.batch):
        L = int(wl.seq_lens[b])
        t = np.arange(L)
        slot = wl.page_table[b, t // 16].astype(np.int64) * 16 + t % 16
        rows = ((slot // 16)[None, :] * H + np.arange(H)[:, None]) * 16 + (slot % 16)[None, :]   # [H, L]
        ref = _sdpa(qf[b], Kr[rows], Vr[rows], wl.softmax_scale)
        np.testing.assert_allclose(got[b], ref, rtol=1e-10, atol=1e-10)


def test_attention_error_report_variants(capsys):
    # decode attention over each variant's cache against attention over the
    # unquantised bf16 K/V (8K workload's values, 3 sequences of 129 tokens)
    wl = inputs.decode_config(2, 1 / 64)
    B = 3
    q = wl.q()[:B]
    rows_k = inputs.rounding_bytes(20, 10 ** 6)
    errs = {}
    for name, fmt, variant in (("nvfp4", oracle.FORMAT_NVFP4, 0), ("mxfp4", oracle.FORMAT_MXFP4, MXFP4),
                               ("nvfp4_sr", oracle.FORMAT_NVFP4, SR),
                               ("nvfp4_hadamard", oracle.FORMAT_NVFP4_HADAMARD, HADAMARD)):
        n = sum(int(l) for l in wl.seq_lens[:B])
        rk = rows_k[: n * wl.num_kv_heads * 128].reshape(n, wl.num_kv_heads, 128)
        rv = rows_k[-n * wl.num_kv_heads * 128:].reshape(n, wl.num_kv_heads, 128)
        c, k, v, slots = _variant_cache(wl, variant, B, rk, rv)
        got, st = oracle.decode_attention_format(c, fmt, q, wl.page_table[:B], wl.seq_lens[:B], wl.softmax_scale)
        assert st == 0
        # exact attention over the bf16 values, gathered in token order
        kf, vf = inputs.bf16_bits_to_f32(k).astype(np.float64), inputs.bf16_bits_to_f32(v).astype(np.float64)
        qf = inputs.bf16_bits_to_f32(q).astype(np.float64)
        rel, start = [], 0
        for b in range(B):
            L = int(wl.seq_lens[b])
            toks = np.concatenate([np.arange(start, start + L - 1), [start + L - 1]])
            ref = _sdpa(qf[b], kf[toks].transpose(1, 0, 2), vf[toks].transpose(1, 0, 2), wl.softmax_scale)
            rel.append(np.abs(got[b] - ref).max(axis=-1) / np.linalg.norm(ref, axis=-1))
            start += L
        errs[name] = float(np.mean(np.concatenate(rel)))
    with capsys.disabled():
        print("\nattention error vs bf16 K/V (mean over rows of max-abs / row norm): " +
              ", ".join(f"{k} {v:.3e}" for k, v in errs.items()))
    assert errs["mxfp4"] > errs["nvfp4"]
