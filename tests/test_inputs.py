"""The seeded input recipe: what the generators promise, checked.

The workloads follow the pages' shapes ("nvfp4-kv-cache-memory-wall",
section 1: 80 layers x 8 KV heads x 128; section 2: values mostly ~0.02 with
6.0 outliers).  These checks hold the generators to that recipe and to their
determinism (any sequence can be regenerated on its own).
"""
import numpy as np

from nvfp4_quantized_paged_quantize_gb300 import inputs


def test_sequences_regenerate_independently():
    a, b = inputs.decode_config(2, 1 / 64), inputs.decode_config(2, 1 / 64)
    k1, v1 = a.prompt_kv(3)
    k2, v2 = b.prompt_kv(3)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    k0, _ = a.prompt_kv(0)
    assert not np.array_equal(k0, k1)
    assert np.array_equal(a.q(), b.q()) and np.array_equal(a.page_table, b.page_table)


def test_headline_outliers_are_eight_per_4096_values():
    wl = inputs.decode_config(2, 1 / 16)                   # 512-token prompts: 8 x 128 values per token
    k, _ = wl.prompt_kv(0)
    x = inputs.bf16_bits_to_f32(k).reshape(-1)
    x = x[: x.size - x.size % 4096].reshape(-1, 4096)
    assert ((x == 6.0).sum(axis=1) == 8).all()
    rest = x[x != 6.0]
    assert abs(float(rest.std()) - 0.02) < 0.002 and abs(float(rest.mean())) < 0.001


def test_page_tables_are_permutations_of_the_pool():
    for index in (1, 2, 4):
        wl = inputs.decode_config(index, 1 / 32)
        used = [wl.page_table[b, : (int(wl.seq_lens[b]) + 15) // 16] for b in range(wl.batch)]
        pages = np.concatenate(used)
        assert len(set(pages.tolist())) == pages.size            # no page shared
        assert pages.min() >= 0 and pages.max() < wl.num_pages
    ragged = inputs.decode_config(4, 1 / 32)
    needed = sum((int(l) + 15) // 16 for l in ragged.seq_lens)
    assert ragged.num_pages >= 1.2 * needed                    # a fragmented pool with holes


def test_ragged_lengths_span_the_range():
    wl = inputs.decode_config(4)
    L = wl.seq_lens - 1                                        # the appended token
    assert L.min() >= 512 and L.max() <= 32768 and wl.batch == 256
    assert np.median(L) < 0.5 * (512 + 32768)                  # log-uniform: most sequences are short


def test_extend_chunk_rows_follow_their_prefix():
    ew = inputs.extend_config(scale=1 / 64, num_layers=2)
    rows = ew.chunk_ws_rows().reshape(ew.batch, ew.chunk_len)
    for b in range(ew.batch):
        assert rows[b, 0] == ew.cu_prefix[b] + ew.prefix_len and (np.diff(rows[b]) == 1).all()
        assert rows[b, -1] < ew.cu_prefix[b + 1]
    assert not np.array_equal(ew.q(0), ew.q(1))                # every layer has its own queries


def test_fp8_field_draws_avoid_nan_codes():
    rng = np.random.default_rng(0)
    b = inputs.fp8_bytes_by_field(rng, (100000,), 0, 14)
    assert not ((b & 0x7F) == 0x7F).any()
    assert set(np.unique((b >> 3) & 0xF).tolist()) == set(range(15))


def test_rounding_bytes_are_uniform():
    r = inputs.rounding_bytes(1, 1 << 20)
    counts = np.bincount(r, minlength=256)
    expected = r.size / 256
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 350                                          # 255 degrees of freedom
