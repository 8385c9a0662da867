"""Seeded synthetic workloads for the NVFP4 paged KV cache.

This module only draws random numbers and builds page tables / slot mappings;
it contains none of the quantisation or attention arithmetic.  Both the CUDA
library's tests and the CPU oracle read the arrays it produces.

Workloads follow the shapes of the source pages: 80 layers x 8 KV heads x
head_dim 128 ("nvfp4-kv-cache-memory-wall", section 1 capacity script), 128K
contexts, and a KV value mix of many small values plus a few large outliers
(same page, section 2 demo: gauss(0, 0.02) with 6.0 outliers).

Every array is drawn from ``numpy.random.default_rng`` on a seed sequence
``[base_seed, stream, index]`` so that any sequence's data can be regenerated
independently (and in parallel) without drawing the others.  bf16 values are
produced by rounding fp32 draws to nearest-even (torch's conversion) and are
returned as ``uint16`` bit patterns.
"""
from __future__ import annotations

import math
import random
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 128
PAGE_SIZE = 16
BASE_SEED = 20261106

# stream ids of the seed sequence
_S_PROMPT_K, _S_PROMPT_V, _S_NEW_K, _S_NEW_V, _S_Q, _S_PAGES, _S_LENS, _S_CHAN = range(8)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even) and return the uint16 bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact: bf16 is the top half of fp32)."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def page_demo_values() -> list:
    """The data set of the two-level-scaling demo ("nvfp4-kv-cache-memory-wall",
    section 2): Python's ``random`` seeded with 20261106, 4096 draws of
    gauss(0, 0.02), then 8 positions drawn with randrange set to 6.0."""
    rnd = random.Random(20261106)
    vals = [rnd.gauss(0, 0.02) for _ in range(4096)]
    for _ in range(8):
        vals[rnd.randrange(len(vals))] = 6.0
    return vals


# --------------------------------------------------------------------------
# value distributions
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class KVDist:
    """How K/V values are drawn.

    kind: "normal" (N(0, sigma)), "student_t" (t(nu) * sigma) or "channel"
    (N(0, 1) times a per-(kv_head, d) multiplier log-uniform in [lo, hi]).
    Outliers: ``per_chunk`` values of ``outlier`` at distinct positions in
    every ``chunk``-value chunk of a flattened [token][head][d] tensor, or a
    fraction ``frac`` of all positions at +-``outlier`` with a random sign.
    """
    kind: str = "normal"
    sigma: float = 1.0
    nu: float = 4.0
    lo: float = 0.1
    hi: float = 10.0
    outlier: float = 0.0
    frac: float = 0.0
    per_chunk: int = 0
    chunk: int = 4096


def _draw(rng: np.random.Generator, n: int, dist: KVDist, channel_mult=None) -> np.ndarray:
    if dist.kind == "normal":
        x = rng.standard_normal(n, dtype=np.float32)
        x *= np.float32(dist.sigma)
    elif dist.kind == "student_t":
        x = (rng.standard_t(dist.nu, n) * dist.sigma).astype(np.float32)
    elif dist.kind == "channel":
        x = rng.standard_normal(n, dtype=np.float32)
        m = channel_mult.reshape(-1)
        x = (x.reshape(-1, m.size) * m).reshape(-1)
    else:
        raise ValueError(dist.kind)
    if dist.per_chunk:
        full = n // dist.chunk
        for c in range(full + 1):
            lo = c * dist.chunk
            size = min(dist.chunk, n - lo)
            if size <= 0:
                break
            k = dist.per_chunk if size == dist.chunk else int(round(dist.per_chunk * size / dist.chunk))
            if k:
                pos = rng.choice(size, size=k, replace=False)
                x[lo + pos] = np.float32(dist.outlier)
    elif dist.frac:
        k = int(round(dist.frac * n))
        if k:
            pos = rng.choice(n, size=k, replace=False)
            sign = np.where(rng.random(k) < 0.5, -1.0, 1.0).astype(np.float32)
            x[pos] = sign * np.float32(dist.outlier)
    return x


# --------------------------------------------------------------------------
# decode workloads (one append + one decode step over a paged cache)
# --------------------------------------------------------------------------

@dataclass
class DecodeWorkload:
    name: str
    seed: int
    prompt_lens: np.ndarray          # int64 [B]: tokens cached before the step
    append: bool                     # the step appends one token per sequence first
    num_q_heads: int
    num_kv_heads: int
    dist: KVDist
    q_sigma: float = 1.0
    calibrated: bool = False         # per-tensor calibrated global scales, else 1.0
    pool_factor: float = 1.0         # physical pages / pages needed (>1 leaves holes)
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    _cache: dict = field(default_factory=dict, repr=False)

    # ---- shapes -----------------------------------------------------------
    @property
    def batch(self) -> int:
        return int(self.prompt_lens.shape[0])

    @property
    def seq_lens(self) -> np.ndarray:
        return (self.prompt_lens + (1 if self.append else 0)).astype(np.int32)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def pages_per_seq(self) -> np.ndarray:
        return (self.seq_lens.astype(np.int64) + self.page_size - 1) // self.page_size

    @property
    def max_pages(self) -> int:
        return int(self.pages_per_seq.max()) if self.batch else 1

    @property
    def num_pages(self) -> int:
        need = int(self.pages_per_seq.sum())
        return max(1, int(math.ceil(need * self.pool_factor)))

    def _rng(self, stream: int, index: int = 0) -> np.random.Generator:
        return np.random.default_rng([self.seed, stream, index])

    # ---- paging -------------------------------------------------------------
    @property
    def page_table(self) -> np.ndarray:
        """int32 [B, max_pages]: a random permutation of the pool (pages past a
        sequence's end are -1); with pool_factor > 1 the unused pages are holes
        scattered through the pool."""
        if "page_table" not in self._cache:
            rng = self._rng(_S_PAGES)
            perm = rng.permutation(self.num_pages).astype(np.int32)
            pt = np.full((self.batch, self.max_pages), -1, np.int32)
            pos = 0
            for b, n in enumerate(self.pages_per_seq):
                pt[b, :n] = perm[pos:pos + n]
                pos += int(n)
            self._cache["page_table"] = pt
        return self._cache["page_table"]

    def slots(self, b: int, start: int, count: int) -> np.ndarray:
        """int64 slot ids of tokens [start, start+count) of sequence b."""
        t = np.arange(start, start + count, dtype=np.int64)
        pages = self.page_table[b, t // self.page_size].astype(np.int64)
        return pages * self.page_size + t % self.page_size

    def append_slots(self) -> np.ndarray:
        return np.array([self.slots(b, int(self.prompt_lens[b]), 1)[0] for b in range(self.batch)],
                        np.int64)

    # ---- values -------------------------------------------------------------
    def _channel_mult(self, which: int) -> np.ndarray | None:
        if self.dist.kind != "channel":
            return None
        key = ("chan", which)
        if key not in self._cache:
            rng = self._rng(_S_CHAN, which)
            u = rng.random((self.num_kv_heads, self.head_dim))
            m = np.exp(np.log(self.dist.lo) + u * (np.log(self.dist.hi) - np.log(self.dist.lo)))
            self._cache[key] = m.astype(np.float32)
        return self._cache[key]

    def prompt_kv(self, b: int):
        """bf16 bits (K, V), each [prompt_len_b, Hkv, d], of sequence b's cached prompt."""
        n = int(self.prompt_lens[b]) * self.num_kv_heads * self.head_dim
        shape = (int(self.prompt_lens[b]), self.num_kv_heads, self.head_dim)
        k = _draw(self._rng(_S_PROMPT_K, b), n, self.dist, self._channel_mult(0))
        v = _draw(self._rng(_S_PROMPT_V, b), n, self.dist, self._channel_mult(1))
        return bf16_bits(k).reshape(shape), bf16_bits(v).reshape(shape)

    def new_kv(self):
        """bf16 bits (K, V), each [B, Hkv, d], of the token appended by the step."""
        shape = (self.batch, self.num_kv_heads, self.head_dim)
        ks, vs = [], []
        for b in range(self.batch):
            n = self.num_kv_heads * self.head_dim
            ks.append(_draw(self._rng(_S_NEW_K, b), n, self.dist, self._channel_mult(0)))
            vs.append(_draw(self._rng(_S_NEW_V, b), n, self.dist, self._channel_mult(1)))
        k = np.concatenate(ks) if ks else np.zeros(0, np.float32)
        v = np.concatenate(vs) if vs else np.zeros(0, np.float32)
        return bf16_bits(k).reshape(shape), bf16_bits(v).reshape(shape)

    def q(self) -> np.ndarray:
        """bf16 bits [B, Hq, d] of the decode queries, N(0, q_sigma)."""
        rng = self._rng(_S_Q)
        x = rng.standard_normal(self.batch * self.num_q_heads * self.head_dim, dtype=np.float32)
        x *= np.float32(self.q_sigma)
        return bf16_bits(x).reshape(self.batch, self.num_q_heads, self.head_dim)

    def all_prompt_kv(self, threads: int = 8):
        """Every sequence's prompt K/V (list of pairs), drawn in parallel threads."""
        with ThreadPoolExecutor(max_workers=threads) as ex:
            return list(ex.map(self.prompt_kv, range(self.batch)))

    def calibration_tensors(self, prompt=None, new=None):
        """The (K, V) bf16 pairs a calibrated global scale is taken over: every
        sequence's prompt and, when the step appends, the new tokens.  Empty
        when the workload keeps the uncalibrated scale 1."""
        if not self.calibrated:
            return []
        pairs = list(prompt if prompt is not None else self.all_prompt_kv())
        if self.append:
            pairs.append(new if new is not None else self.new_kv())
        return pairs

    def kv_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    def algorithmic_bytes(self) -> int:
        """Decode bytes: 144 B per token per KV head (K and V: 64 B data + 8 B
        scales each) + q (bf16) + out (fp32)."""
        kv = self.kv_tokens() * self.num_kv_heads * 2 * (self.head_dim // 2 + self.head_dim // 16)
        qb = self.batch * self.num_q_heads * self.head_dim * 2
        ob = self.batch * self.num_q_heads * self.head_dim * 4
        return kv + qb + ob


def _loguniform_ints(rng, n, lo, hi) -> np.ndarray:
    u = rng.random(n)
    return np.floor(np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))).astype(np.int64).clip(lo, hi)


def decode_config(index: int, scale: float = 1.0) -> DecodeWorkload:
    """Decode workloads 1-4 (index), optionally with every length scaled down.

    1 tiny correctness: B=2, prompts {100, 257}, 8 q / 2 KV heads, N(0,1) with
      0.1% of entries at +-20, global scale 1, shuffled page table.
    2 decode at the pages' shape: B=32, ctx 8192 (+1 appended), 64 q / 8 KV
      heads, N(0,0.02) with 8 of every 4096 values = 6.0, q ~ N(0,1).
    3 long context: B=4, ctx 131072 (no append), 64 / 8 heads, N(0,1) times a
      per-channel multiplier log-uniform in [0.1, 10], calibrated global scale.
    4 ragged batch: 256 sequences, lengths log-uniform in [512, 32768] (+1
      appended), 32 / 8 heads, Student-t(4) * 0.05, fragmented page pool.
    """
    seed = BASE_SEED + index
    s = lambda n: max(1, int(round(n * scale)))
    if index == 1:
        return DecodeWorkload("tiny_b2_gqa4", seed, np.array([s(100), s(257)], np.int64), True, 8, 2,
                              KVDist("normal", 1.0, outlier=20.0, frac=0.001))
    if index == 2:
        return DecodeWorkload("decode_b32_ctx8k_h64kv8", seed, np.full(32, s(8192), np.int64), True,
                              64, 8, KVDist("normal", 0.02, outlier=6.0, per_chunk=8, chunk=4096))
    if index == 3:
        return DecodeWorkload("decode_b4_ctx128k_h64kv8", seed, np.full(4, s(131072), np.int64),
                              False, 64, 8, KVDist("channel", lo=0.1, hi=10.0), calibrated=True)
    if index == 4:
        rng = np.random.default_rng([seed, _S_LENS])
        lens = _loguniform_ints(rng, 256, 512, 32768)
        lens = np.maximum(1, np.round(lens * scale)).astype(np.int64)
        return DecodeWorkload("ragged_b256_ctx512to32k_h32kv8", seed, lens, True, 32, 8,
                              KVDist("student_t", 0.05, nu=4.0), pool_factor=1.25)
    raise ValueError(index)


# --------------------------------------------------------------------------
# extend workload: NVFP4 prefix -> FP8 workspace, plus a quantize-write chunk
# --------------------------------------------------------------------------

@dataclass
class ExtendWorkload:
    name: str
    seed: int
    num_layers: int
    batch: int
    prefix_len: int
    chunk_len: int
    num_kv_heads: int
    dist: KVDist
    num_q_heads: int = 64
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    _cache: dict = field(default_factory=dict, repr=False)

    @property
    def prefix_lens(self) -> np.ndarray:
        return np.full(self.batch, self.prefix_len, np.int32)

    @property
    def cu_q(self) -> np.ndarray:
        """Query offsets of the chunk tokens: sequence b owns [cu_q[b], cu_q[b+1])."""
        return np.arange(self.batch + 1, dtype=np.int64) * self.chunk_len

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def chunk_ws_rows(self) -> np.ndarray:
        """Workspace row of every chunk token: right after its sequence's prefix."""
        t = np.arange(self.chunk_len, dtype=np.int64)
        return np.concatenate([self.cu_prefix[b] + self.prefix_len + t for b in range(self.batch)])

    def q(self, layer: int) -> np.ndarray:
        """bf16 bits [batch * chunk_len, Hq, d] of the chunk's queries, N(0, 1)."""
        rng = np.random.default_rng([self.seed, _S_Q, layer])
        n = self.batch * self.chunk_len * self.num_q_heads * self.head_dim
        return bf16_bits(rng.standard_normal(n, dtype=np.float32)).reshape(
            self.batch * self.chunk_len, self.num_q_heads, self.head_dim)

    def attention_flops_per_layer(self) -> int:
        """2 d flops for q.k and 2 d for p.v per (query token, query head, visible
        key); chunk token t of a sequence sees prefix_len + t + 1 keys."""
        C, P = self.chunk_len, self.prefix_len
        keys = C * P + C * (C + 1) // 2
        return 4 * self.head_dim * self.num_q_heads * self.batch * keys

    @property
    def cu_prefix(self) -> np.ndarray:
        """Workspace row offsets: each sequence's prefix rows are followed by
        room for its new chunk (rows the dequant leaves untouched)."""
        per = self.prefix_len + self.chunk_len
        return (np.arange(self.batch + 1, dtype=np.int64) * per)

    @property
    def total_rows(self) -> int:
        return int(self.cu_prefix[-1])

    @property
    def pages_per_seq(self) -> int:
        return (self.prefix_len + self.chunk_len + self.page_size - 1) // self.page_size

    @property
    def num_pages(self) -> int:
        return self.batch * self.pages_per_seq

    @property
    def page_table(self) -> np.ndarray:
        if "page_table" not in self._cache:
            rng = np.random.default_rng([self.seed, _S_PAGES])
            perm = rng.permutation(self.num_pages).astype(np.int32)
            self._cache["page_table"] = perm.reshape(self.batch, self.pages_per_seq)
        return self._cache["page_table"]

    def slots(self, b: int, start: int, count: int) -> np.ndarray:
        t = np.arange(start, start + count, dtype=np.int64)
        return self.page_table[b, t // self.page_size].astype(np.int64) * self.page_size + t % self.page_size

    def prefix_slots(self) -> np.ndarray:
        return np.concatenate([self.slots(b, 0, self.prefix_len) for b in range(self.batch)])

    def chunk_slots(self) -> np.ndarray:
        return np.concatenate([self.slots(b, self.prefix_len, self.chunk_len) for b in range(self.batch)])

    def _kv(self, layer: int, stream: int, tokens: int, b: int):
        n = tokens * self.num_kv_heads * self.head_dim
        shape = (tokens, self.num_kv_heads, self.head_dim)
        rng = np.random.default_rng([self.seed, stream, layer * 100003 + b])
        return bf16_bits(_draw(rng, n, self.dist)).reshape(shape)

    def prefix_kv(self, layer: int, b: int):
        return (self._kv(layer, _S_PROMPT_K, self.prefix_len, b),
                self._kv(layer, _S_PROMPT_V, self.prefix_len, b))

    def chunk_kv(self, layer: int, b: int):
        return (self._kv(layer, _S_NEW_K, self.chunk_len, b),
                self._kv(layer, _S_NEW_V, self.chunk_len, b))

    def dequant_bytes_per_layer(self) -> int:
        """9/16 B read + 1 B written per value of every prefix token, K and V."""
        vals = self.batch * self.prefix_len * self.num_kv_heads * self.head_dim * 2
        return vals * 9 // 16 + vals

    def quantize_bytes_per_layer(self) -> int:
        """2 B read + 9/16 B written per value of every new token, K and V, plus
        8 B of slot mapping per token."""
        toks = self.batch * self.chunk_len
        vals = toks * self.num_kv_heads * self.head_dim * 2
        return vals * 2 + vals * 9 // 16 + toks * 8


def extend_config(scale: float = 1.0, num_layers: int = 80) -> ExtendWorkload:
    """Workload 5: 80 layers x 8 KV heads, 16 sequences each with a 16384-token
    NVFP4 prefix and a 2048-token new chunk; N(0, 0.02) with 0.2% outliers at
    +-6; global scale 1 and workspace scale 1."""
    s = lambda n: max(1, int(round(n * scale)))
    return ExtendWorkload("extend_b16_prefix16k_chunk2k_kv8", BASE_SEED + 5, num_layers, 16,
                          s(16384), s(2048), 8, KVDist("normal", 0.02, outlier=6.0, frac=0.002))


# --------------------------------------------------------------------------
# random bytes drawn by the stochastic-rounding variant (an input of the method)
# --------------------------------------------------------------------------

_S_ROUND = 9


def rounding_bytes(index: int, n: int) -> np.ndarray:
    """n uniform random bytes for stochastic rounding, one per value."""
    rng = np.random.default_rng([BASE_SEED, _S_ROUND, index])
    return rng.integers(0, 256, n, dtype=np.uint8)


# --------------------------------------------------------------------------
# extend attention over a given FP8 workspace (ragged cases for the tests)
# --------------------------------------------------------------------------

def fp8_bytes_by_field(rng: np.random.Generator, shape, exp_lo: int, exp_hi: int) -> np.ndarray:
    """Random E4M3 bytes drawn field by field: a uniform sign bit, a uniform
    4-bit exponent field in [exp_lo, exp_hi] and a uniform 3-bit mantissa
    (exp_hi <= 14 keeps clear of the NaN codes 0x7F / 0xFF)."""
    sign = rng.integers(0, 2, shape, dtype=np.uint8) << 7
    exp = rng.integers(exp_lo, exp_hi + 1, shape, dtype=np.uint8) << 3
    man = rng.integers(0, 8, shape, dtype=np.uint8)
    return (sign | exp | man).astype(np.uint8)


@dataclass
class ExtendAttnCase:
    """A ragged extend-attention problem over an FP8 workspace: sequence b has
    prefix_lens[b] cached rows and chunk_lens[b] new tokens, its rows starting
    at cu_prefix[b] with `gap` unused rows before the next sequence."""
    name: str
    seed: int
    prefix_lens: np.ndarray
    chunk_lens: np.ndarray
    num_q_heads: int
    num_kv_heads: int
    gap: int = 3
    k_exp: tuple = (3, 8)     # E4M3 exponent-field range of K bytes (magnitudes 2^-4 .. 3.75)
    v_exp: tuple = (1, 9)
    head_dim: int = HEAD_DIM

    @property
    def batch(self) -> int:
        return int(self.prefix_lens.shape[0])

    @property
    def cu_prefix(self) -> np.ndarray:
        per = self.prefix_lens.astype(np.int64) + self.chunk_lens.astype(np.int64) + self.gap
        return np.concatenate([[0], np.cumsum(per)]).astype(np.int64)

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.chunk_lens.astype(np.int64))]).astype(np.int64)

    @property
    def total_rows(self) -> int:
        return int(self.cu_prefix[-1])

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def workspace(self):
        """(ws_k, ws_v): uint8 E4M3 [total_rows, Hkv, d], every row drawn (gap rows too)."""
        rng = np.random.default_rng([self.seed, _S_PROMPT_K])
        shape = (self.total_rows, self.num_kv_heads, self.head_dim)
        return fp8_bytes_by_field(rng, shape, *self.k_exp), fp8_bytes_by_field(rng, shape, *self.v_exp)

    def q(self) -> np.ndarray:
        rng = np.random.default_rng([self.seed, _S_Q])
        n = self.total_q * self.num_q_heads * self.head_dim
        return bf16_bits(rng.standard_normal(n, dtype=np.float32)).reshape(
            self.total_q, self.num_q_heads, self.head_dim)

    def flops(self) -> int:
        C = self.chunk_lens.astype(np.int64)
        keys = int((C * self.prefix_lens.astype(np.int64) + C * (C + 1) // 2).sum())
        return 4 * self.head_dim * self.num_q_heads * keys


def extend_attn_case(index: int) -> ExtendAttnCase:
    """Ragged extend-attention cases for the parity tests.

    1 three sequences, GQA 4 (8 / 2 heads): prefixes {0, 37, 300}, chunks {19, 1, 130}
    2 GQA 8 (16 / 2 heads), chunks that are not multiples of 16 tokens: prefixes
      {129, 1000}, chunks {33, 260}
    3 one sequence, G = 1 (2 / 2 heads), prefix 256, chunk 64
    4 G = 16 (32 / 2 heads): prefixes {5, 700}, chunks {17, 40}
    """
    seed = BASE_SEED + 100 + index
    a = lambda *v: np.array(v, np.int32)
    if index == 1:
        return ExtendAttnCase("extend_attn_gqa4", seed, a(0, 37, 300), a(19, 1, 130), 8, 2)
    if index == 2:
        return ExtendAttnCase("extend_attn_gqa8", seed, a(129, 1000), a(33, 260), 16, 2)
    if index == 3:
        return ExtendAttnCase("extend_attn_mha", seed, a(256), a(64), 2, 2)
    if index == 4:
        return ExtendAttnCase("extend_attn_gqa16", seed, a(5, 700), a(17, 40), 32, 2)
    raise ValueError(index)
