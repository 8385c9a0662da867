"""CPU oracle for the NVFP4 paged KV cache -- TEST INFRASTRUCTURE ONLY.

This package is the independent reference the CUDA library is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import it; the product path never does.  It shares no code
with the CUDA library: the arithmetic lives in ``nvfp4_oracle.c`` (plain C,
compiled by ``oracle/build.py``), and this module only marshals numpy arrays
into it through ctypes.

bf16 tensors travel as ``uint16`` bit patterns (numpy has no bf16 dtype).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

BLOCK = 16


class _CCache(ctypes.Structure):
    _fields_ = [
        ("k_data", ctypes.c_void_p),
        ("v_data", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("num_pages", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("k_global_scale", ctypes.c_float),
        ("v_global_scale", ctypes.c_float),
    ]


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u8, f32, f64, i64, i32, vp = (ctypes.c_uint8, ctypes.c_float, ctypes.c_double,
                                      ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p)
        L.nvfp4_oracle_e2m1_value.argtypes = [u8]
        L.nvfp4_oracle_e2m1_value.restype = f64
        L.nvfp4_oracle_e4m3_value.argtypes = [u8]
        L.nvfp4_oracle_e4m3_value.restype = f64
        L.nvfp4_oracle_e2m1_encode.argtypes = [f32]
        L.nvfp4_oracle_e2m1_encode.restype = u8
        L.nvfp4_oracle_e4m3_encode.argtypes = [f32]
        L.nvfp4_oracle_e4m3_encode.restype = u8
        L.nvfp4_oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.nvfp4_oracle_bf16_to_float.restype = f32
        L.nvfp4_oracle_quantize_block.argtypes = [vp, f32, vp, vp]
        L.nvfp4_oracle_quantize_block.restype = None
        L.nvfp4_oracle_dequant_value.argtypes = [u8, u8, f32]
        L.nvfp4_oracle_dequant_value.restype = f64
        L.nvfp4_oracle_demo_fake_quant.argtypes = [vp, i64, i64, vp]
        L.nvfp4_oracle_demo_fake_quant.restype = None
        L.nvfp4_oracle_row_bytes.argtypes = [ctypes.c_int]
        L.nvfp4_oracle_row_bytes.restype = i64
        L.nvfp4_oracle_row_scale_bytes.argtypes = [ctypes.c_int]
        L.nvfp4_oracle_row_scale_bytes.restype = i64
        L.nvfp4_oracle_quantize_append.argtypes = [ctypes.POINTER(_CCache), vp, vp, vp, i64]
        L.nvfp4_oracle_quantize_append.restype = ctypes.c_int
        L.nvfp4_oracle_decode_attention.argtypes = [ctypes.POINTER(_CCache), vp, vp, i32, vp,
                                                    i32, i32, f64, vp]
        L.nvfp4_oracle_decode_attention.restype = ctypes.c_int
        L.nvfp4_oracle_decode_attention_heads.argtypes = [ctypes.POINTER(_CCache), vp, vp, i32, vp,
                                                          i32, i32, f64, i32, i32, vp]
        L.nvfp4_oracle_decode_attention_heads.restype = ctypes.c_int
        L.nvfp4_oracle_dequant_to_fp8_workspace.argtypes = [ctypes.POINTER(_CCache), vp, i32, vp,
                                                            vp, i32, f32, f32, vp, vp]
        L.nvfp4_oracle_dequant_to_fp8_workspace.restype = ctypes.c_int
        L.nvfp4_oracle_tensor_amax.argtypes = [vp, i64]
        L.nvfp4_oracle_tensor_amax.restype = f32
        L.nvfp4_oracle_calibrated_global_scale.argtypes = [f32]
        L.nvfp4_oracle_calibrated_global_scale.restype = f32
        L.nvfp4_oracle_e8m0_value.argtypes = [u8]
        L.nvfp4_oracle_e8m0_value.restype = f64
        L.nvfp4_oracle_mxfp4_quantize_block.argtypes = [vp, vp, vp]
        L.nvfp4_oracle_mxfp4_quantize_block.restype = None
        L.nvfp4_oracle_mxfp4_dequant_value.argtypes = [u8, u8]
        L.nvfp4_oracle_mxfp4_dequant_value.restype = f64
        L.nvfp4_oracle_e2m1_encode_sr.argtypes = [f32, u8]
        L.nvfp4_oracle_e2m1_encode_sr.restype = u8
        L.nvfp4_oracle_quantize_block_sr.argtypes = [vp, f32, vp, vp, vp]
        L.nvfp4_oracle_quantize_block_sr.restype = None
        L.nvfp4_oracle_hadamard.argtypes = [vp, ctypes.c_int, vp]
        L.nvfp4_oracle_hadamard.restype = ctypes.c_int
        L.nvfp4_oracle_decode_attention_format.argtypes = [ctypes.POINTER(_CCache), ctypes.c_int, vp, vp, i32, vp,
                                                           i32, i32, f64, vp]
        L.nvfp4_oracle_decode_attention_format.restype = ctypes.c_int
        L.nvfp4_oracle_bf16_to_fp8_workspace.argtypes = [vp, vp, vp, i64, i32, i32, i64, f32, f32, vp, vp]
        L.nvfp4_oracle_bf16_to_fp8_workspace.restype = ctypes.c_int
        L.nvfp4_oracle_extend_attention_rows.argtypes = [vp, vp, i64, i32, i32, f32, f32, vp, i32, vp, vp, vp,
                                                         i32, f64, vp, i64, vp]
        L.nvfp4_oracle_extend_attention_rows.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


# --------------------------------------------------------------------------
# formats
# --------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().nvfp4_oracle_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return lib().nvfp4_oracle_e4m3_value(code)


def e2m1_encode(y) -> int:
    return lib().nvfp4_oracle_e2m1_encode(float(np.float32(y)))


def e4m3_encode(z) -> int:
    return lib().nvfp4_oracle_e4m3_encode(float(np.float32(z)))


def quantize_block(x, g):
    """One 16-value block -> (8 packed bytes, E4M3 scale byte)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (BLOCK,)
    packed = np.zeros(BLOCK // 2, np.uint8)
    scale = np.zeros(1, np.uint8)
    lib().nvfp4_oracle_quantize_block(_ptr(x), float(np.float32(g)), _ptr(packed), _ptr(scale))
    return packed, int(scale[0])


def dequant_value(code: int, scale: int, g) -> float:
    return lib().nvfp4_oracle_dequant_value(code, scale, float(np.float32(g)))


def demo_fake_quant(x, block: int) -> np.ndarray:
    """The page demo's binary64 fake-quantisation (unrounded block scale)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().nvfp4_oracle_demo_fake_quant(_ptr(x), x.size, block, _ptr(out))
    return out


def row_bytes(head_dim: int) -> int:
    return lib().nvfp4_oracle_row_bytes(head_dim)


def row_scale_bytes(head_dim: int) -> int:
    return lib().nvfp4_oracle_row_scale_bytes(head_dim)


# --------------------------------------------------------------------------
# paged cache
# --------------------------------------------------------------------------

class Cache:
    """Host-side NVFP4 paged cache (numpy arrays in the oracle's layout)."""

    def __init__(self, num_pages, num_kv_heads, head_dim=128, page_size=16,
                 k_global_scale=1.0, v_global_scale=1.0, arrays=None):
        self.num_pages = int(num_pages)
        self.num_kv_heads = int(num_kv_heads)
        self.head_dim = int(head_dim)
        self.page_size = int(page_size)
        self.k_global_scale = float(np.float32(k_global_scale))
        self.v_global_scale = float(np.float32(v_global_scale))
        rows = self.num_pages * self.num_kv_heads * self.page_size
        if arrays is None:
            self.k_data = np.zeros((rows, row_bytes(head_dim)), np.uint8)
            self.v_data = np.zeros((rows, row_bytes(head_dim)), np.uint8)
            self.k_scale = np.zeros((rows, row_scale_bytes(head_dim)), np.uint8)
            self.v_scale = np.zeros((rows, row_scale_bytes(head_dim)), np.uint8)
        else:
            self.k_data, self.v_data, self.k_scale, self.v_scale = (
                np.ascontiguousarray(a, dtype=np.uint8).reshape(rows, -1) for a in arrays)

    def _c(self) -> _CCache:
        return _CCache(_ptr(self.k_data), _ptr(self.v_data), _ptr(self.k_scale),
                       _ptr(self.v_scale), self.num_pages, self.num_kv_heads, self.head_dim,
                       self.page_size, self.k_global_scale, self.v_global_scale)


def quantize_append(cache: Cache, k_bf16, v_bf16, slot_mapping) -> int:
    k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
    v = np.ascontiguousarray(v_bf16, dtype=np.uint16)
    s = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    n = s.shape[0]
    assert k.shape == v.shape == (n, cache.num_kv_heads, cache.head_dim)
    c = cache._c()
    return lib().nvfp4_oracle_quantize_append(ctypes.byref(c), _ptr(k), _ptr(v), _ptr(s), n)


def decode_attention(cache: Cache, q_bf16, page_table, seq_lens, softmax_scale, heads=None):
    """fp64 decode attention; returns (out[B, Hq, d] float64, status).

    heads=(begin, end) computes only those query heads (other rows stay 0)."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, d = q.shape
    assert d == cache.head_dim and pt.shape[0] == B and sl.shape == (B,)
    out = np.zeros((B, Hq, d), np.float64)
    c = cache._c()
    hb, he = (0, Hq) if heads is None else heads
    st = lib().nvfp4_oracle_decode_attention_heads(ctypes.byref(c), _ptr(q), _ptr(pt), pt.shape[1],
                                                   _ptr(sl), B, Hq, float(softmax_scale), hb, he,
                                                   _ptr(out))
    return out, st


def dequant_to_fp8_workspace(cache: Cache, page_table, prefix_lens, cu_prefix, total_rows,
                             k_ws_scale=1.0, v_ws_scale=1.0):
    """FP8 E4M3 workspace bytes; returns (ws_k, ws_v, status), [rows, Hkv, d] uint8."""
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    pl = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    cu = np.ascontiguousarray(cu_prefix, dtype=np.int64)
    B = pl.shape[0]
    ws_k = np.zeros((total_rows, cache.num_kv_heads, cache.head_dim), np.uint8)
    ws_v = np.zeros_like(ws_k)
    c = cache._c()
    st = lib().nvfp4_oracle_dequant_to_fp8_workspace(
        ctypes.byref(c), _ptr(pt), pt.shape[1], _ptr(pl), _ptr(cu), B,
        float(np.float32(k_ws_scale)), float(np.float32(v_ws_scale)), _ptr(ws_k), _ptr(ws_v))
    return ws_k, ws_v, st


def dequantize_rows(cache: Cache, which: str, rows) -> np.ndarray:
    """fp64 dequantised cache rows (for test cross-checks); rows index the flat row axis."""
    lb = lib()
    data = cache.k_data if which == "k" else cache.v_data
    scl = cache.k_scale if which == "k" else cache.v_scale
    g = cache.k_global_scale if which == "k" else cache.v_global_scale
    codes = np.arange(16, dtype=np.uint8)
    e2m1 = np.array([lb.nvfp4_oracle_e2m1_value(int(c)) for c in codes])
    e4m3 = np.array([lb.nvfp4_oracle_e4m3_value(int(c)) for c in range(256)])
    rows = np.asarray(rows)
    d = data[rows]
    lo, hi = d & 0xF, d >> 4
    code = np.stack([lo, hi], axis=-1).reshape(len(rows), -1)
    sc = np.repeat(e4m3[scl[rows]], BLOCK, axis=-1)
    return e2m1[code] * sc * np.float64(np.float32(g))




def tensor_amax(x_bf16) -> float:
    """Largest |x| of a bf16 tensor (uint16 bit patterns); 0 when empty."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1)
    return float(lib().nvfp4_oracle_tensor_amax(_ptr(x), x.size))


def calibrated_global_scale(amax: float) -> float:
    """g = amax / (6 * 448) in binary32 (1 when amax is 0)."""
    return float(lib().nvfp4_oracle_calibrated_global_scale(float(np.float32(amax))))


def bf16_to_fp8_workspace(k_bf16, v_bf16, ws_rows, ws_k, ws_v, k_ws_scale=1.0, v_ws_scale=1.0) -> int:
    """The chunk's K/V (bf16 bits [n, Hkv, d]) into workspace rows ws_rows[t]
    (in place in ws_k, ws_v: uint8 [rows, Hkv, d]); returns the status."""
    k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
    v = np.ascontiguousarray(v_bf16, dtype=np.uint16)
    r = np.ascontiguousarray(ws_rows, dtype=np.int64)
    assert ws_k.flags["C_CONTIGUOUS"] and ws_v.flags["C_CONTIGUOUS"]
    n, H, d = k.shape
    return lib().nvfp4_oracle_bf16_to_fp8_workspace(_ptr(k), _ptr(v), _ptr(r), n, H, d, ws_k.shape[0],
                                                    float(np.float32(k_ws_scale)), float(np.float32(v_ws_scale)),
                                                    _ptr(ws_k), _ptr(ws_v))


def extend_attention_rows(ws_k, ws_v, q_bf16, cu_q, cu_prefix, prefix_lens, softmax_scale, pairs,
                          k_ws_scale=1.0, v_ws_scale=1.0):
    """fp64 extend-attention output rows for (global query token, query head)
    pairs; q_bf16 [total_q, Hq, d].  Returns (out [len(pairs), d], status)."""
    wk = np.ascontiguousarray(ws_k, dtype=np.uint8)
    wv = np.ascontiguousarray(ws_v, dtype=np.uint8)
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    cq = np.ascontiguousarray(cu_q, dtype=np.int64)
    cp = np.ascontiguousarray(cu_prefix, dtype=np.int64)
    pl = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    out = np.zeros((pr.shape[0], wk.shape[2]), np.float64)
    st = lib().nvfp4_oracle_extend_attention_rows(_ptr(wk), _ptr(wv), wk.shape[0], wk.shape[1], wk.shape[2],
                                                  float(np.float32(k_ws_scale)), float(np.float32(v_ws_scale)),
                                                  _ptr(q), q.shape[1], _ptr(cq), _ptr(cp), _ptr(pl), pl.shape[0],
                                                  float(softmax_scale), _ptr(pr), pr.shape[0], _ptr(out))
    return out, st


def extend_attention(ws_k, ws_v, q_bf16, cu_q, cu_prefix, prefix_lens, softmax_scale, k_ws_scale=1.0,
                     v_ws_scale=1.0):
    """Every output row: fp64 [total_q, Hq, d] and the status."""
    total_q, Hq = q_bf16.shape[0], q_bf16.shape[1]
    pairs = np.stack(np.meshgrid(np.arange(total_q), np.arange(Hq), indexing="ij"), -1).reshape(-1, 2)
    out, st = extend_attention_rows(ws_k, ws_v, q_bf16, cu_q, cu_prefix, prefix_lens, softmax_scale, pairs,
                                    k_ws_scale, v_ws_scale)
    return out.reshape(total_q, Hq, -1), st



# --------------------------------------------------------------------------
# format variants (MXFP4, stochastic rounding, Hadamard rotation)
# --------------------------------------------------------------------------

MX_BLOCK = 32


def e8m0_value(code: int) -> float:
    return lib().nvfp4_oracle_e8m0_value(code)


def mxfp4_quantize_block(x):
    """One 32-value block -> (16 packed bytes, E8M0 scale byte)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (MX_BLOCK,)
    packed = np.zeros(MX_BLOCK // 2, np.uint8)
    scale = np.zeros(1, np.uint8)
    lib().nvfp4_oracle_mxfp4_quantize_block(_ptr(x), _ptr(packed), _ptr(scale))
    return packed, int(scale[0])


def mxfp4_dequant_value(code: int, scale: int) -> float:
    return lib().nvfp4_oracle_mxfp4_dequant_value(code, scale)


def e2m1_encode_sr(y, r: int) -> int:
    return lib().nvfp4_oracle_e2m1_encode_sr(float(np.float32(y)), int(r))


def quantize_block_sr(x, g, r):
    """One 16-value block with stochastic element rounding (r: 16 random bytes)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rr = np.ascontiguousarray(r, dtype=np.uint8)
    assert x.shape == (BLOCK,) and rr.shape == (BLOCK,)
    packed = np.zeros(BLOCK // 2, np.uint8)
    scale = np.zeros(1, np.uint8)
    lib().nvfp4_oracle_quantize_block_sr(_ptr(x), float(np.float32(g)), _ptr(rr), _ptr(packed), _ptr(scale))
    return packed, int(scale[0])


def hadamard(x) -> np.ndarray:
    """Orthonormal Walsh-Hadamard transform (Sylvester order, binary32 butterflies) of a vector."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.zeros_like(x)
    assert lib().nvfp4_oracle_hadamard(_ptr(x), x.shape[0], _ptr(y)) == 0
    return y


def _unpack(packed) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    return np.stack([p & 0xF, p >> 4], axis=-1).reshape(-1)


def fake_quant(x, variant: str, g: float = 1.0, rand=None) -> np.ndarray:
    """Quantise then dequantise (fp64) a 1-D array whose length is a multiple of 128,
    in one of the variants: "nvfp4" (blocks of 16, E4M3 scale, nearest even),
    "nvfp4_sr" (elements rounded stochastically with rand, one byte per value),
    "nvfp4_hadamard" (each 128-value vector rotated first and rotated back after),
    "mxfp4" (blocks of 32, E8M0 scale)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.zeros(x.shape[0], np.float64)
    e2m1 = np.array([e2m1_value(c) for c in range(16)])
    if variant == "mxfp4":
        for i in range(0, x.shape[0], MX_BLOCK):
            packed, sc = mxfp4_quantize_block(x[i:i + MX_BLOCK])
            out[i:i + MX_BLOCK] = e2m1[_unpack(packed)] * e8m0_value(sc)
        return out
    gg = float(np.float32(g))
    vecs = x.reshape(-1, 128)
    if variant == "nvfp4_hadamard":
        vecs = np.stack([hadamard(v) for v in vecs])
    flat = vecs.reshape(-1)
    for i in range(0, flat.shape[0], BLOCK):
        blk = flat[i:i + BLOCK]
        if variant == "nvfp4_sr":
            packed, sc = quantize_block_sr(blk, gg, rand[i:i + BLOCK])
        else:
            packed, sc = quantize_block(blk, gg)
        out[i:i + BLOCK] = e2m1[_unpack(packed)] * e4m3_value(sc) * gg
    if variant == "nvfp4_hadamard":
        # the rotation is orthonormal: its transpose (itself) undoes it, here in fp64
        n = 128
        h = np.array([[1.0]])
        while h.shape[0] < n:
            h = np.block([[h, h], [h, -h]])
        out = (out.reshape(-1, n) @ (h / np.sqrt(n))).reshape(-1)
    return out



FORMAT_NVFP4, FORMAT_NVFP4_HADAMARD, FORMAT_MXFP4 = 0, 1, 2


def decode_attention_format(cache: Cache, fmt: int, q_bf16, page_table, seq_lens, softmax_scale):
    """fp64 decode attention over a variant's cache (FORMAT_*); for MXFP4 the
    cache's scale arrays hold head_dim / 32 E8M0 bytes per row."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, d = q.shape
    out = np.zeros((B, Hq, d), np.float64)
    c = cache._c()
    st = lib().nvfp4_oracle_decode_attention_format(ctypes.byref(c), int(fmt), _ptr(q), _ptr(pt), pt.shape[1],
                                                    _ptr(sl), B, Hq, float(softmax_scale), _ptr(out))
    return out, st


__all__ = [name for name in dir() if not name.startswith("_")]
