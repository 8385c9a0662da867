"""nvfp4kv: an NVFP4 paged KV cache for one GB300 (sm_103a).

All compute lives in the CUDA library ``libnvfp4kv.so`` whose C ABI is
declared in ``include/nvfp4kv.h``.  This module is a thin ctypes binding with
the same function names: it only turns torch tensors into pointers and sizes
and raises on a non-zero status.  PyTorch provides device memory and streams.
There is no CPU fallback: if the library cannot be loaded, every call raises.

The seeded workload generators live in ``nvfp4_quantized_paged_quantize_gb300.inputs``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "_build", "libnvfp4kv.so")

NVFP4KV_OK = 0
NVFP4KV_ERR_INVALID_ARGUMENT = -1
NVFP4KV_ERR_UNSUPPORTED = -2
NVFP4KV_ERR_CUDA = -3
NVFP4KV_ERR_WORKSPACE = -4

NVFP4KV_DEVERR_SLOT = 1
NVFP4KV_DEVERR_PAGE = 2
NVFP4KV_DEVERR_LENGTH = 4
NVFP4KV_DEVERR_TIMEOUT = 8
NVFP4KV_DEVERR_ROW = 16
NVFP4KV_PROBE_DECODE_PATTERN = 0
NVFP4KV_PROBE_WHOLE_PAGES = 1
NVFP4KV_VARIANT_SR = 1
NVFP4KV_VARIANT_HADAMARD = 2
NVFP4KV_VARIANT_MXFP4 = 3

HEAD_DIM = 128
PAGE_SIZE = 16
# bytes of one page-head (16 tokens of one KV head): K data, K scales, V data, V scales
NVFP4KV_PAGE_HEAD_BYTES = 2304
NVFP4KV_MXFP4_PAGE_HEAD_BYTES = 2176

_lib = None


class Nvfp4kvError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        msg = nvfp4kv_status_string(status) if _lib is not None else str(status)
        if _lib is not None and status == NVFP4KV_ERR_CUDA:
            msg += ": " + _lib.nvfp4kv_last_cuda_error().decode()
        super().__init__(f"{func} failed: {msg} ({status})")


class _CCache(ctypes.Structure):
    _fields_ = [
        ("pages", ctypes.c_void_p),
        ("num_pages", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("k_global_scale", ctypes.c_float),
        ("v_global_scale", ctypes.c_float),
    ]


def load(path: str | None = None, build_if_missing: bool = True):
    """Load libnvfp4kv.so (building it in-tree first if it is missing or stale).

    Raises if the library cannot be built or loaded: there is no fallback path.
    """
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = LIB_PATH
        if build_if_missing:
            from . import build as _build

            path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libnvfp4kv.so not found at {path}; run build() first")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    pc = ctypes.POINTER(_CCache)
    L.nvfp4kv_cache_bytes.argtypes = [i64, i32, i32, i32, ctypes.POINTER(sz)]
    L.nvfp4kv_quantize_append.argtypes = [pc, vp, vp, vp, i64, vp, vp]
    L.nvfp4kv_decode_workspace_size.argtypes = [pc, i32, i32, ctypes.POINTER(sz)]
    L.nvfp4kv_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.nvfp4kv_decode_workspace_bytes.restype = sz
    L.nvfp4kv_decode_attention.argtypes = [pc, vp, vp, vp, i32, vp, i32, i32, f32, vp, sz, vp, vp]
    L.nvfp4kv_dequant_to_fp8_workspace.argtypes = [pc, vp, i32, vp, vp, i32, i64, f32, f32, vp, vp, vp, vp]
    L.nvfp4kv_decode_attention_static.argtypes = [pc, vp, vp, vp, i32, vp, i32, i32, f32, vp, vp]
    L.nvfp4kv_append_decode_attention.argtypes = [pc, vp, vp, vp, i64, vp, vp, vp, i32, vp, i32, i32, f32, vp, sz,
                                                  vp, vp]
    L.nvfp4kv_tensor_amax.argtypes = [vp, i64, vp, ctypes.c_int, vp]
    L.nvfp4kv_quantize_append_variant.argtypes = [ctypes.c_int, pc, vp, vp, vp, i64, vp, vp, vp, vp]
    L.nvfp4kv_quantize_append_fp8.argtypes = [pc, vp, vp, vp, i64, vp, i64, f32, f32, vp, vp, vp, vp]
    L.nvfp4kv_bf16_to_fp8_workspace.argtypes = [vp, vp, vp, i64, i32, i32, i64, f32, f32, vp, vp, vp, vp]
    L.nvfp4kv_extend_attention.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, i64, i32, i32, i32, f32, f32, f32, vp,
                                           vp, vp]
    L.nvfp4kv_calibrated_global_scale.argtypes = [f32, ctypes.POINTER(f32)]
    L.nvfp4kv_stream_probe.argtypes = [pc, vp, i32, vp, i32, ctypes.c_int, vp, vp, vp]
    L.nvfp4kv_decode_attention_variant.argtypes = [ctypes.c_int, pc, vp, vp, vp, i32, vp, i32, i32, f32, vp, sz, vp,
                                                   vp]
    L.nvfp4kv_last_cuda_error.argtypes = []
    L.nvfp4kv_last_cuda_error.restype = ctypes.c_char_p
    L.nvfp4kv_status_string.argtypes = [ctypes.c_int]
    L.nvfp4kv_status_string.restype = ctypes.c_char_p
    for name in ("nvfp4kv_cache_bytes", "nvfp4kv_quantize_append", "nvfp4kv_decode_workspace_size",
                 "nvfp4kv_decode_attention", "nvfp4kv_dequant_to_fp8_workspace",
                 "nvfp4kv_decode_attention_static", "nvfp4kv_append_decode_attention",
                 "nvfp4kv_tensor_amax", "nvfp4kv_calibrated_global_scale", "nvfp4kv_bf16_to_fp8_workspace",
                 "nvfp4kv_extend_attention", "nvfp4kv_quantize_append_fp8", "nvfp4kv_quantize_append_variant",
                 "nvfp4kv_stream_probe", "nvfp4kv_decode_attention_variant"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _L():
    return _lib if _lib is not None else load()


def _ptr(x) -> int | None:
    """Device pointer of a tensor (or an int address); None stays NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(func: str, status: int) -> None:
    if status != NVFP4KV_OK:
        raise Nvfp4kvError(func, status)


@dataclass
class Cache:
    """One layer's paged NVFP4 cache: one caller-owned device byte pool.

    pages: uint8 [num_pages, num_kv_heads, 2304]; each page-head holds K data
    (16 x 64 bytes), K scales (16 x 8 E4M3 bytes), V data, V scales, in that
    order (include/nvfp4kv.h).  With mxfp4=True the pool holds the MXFP4
    variant's page-heads of 2176 bytes (4 E8M0 scale bytes per row).

    k_data ([num_pages, num_kv_heads, 16, 64]) and k_scale / v_scale
    ([num_pages, num_kv_heads, 16, 8], or 4 for MXFP4) are views of the pool,
    indexed [page, head, token row, block] (V scales are stored block-major;
    their view is transposed).  V data is stored by token pair: v_pairs
    ([num_pages, num_kv_heads, 8, 128]) is the view of it, byte d of pair row p
    holding dimension d of token 2p (low nibble) and of token 2p + 1 (high
    nibble).  v_data is a copy in K's row layout ([..., 16, 64], value 2j of a
    row in the low nibble of byte j), and set_v_data writes one.
    """
    pages: object
    num_pages: int
    num_kv_heads: int
    k_global_scale: float = 1.0
    v_global_scale: float = 1.0
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    mxfp4: bool = False

    @classmethod
    def empty(cls, num_pages, num_kv_heads, device="cuda", k_global_scale=1.0, v_global_scale=1.0,
              zero=False, mxfp4=False):
        import torch

        mk = torch.zeros if zero else torch.empty
        phb = NVFP4KV_MXFP4_PAGE_HEAD_BYTES if mxfp4 else NVFP4KV_PAGE_HEAD_BYTES
        return cls(mk((num_pages, num_kv_heads, phb), dtype=torch.uint8, device=device), num_pages, num_kv_heads,
                   k_global_scale, v_global_scale, mxfp4=mxfp4)

    # byte ranges of a page-head: K data, K scales, V data, V scales
    def _parts(self):
        d = PAGE_SIZE * (HEAD_DIM // 2)
        sc = PAGE_SIZE * (HEAD_DIM // (32 if self.mxfp4 else 16))
        return (0, d), (d, d + sc), (d + sc, 2 * d + sc), (2 * d + sc, 2 * d + 2 * sc)

    def _view(self, part, row_bytes, rows=PAGE_SIZE):
        lo, hi = self._parts()[part]
        return self.pages[:, :, lo:hi].unflatten(-1, (rows, row_bytes))

    @property
    def k_data(self):
        return self._view(0, HEAD_DIM // 2)

    @property
    def k_scale(self):
        return self._view(1, HEAD_DIM // (32 if self.mxfp4 else 16))

    @property
    def v_pairs(self):
        return self._view(2, HEAD_DIM, PAGE_SIZE // 2)

    @property
    def v_data(self):
        import torch

        raw = self.v_pairs                                     # [P, H, 8, 128]: tokens 2p, 2p + 1
        nib = torch.stack((raw & 15, raw >> 4), dim=-2)         # [P, H, 8, 2, 128]
        nib = nib.reshape(*raw.shape[:2], PAGE_SIZE, HEAD_DIM)  # [P, H, 16, 128]: token, dimension
        return nib[..., 0::2] | (nib[..., 1::2] << 4)

    def set_v_data(self, rows):
        """Write V data given in K's row layout ([P, H, 16, 64] uint8, on the pool's device)."""
        import torch

        nib = torch.stack((rows & 15, rows >> 4), dim=-1)       # [P, H, 16, 64, 2]
        nib = nib.reshape(*rows.shape[:2], PAGE_SIZE // 2, 2, HEAD_DIM)
        self.v_pairs.copy_(nib[..., 0, :] | (nib[..., 1, :] << 4))

    @property
    def v_scale(self):
        lo, hi = self._parts()[3]
        blocks = HEAD_DIM // (32 if self.mxfp4 else 16)
        return self.pages[:, :, lo:hi].unflatten(-1, (blocks, PAGE_SIZE)).transpose(-1, -2)

    def c_struct(self) -> _CCache:
        return _CCache(_ptr(self.pages), int(self.num_pages), int(self.num_kv_heads), int(self.head_dim),
                       int(self.page_size), float(self.k_global_scale), float(self.v_global_scale))


def nvfp4kv_status_string(status: int) -> str:
    return _L().nvfp4kv_status_string(int(status)).decode()


def nvfp4kv_cache_bytes(num_pages: int, num_kv_heads: int, head_dim: int = HEAD_DIM,
                        page_size: int = PAGE_SIZE) -> int:
    """Bytes of the pool of a cache of this shape (9/16 byte per K or V value)."""
    n = ctypes.c_size_t()
    _check("nvfp4kv_cache_bytes",
           _L().nvfp4kv_cache_bytes(num_pages, num_kv_heads, head_dim, page_size, ctypes.byref(n)))
    return n.value


def nvfp4kv_quantize_append(cache: Cache, k, v, slot_mapping, device_status=None, stream=None) -> None:
    """k, v: bf16 [n, Hkv, 128] device tensors; slot_mapping: int64 [n] device tensor."""
    n = int(slot_mapping.shape[0]) if hasattr(slot_mapping, "shape") else int(slot_mapping[1])
    c = cache.c_struct()
    _check("nvfp4kv_quantize_append",
           _L().nvfp4kv_quantize_append(ctypes.byref(c), _ptr(k), _ptr(v), _ptr(slot_mapping), n,
                                        _ptr(device_status), _stream(stream)))


def nvfp4kv_decode_workspace_size(cache: Cache, batch: int, num_q_heads: int) -> int:
    n = ctypes.c_size_t()
    c = cache.c_struct()
    _check("nvfp4kv_decode_workspace_size",
           _L().nvfp4kv_decode_workspace_size(ctypes.byref(c), batch, num_q_heads, ctypes.byref(n)))
    return n.value


def nvfp4kv_decode_workspace_bytes(batch: int, num_q_heads: int, max_seq_len: int, num_sms: int) -> int:
    """Workspace bytes for a batch shape on a device with num_sms SMs (0 for invalid sizes)."""
    return int(_L().nvfp4kv_decode_workspace_bytes(int(batch), int(num_q_heads), int(max_seq_len), int(num_sms)))


def nvfp4kv_decode_attention(cache: Cache, q, out, page_table, seq_lens, softmax_scale: float, workspace,
                             device_status=None, stream=None, workspace_bytes: int | None = None) -> None:
    """q: bf16 [B, Hq, 128]; out: fp32 [B, Hq, 128]; page_table: int32 [B, max_pages];
    seq_lens: int32 [B]; workspace: zero-initialised device buffer (see the header)."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    maxp = int(page_table.shape[1])
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    c = cache.c_struct()
    _check("nvfp4kv_decode_attention",
           _L().nvfp4kv_decode_attention(ctypes.byref(c), _ptr(q), _ptr(out), _ptr(page_table), maxp,
                                         _ptr(seq_lens), B, Hq, float(softmax_scale), _ptr(workspace),
                                         workspace_bytes, _ptr(device_status), _stream(stream)))


def nvfp4kv_decode_attention_variant(variant: int, cache: Cache, q, out, page_table, seq_lens, softmax_scale: float,
                                     workspace, device_status=None, stream=None,
                                     workspace_bytes: int | None = None) -> None:
    """Decode attention over a format variant's cache (NVFP4KV_VARIANT_SR / _HADAMARD / _MXFP4; see
    include/nvfp4kv.h); arguments as nvfp4kv_decode_attention."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    maxp = int(page_table.shape[1])
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    c = cache.c_struct()
    _check("nvfp4kv_decode_attention_variant",
           _L().nvfp4kv_decode_attention_variant(int(variant), ctypes.byref(c), _ptr(q), _ptr(out), _ptr(page_table),
                                                 maxp, _ptr(seq_lens), B, Hq, float(softmax_scale), _ptr(workspace),
                                                 workspace_bytes, _ptr(device_status), _stream(stream)))


def nvfp4kv_append_decode_attention(cache: Cache, k, v, slot_mapping, q, out, page_table, seq_lens,
                                    softmax_scale: float, workspace, device_status=None, stream=None,
                                    workspace_bytes: int | None = None) -> None:
    """One decode step: quantize-append of k, v at slot_mapping, then decode
    attention of q over the cache (see include/nvfp4kv.h)."""
    n = int(slot_mapping.shape[0])
    B, Hq = int(q.shape[0]), int(q.shape[1])
    maxp = int(page_table.shape[1])
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    c = cache.c_struct()
    _check("nvfp4kv_append_decode_attention",
           _L().nvfp4kv_append_decode_attention(ctypes.byref(c), _ptr(k), _ptr(v), _ptr(slot_mapping), n, _ptr(q),
                                                _ptr(out), _ptr(page_table), maxp, _ptr(seq_lens), B, Hq,
                                                float(softmax_scale), _ptr(workspace), workspace_bytes,
                                                _ptr(device_status), _stream(stream)))


def nvfp4kv_decode_attention_static(cache: Cache, q, out, page_table, seq_lens, softmax_scale: float,
                                    device_status=None, stream=None) -> None:
    """nvfp4kv_decode_attention for callers that cannot allocate: the split-K
    scratch is the library's fixed device array (see include/nvfp4kv.h), so
    calls that overlap on the GPU must not be issued."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    maxp = int(page_table.shape[1])
    c = cache.c_struct()
    _check("nvfp4kv_decode_attention_static",
           _L().nvfp4kv_decode_attention_static(ctypes.byref(c), _ptr(q), _ptr(out), _ptr(page_table), maxp,
                                                _ptr(seq_lens), B, Hq, float(softmax_scale),
                                                _ptr(device_status), _stream(stream)))


def nvfp4kv_dequant_to_fp8_workspace(cache: Cache, page_table, prefix_lens, cu_prefix, ws_k, ws_v,
                                     k_ws_scale: float = 1.0, v_ws_scale: float = 1.0, device_status=None,
                                     stream=None) -> None:
    """ws_k, ws_v: uint8 [total_rows, Hkv, 128] device tensors (E4M3 bytes)."""
    B = int(prefix_lens.shape[0])
    maxp = int(page_table.shape[1])
    total_rows = int(ws_k.shape[0])
    c = cache.c_struct()
    _check("nvfp4kv_dequant_to_fp8_workspace",
           _L().nvfp4kv_dequant_to_fp8_workspace(ctypes.byref(c), _ptr(page_table), maxp, _ptr(prefix_lens),
                                                 _ptr(cu_prefix), B, total_rows, float(k_ws_scale),
                                                 float(v_ws_scale), _ptr(ws_k), _ptr(ws_v),
                                                 _ptr(device_status), _stream(stream)))


def nvfp4kv_quantize_append_variant(variant: int, cache: "Cache", k, v, slot_mapping, rand_k=None, rand_v=None,
                                    device_status=None, stream=None) -> None:
    """Quantize-append of a format variant (NVFP4KV_VARIANT_SR / _HADAMARD / _MXFP4); for MXFP4 the
    cache is an MXFP4 pool (Cache.empty(..., mxfp4=True): 4 E8M0 scale bytes per row)."""
    c = cache.c_struct()
    _check("nvfp4kv_quantize_append_variant",
           _L().nvfp4kv_quantize_append_variant(int(variant), ctypes.byref(c), _ptr(k), _ptr(v), _ptr(slot_mapping),
                                                int(k.shape[0]), _ptr(rand_k), _ptr(rand_v), _ptr(device_status),
                                                _stream(stream)))


def nvfp4kv_quantize_append_fp8(cache: "Cache", k, v, slot_mapping, ws_rows, ws_k, ws_v, k_ws_scale: float = 1.0,
                                v_ws_scale: float = 1.0, device_status=None, stream=None) -> None:
    """nvfp4kv_quantize_append and nvfp4kv_bf16_to_fp8_workspace of the same tokens in one pass."""
    n = int(k.shape[0])
    c = cache.c_struct()
    _check("nvfp4kv_quantize_append_fp8",
           _L().nvfp4kv_quantize_append_fp8(ctypes.byref(c), _ptr(k), _ptr(v), _ptr(slot_mapping), n, _ptr(ws_rows),
                                            int(ws_k.shape[0]), float(k_ws_scale), float(v_ws_scale), _ptr(ws_k),
                                            _ptr(ws_v), _ptr(device_status), _stream(stream)))


def nvfp4kv_bf16_to_fp8_workspace(k, v, ws_rows, ws_k, ws_v, k_ws_scale: float = 1.0, v_ws_scale: float = 1.0,
                                  device_status=None, stream=None) -> None:
    """The chunk's K/V (bf16 [n, Hkv, 128]) into FP8 workspace rows ws_rows[t] (int64 [n]; < 0 skips)
    of ws_k, ws_v (uint8 [total_rows, Hkv, 128])."""
    n, hkv, d = (int(x) for x in k.shape)
    _check("nvfp4kv_bf16_to_fp8_workspace",
           _L().nvfp4kv_bf16_to_fp8_workspace(_ptr(k), _ptr(v), _ptr(ws_rows), n, hkv, d, int(ws_k.shape[0]),
                                              float(k_ws_scale), float(v_ws_scale), _ptr(ws_k), _ptr(ws_v),
                                              _ptr(device_status), _stream(stream)))


def nvfp4kv_extend_attention(q, cu_q, max_q_len: int, ws_k, ws_v, cu_prefix, prefix_lens, out,
                             softmax_scale: float, k_ws_scale: float = 1.0, v_ws_scale: float = 1.0,
                             device_status=None, stream=None) -> None:
    """Causal extend attention of the chunk queries q (bf16 [total_q, Hq, 128]; sequence b owns
    [cu_q[b], cu_q[b+1])) over the FP8 workspace (uint8 [total_rows, Hkv, 128]; sequence b's key j
    at row cu_prefix[b] + j, prefix_lens[b] cached keys first); out: fp32 [total_q, Hq, 128]."""
    B = int(prefix_lens.shape[0])
    hq, d = int(q.shape[1]), int(q.shape[2])
    _check("nvfp4kv_extend_attention",
           _L().nvfp4kv_extend_attention(_ptr(q), _ptr(cu_q), int(max_q_len), _ptr(ws_k), _ptr(ws_v),
                                         _ptr(cu_prefix), _ptr(prefix_lens), B, int(ws_k.shape[0]), hq,
                                         int(ws_k.shape[1]), d, float(k_ws_scale), float(v_ws_scale),
                                         float(softmax_scale), _ptr(out), _ptr(device_status), _stream(stream)))


def nvfp4kv_tensor_amax(x, amax, accumulate: bool = False, stream=None) -> None:
    """max |x| of a contiguous bf16 device tensor into amax (a float32 device tensor of one element);
    with accumulate, max(amax, max |x|)."""
    import torch

    if x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 tensor")
    if amax.dtype != torch.float32 or amax.numel() != 1:
        raise ValueError("amax must be a one-element float32 tensor")
    _check("nvfp4kv_tensor_amax",
           _L().nvfp4kv_tensor_amax(_ptr(x) if x.numel() else None, int(x.numel()), _ptr(amax),
                                    int(bool(accumulate)), _stream(stream)))


def nvfp4kv_stream_probe(cache: Cache, page_table, seq_lens, sink, mode: int = NVFP4KV_PROBE_DECODE_PATTERN,
                         device_status=None, stream=None) -> None:
    """Read every cached page-head of the batch once with no attention math (a measurement aid):
    the decode's pattern, or whole pages by bulk copy; sink: a uint32 device tensor of one element."""
    c = cache.c_struct()
    _check("nvfp4kv_stream_probe",
           _L().nvfp4kv_stream_probe(ctypes.byref(c), _ptr(page_table), int(page_table.shape[1]), _ptr(seq_lens),
                                     int(seq_lens.shape[0]), int(mode), _ptr(sink), _ptr(device_status),
                                     _stream(stream)))


def nvfp4kv_calibrated_global_scale(amax: float) -> float:
    """The FP32 global scale that maps amax onto 6 * 448 (1.0 when amax == 0)."""
    g = ctypes.c_float()
    _check("nvfp4kv_calibrated_global_scale", _L().nvfp4kv_calibrated_global_scale(float(amax), ctypes.byref(g)))
    return g.value


__all__ = ["Cache", "Nvfp4kvError", "load", "NVFP4KV_PAGE_HEAD_BYTES", "NVFP4KV_MXFP4_PAGE_HEAD_BYTES",
           "nvfp4kv_cache_bytes", "nvfp4kv_quantize_append",
           "nvfp4kv_decode_workspace_size", "nvfp4kv_decode_workspace_bytes", "nvfp4kv_decode_attention", "nvfp4kv_dequant_to_fp8_workspace",
           "nvfp4kv_status_string", "nvfp4kv_decode_attention_static", "nvfp4kv_append_decode_attention",
           "nvfp4kv_tensor_amax", "nvfp4kv_calibrated_global_scale", "nvfp4kv_bf16_to_fp8_workspace",
           "nvfp4kv_extend_attention", "nvfp4kv_quantize_append_fp8", "nvfp4kv_quantize_append_variant",
           "nvfp4kv_stream_probe", "NVFP4KV_PROBE_DECODE_PATTERN", "NVFP4KV_PROBE_WHOLE_PAGES",
           "nvfp4kv_decode_attention_variant"]
