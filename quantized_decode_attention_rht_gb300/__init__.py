"""Rotate-then-quantize KV-cache compression and decode attention for GB300 (sm_103a).

This module is a thin ctypes binding over ``libkvq.so`` (C ABI in ``include/kvq.h``):
each ``kvq_*`` function here marshals torch tensors (device pointers, the current CUDA
stream) into the C call of the same name and raises ``KvqError`` on a failed status.
All arithmetic of the method runs in the library's CUDA kernels; there is no CPU path.
PyTorch is used for device memory and streams only.

``PagedCache`` is a convenience owner of one tier's device buffers (pool rows, side
data, codebook tables, signs) laid out as the header describes.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

FMT_CODEBOOK, FMT_FP16, FMT_FP8_E4M3, FMT_INT4_G32, FMT_CODEBOOK_QJL, FMT_CODEBOOK_OUTLIER = 0, 1, 2, 3, 4, 5
FORMATS = {"codebook": FMT_CODEBOOK, "fp16": FMT_FP16, "fp8_e4m3": FMT_FP8_E4M3, "int4_g32": FMT_INT4_G32,
           "codebook_qjl": FMT_CODEBOOK_QJL, "codebook_outlier": FMT_CODEBOOK_OUTLIER}
QJL_DIM = 128
OUTLIER_CHANNELS = 8
MAX_TIERS = 4
INT4_GROUP = 32

STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARGUMENT", 2: "KVQ_ERR_UNSUPPORTED",
          3: "KVQ_ERR_WORKSPACE_TOO_SMALL", 4: "KVQ_ERR_CUDA"}


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class KvqCache(ctypes.Structure):
    """Mirror of ``struct kvq_cache``."""

    _fields_ = [
        ("head_dim", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("k_format", ctypes.c_int32), ("v_format", ctypes.c_int32),
        ("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32),
        ("k_rows", ctypes.c_void_p), ("v_rows", ctypes.c_void_p),
        ("k_aux", ctypes.c_void_p), ("v_aux", ctypes.c_void_p),
        ("k_centroids", ctypes.c_void_p), ("k_bounds", ctypes.c_void_p),
        ("v_centroids", ctypes.c_void_p), ("v_bounds", ctypes.c_void_p),
        ("k_signs", ctypes.c_void_p), ("v_signs", ctypes.c_void_p),
        ("k_qjl", ctypes.c_void_p), ("k_outliers", ctypes.c_void_p),
    ]


class KvqTierView(ctypes.Structure):
    """Mirror of ``struct kvq_tier_view``."""

    _fields_ = [("cache", ctypes.POINTER(KvqCache)), ("block_table", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("max_pages", ctypes.c_int32)]


class KvqDecodeOptions(ctypes.Structure):
    """Mirror of ``struct kvq_decode_options``."""

    _fields_ = [("score_gate", ctypes.c_int32), ("spike_flags", ctypes.c_void_p), ("status", ctypes.c_void_p)]


SCORE_GATE_NATS = 16.0
# device-side error bits of a decode call (kvq_decode_options.status)
DEVERR_COPY_TIMEOUT, DEVERR_PAGE_INDEX, DEVERR_SEQ_LEN = 1, 2, 4

_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded libkvq.so.  Raises if it has not been built (no fallback exists)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m quantized_decode_attention_rht_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        h.kvq_status_string.restype = ctypes.c_char_p
        h.kvq_status_string.argtypes = [ctypes.c_int]
        h.kvq_kernel_launches.restype = ctypes.c_uint64
        h.kvq_kernel_launches.argtypes = []
        i32, vp, sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
        dp, fp = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)
        szp = ctypes.POINTER(ctypes.c_size_t)
        sigs = {
            "kvq_row_bytes": [i32, i32, i32, szp, szp],
            "kvq_lloyd_max_codebook": [i32, dp, dp],
            "kvq_uniform_codebook": [i32, dp, dp],
            "kvq_codebook_tables": [i32, dp, fp, fp],
            "kvq_make_signs": [ctypes.c_uint64, i32, i32, i32, vp, vp],
            "kvq_quantize_append": [ctypes.POINTER(KvqCache), vp, vp, i32, vp, vp],
            "kvq_requantize": [ctypes.POINTER(KvqCache), vp, ctypes.POINTER(KvqCache), vp, i32, vp],
            "kvq_outlier_calibrate": [vp, i32, i32, i32, vp, vp],
            "kvq_decode_workspace_size": [ctypes.POINTER(KvqTierView), i32, i32, i32, i32, szp],
            "kvq_decode_attention": [ctypes.POINTER(KvqTierView), i32, vp, i32, i32, i32, vp, vp, sz, vp],
            "kvq_decode_attention_ex": [ctypes.POINTER(KvqTierView), i32, vp, i32, i32, i32, vp, vp, sz,
                                        ctypes.POINTER(KvqDecodeOptions), vp],
            "kvq_decode_attention_noalloc": [ctypes.POINTER(KvqTierView), i32, vp, i32, i32, i32, vp, vp],
        }
        for name, args in sigs.items():
            f = getattr(h, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        _lib_handle = h
    return _lib_handle


def _check(status: int, what: str) -> None:
    if status != 0:
        raise KvqError(status, what)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dense(*tensors) -> None:
    """The C ABI takes dense row-major buffers: refuse strided views rather than read them
    in the wrong order."""
    for t in tensors:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors passed to libkvq must be contiguous")


def _arg(t, name: str, dtype: str, shape=None, min_numel: int = 0) -> None:
    """The C ABI takes device pointers of fixed element types: refuse a host tensor, another
    dtype, a shape that disagrees with the call (None entries in `shape` are free) or fewer
    elements than the call reads, before the library is called."""
    if t is None:
        return
    import torch
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != getattr(torch, dtype):
        raise TypeError(f"{name} must be torch.{dtype}, got {t.dtype}")
    if shape is not None and (t.dim() != len(shape) or any(w is not None and w != n for w, n in zip(shape, t.shape))):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)} (None: any)")
    if t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the call reads {min_numel}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


# ----------------------------------------------------------------------------- host-side entry points


def kvq_status_string(status: int) -> str:
    return lib().kvq_status_string(status).decode()


def kvq_kernel_launches() -> int:
    """Kernels this library has launched since it was loaded (all devices and streams)."""
    return int(lib().kvq_kernel_launches())


def kvq_row_bytes(fmt, bits: int, head_dim: int):
    fmt = FORMATS.get(fmt, fmt)
    row, aux = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().kvq_row_bytes(fmt, bits, head_dim, ctypes.byref(row), ctypes.byref(aux)), "kvq_row_bytes")
    return row.value, aux.value


def _codebook(fn, bits):
    n = 1 << bits
    c = np.zeros(n, dtype=np.float64)
    b = np.zeros(n - 1, dtype=np.float64)
    _check(fn(bits, c.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
              b.ctypes.data_as(ctypes.POINTER(ctypes.c_double))), fn.__name__)
    return c, b


def kvq_lloyd_max_codebook(bits: int):
    return _codebook(lib().kvq_lloyd_max_codebook, bits)


def kvq_uniform_codebook(bits: int):
    return _codebook(lib().kvq_uniform_codebook, bits)


def kvq_codebook_tables(bits: int, centroids: np.ndarray):
    n = 1 << bits
    c = np.ascontiguousarray(centroids, dtype=np.float64)
    c32 = np.zeros(n, dtype=np.float32)
    b32 = np.zeros(n - 1, dtype=np.float32)
    _check(lib().kvq_codebook_tables(bits, c.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                     c32.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                     b32.ctypes.data_as(ctypes.POINTER(ctypes.c_float))), "kvq_codebook_tables")
    return c32, b32


def kvq_make_signs(seed: int, layer: int, num_kv_heads: int, head_dim: int):
    """int8 [num_kv_heads, head_dim] +1/-1 sign vectors for keys and values of one layer
    (numpy arrays, computed on the host by the library)."""
    k = np.zeros((num_kv_heads, head_dim), dtype=np.int8)
    v = np.zeros((num_kv_heads, head_dim), dtype=np.int8)
    _check(lib().kvq_make_signs(seed & ((1 << 64) - 1), layer, num_kv_heads, head_dim, k.ctypes.data, v.ctypes.data),
           "kvq_make_signs")
    return k, v


# ----------------------------------------------------------------------------- GPU entry points


def kvq_quantize_append(cache: KvqCache, k, v, slot_mapping, stream=None) -> None:
    """k, v: fp16 CUDA tensors [T, Hkv, D] (either may be None); slot_mapping: int32 [T]."""
    _dense(k, v, slot_mapping)
    if k is None and v is None:
        raise ValueError("kvq_quantize_append needs k or v")
    t = (k if k is not None else v).shape[0]
    for x, name in ((k, "k"), (v, "v")):
        _arg(x, name, "float16", (t, cache.num_kv_heads, cache.head_dim))
    _arg(slot_mapping, "slot_mapping", "int32", (None,), min_numel=t)
    _check(lib().kvq_quantize_append(ctypes.byref(cache), _ptr(k), _ptr(v), t, _ptr(slot_mapping),
                                     _stream(stream)), "kvq_quantize_append")


def kvq_outlier_calibrate(k, out_idx, stream=None) -> None:
    """k: fp16 CUDA tensor [N, Hkv, D] (the calibration tokens' keys); out_idx: int32 CUDA
    tensor [Hkv, OUTLIER_CHANNELS], written with each head's largest-variance channels."""
    _dense(k, out_idx)
    _arg(k, "k", "float16", (None, None, None))
    n, hkv, d = k.shape
    _arg(out_idx, "out_idx", "int32", (hkv, OUTLIER_CHANNELS))
    _check(lib().kvq_outlier_calibrate(_ptr(k), n, hkv, d, _ptr(out_idx), _stream(stream)), "kvq_outlier_calibrate")


def kvq_requantize(src: KvqCache, src_slots, dst: KvqCache, dst_slots, stream=None) -> None:
    """Move tokens from an fp16 tier (a recent-token window) into another tier, re-encoding
    their rows; src_slots / dst_slots: int32 CUDA tensors [T]."""
    _dense(src_slots, dst_slots)
    _arg(src_slots, "src_slots", "int32", (None,))
    _arg(dst_slots, "dst_slots", "int32", (None,), min_numel=int(src_slots.shape[0]))
    _check(lib().kvq_requantize(ctypes.byref(src), _ptr(src_slots), ctypes.byref(dst), _ptr(dst_slots),
                                int(src_slots.shape[0]), _stream(stream)), "kvq_requantize")


def _views(tiers: Sequence["TierView"], batch: int = 0):
    """The tiers as the C ABI's array; `batch` > 0: the call reads that many rows of every
    block table and entries of every length array."""
    arr = (KvqTierView * len(tiers))()
    for i, t in enumerate(tiers):
        _dense(t.block_table, t.seq_lens)
        _arg(t.block_table, "block_table", "int32", (None, None))
        _arg(t.seq_lens, "seq_lens", "int32", (None,), min_numel=batch)
        if batch and t.block_table is not None and t.block_table.shape[0] < batch:
            raise ValueError(f"block_table has {t.block_table.shape[0]} rows for {batch} sequences")
        arr[i].cache = ctypes.pointer(t.cache.struct)
        arr[i].block_table = _ptr(t.block_table)
        arr[i].seq_lens = _ptr(t.seq_lens)
        arr[i].max_pages = int(t.block_table.shape[1]) if t.block_table is not None else 0
    return arr


def kvq_decode_workspace_size(tiers, batch: int, num_q_heads: int, split_tokens: int = 0) -> int:
    arr = _views(tiers)
    n = ctypes.c_size_t()
    _check(lib().kvq_decode_workspace_size(arr, len(tiers), batch, num_q_heads, split_tokens, ctypes.byref(n)),
           "kvq_decode_workspace_size")
    return n.value


def _decode_args(tiers, q, out):
    """q: fp16 [B, Hq, D] with D the tiers' head_dim; out: fp32 of q's shape.  Returns (B, Hq)."""
    if not tiers:
        raise ValueError("decode attention needs at least one tier")
    _arg(q, "q", "float16", (None, None, tiers[0].cache.struct.head_dim))
    _arg(out, "out", "float32", tuple(q.shape))
    return int(q.shape[0]), int(q.shape[1])


def kvq_decode_attention(tiers, q, out, workspace, split_tokens: int = 0, stream=None, score_gate: bool = False,
                         spike_flags=None, status=None) -> None:
    """q: fp16 [B, Hq, D]; out: fp32 [B, Hq, D]; workspace: uint8 CUDA tensor.
    score_gate / spike_flags (int32 [B, Hq] CUDA tensor) / status (int32 CUDA tensor of one
    element, receives the call's DEVERR_* bits): the options of kvq_decode_attention_ex
    (FoveatedKV score-gated value loading and spike detection, the device error report)."""
    _dense(q, out, workspace, spike_flags, status)
    b, hq = _decode_args(tiers, q, out)
    _arg(spike_flags, "spike_flags", "int32", (b, hq))
    _arg(status, "status", "int32", None, min_numel=1)
    if workspace is not None and not getattr(workspace, "is_cuda", False):
        raise ValueError("workspace must be a CUDA tensor")
    arr = _views(tiers, b)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if not score_gate and spike_flags is None and status is None:
        _check(lib().kvq_decode_attention(arr, len(tiers), _ptr(q), b, hq, split_tokens, _ptr(out),
                                          _ptr(workspace), ws_bytes, _stream(stream)), "kvq_decode_attention")
        return
    opts = KvqDecodeOptions(1 if score_gate else 0, _ptr(spike_flags), _ptr(status))
    _check(lib().kvq_decode_attention_ex(arr, len(tiers), _ptr(q), b, hq, split_tokens, _ptr(out), _ptr(workspace),
                                         ws_bytes, ctypes.byref(opts), _stream(stream)), "kvq_decode_attention_ex")


NOALLOC_SCRATCH_BYTES = 32 << 20


def kvq_decode_attention_noalloc(tiers, q, out, split_tokens: int = 0, stream=None) -> None:
    """Decode attention using the library's static device scratch (no allocation anywhere);
    for callers that may not allocate device memory.  Calls that overlap on the GPU race on
    the shared scratch."""
    _dense(q, out)
    b, hq = _decode_args(tiers, q, out)
    arr = _views(tiers, b)
    _check(lib().kvq_decode_attention_noalloc(arr, len(tiers), _ptr(q), b, hq, split_tokens, _ptr(out),
                                              _stream(stream)), "kvq_decode_attention_noalloc")


# ----------------------------------------------------------------------------- device buffers


class PagedCache:
    """Owns the device buffers of one tier (torch allocations) and its ``KvqCache`` struct.

    k_format / v_format: "codebook" | "fp16" | "fp8_e4m3" | "int4_g32", and for keys also
    "codebook_qjl" (codes + residual sign sketch); codebook tiers take `k_bits` / `v_bits` and
    a codebook kind ("lloyd_max" or "uniform") computed by the library.
    k_signs / v_signs: int8 [Hkv, D] tensors or arrays of +1/-1 (shared by every tier).
    k_qjl: float32 [QJL_DIM, D] projection (tensor or array) for "codebook_qjl" keys.
    k_outliers: int32 [Hkv, OUTLIER_CHANNELS] channels (tensor or array) for
    "codebook_outlier" keys (e.g. from kvq_outlier_calibrate)."""

    def __init__(self, head_dim, num_kv_heads, num_pages, k_format, v_format, k_bits=0, v_bits=0,
                 k_signs=None, v_signs=None, page_size=16, codebook="lloyd_max", device="cuda", k_qjl=None,
                 k_outliers=None):
        import torch
        self.head_dim, self.num_kv_heads, self.num_pages, self.page_size = head_dim, num_kv_heads, num_pages, page_size
        self.k_format, self.v_format = FORMATS.get(k_format, k_format), FORMATS.get(v_format, v_format)
        self.k_bits, self.v_bits = k_bits, v_bits
        dev = torch.device(device)

        def side(fmt, bits):
            row, aux = kvq_row_bytes(fmt, bits, head_dim)
            rows = torch.zeros((num_pages, num_kv_heads, page_size, row), dtype=torch.uint8, device=dev)
            a = None
            if aux and fmt == FMT_CODEBOOK_OUTLIER:  # byte records (norm, scale, int8 values)
                a = torch.zeros((num_pages, num_kv_heads, page_size, aux), dtype=torch.uint8, device=dev)
            elif aux:
                a = torch.zeros((num_pages, num_kv_heads, page_size, aux // 2), dtype=torch.float16, device=dev)
            cent = bnd = None
            if fmt in (FMT_CODEBOOK, FMT_CODEBOOK_QJL, FMT_CODEBOOK_OUTLIER):
                c = (kvq_lloyd_max_codebook if codebook == "lloyd_max" else kvq_uniform_codebook)(bits)[0]
                c32, b32 = kvq_codebook_tables(bits, c)
                cent = torch.from_numpy(c32).to(dev)
                bnd = torch.from_numpy(b32).to(dev)
            return rows, a, cent, bnd

        self.k_rows, self.k_aux, self.k_centroids, self.k_bounds = side(self.k_format, k_bits)
        self.v_rows, self.v_aux, self.v_centroids, self.v_bounds = side(self.v_format, v_bits)
        self.k_signs = torch.as_tensor(np.asarray(k_signs, dtype=np.int8)).to(dev) if not hasattr(k_signs, "data_ptr") else k_signs
        self.v_signs = torch.as_tensor(np.asarray(v_signs, dtype=np.int8)).to(dev) if not hasattr(v_signs, "data_ptr") else v_signs
        self.k_qjl = None
        if k_qjl is not None:
            self.k_qjl = (k_qjl if hasattr(k_qjl, "data_ptr")
                          else torch.as_tensor(np.asarray(k_qjl, dtype=np.float32)).to(dev)).contiguous()
        s = KvqCache()
        s.head_dim, s.num_kv_heads, s.page_size, s.num_pages = head_dim, num_kv_heads, page_size, num_pages
        s.k_format, s.v_format, s.k_bits, s.v_bits = self.k_format, self.v_format, k_bits, v_bits
        s.k_rows, s.v_rows = _ptr(self.k_rows), _ptr(self.v_rows)
        s.k_aux, s.v_aux = _ptr(self.k_aux), _ptr(self.v_aux)
        s.k_centroids, s.k_bounds = _ptr(self.k_centroids), _ptr(self.k_bounds)
        s.v_centroids, s.v_bounds = _ptr(self.v_centroids), _ptr(self.v_bounds)
        s.k_signs, s.v_signs = _ptr(self.k_signs), _ptr(self.v_signs)
        s.k_qjl = _ptr(self.k_qjl)
        self.k_outliers = None
        if k_outliers is not None:
            self.k_outliers = (k_outliers if hasattr(k_outliers, "data_ptr")
                               else torch.as_tensor(np.asarray(k_outliers, dtype=np.int32)).to(dev)).contiguous()
        s.k_outliers = _ptr(self.k_outliers)
        self.struct = s

    def append(self, k, v, slot_mapping, stream=None) -> None:
        kvq_quantize_append(self.struct, k, v, slot_mapping, stream)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.k_rows, self.v_rows, self.k_aux, self.v_aux)
                   if t is not None)


class TierView:
    """A tier as seen by one decode call: cache + block table [B, max_pages] + lens [B] (int32)."""

    def __init__(self, cache: PagedCache, block_table, seq_lens):
        self.cache, self.block_table, self.seq_lens = cache, block_table, seq_lens
