"""Encode K/V vectors into a paged pool, and read them back (oracle; test infrastructure).

Sources:
  * VeloxQuant-MLX page, section "Stage 2: Lloyd-Max Scalar Quantization": after
    the rotation each vector is normalised to unit norm, the norm is kept as fp16,
    and every coordinate is replaced by the index of its nearest centroid.
  * VeloxQuant-MLX page, section "Memory Layout: What Actually Gets Stored": per
    token and head the record is the packed indices plus the fp16 norm.
  * FoveatedKV page, section "The VR headset thing": near tier fp16, far tier fp8
    E4M3 keys and INT4 values; every token still contributes to attention.

Readings taken:
  * unit-norm coordinates of a d-dimensional rotated vector are about N(0, 1/d),
    so the N(0,1) codebook is applied to u = sqrt(d) * x~ / ||x~||, and a code
    decodes to ||x~||_fp16 * C[idx] / sqrt(d) (normalise by the exact norm, store
    it as fp16, decode with the stored fp16 norm);
  * a zero vector has norm 0 and u = 0;
  * "nearest centroid" is taken as idx = #{i : u > Bd_i} with the float32 midpoint
    boundaries, so a value exactly on a boundary goes to the lower index;
  * fp16 / fp8 / INT4 tiers store the rotated vector x~ itself (no unit norm);
  * pool layout: rows[page][kv_head][slot_in_page][row_bytes], side data
    (fp16 norm or fp16 group scales) aux[page][kv_head][slot_in_page][...]; a token
    of sequence b at position t lives in page block_table[b][t // page_size] at slot
    t % page_size.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

from . import formats
from .rotation import rotate, unrotate

CODEBOOK, FP16, FP8_E4M3, INT4_G32 = "codebook", "fp16", "fp8_e4m3", "int4_g32"


def encode(x16: np.ndarray, s: np.ndarray, fmt: str, bits: int = 0,
           bounds32: Optional[np.ndarray] = None):
    """Encode fp16 vectors x16 [..., d] rotated with signs s [d] (broadcastable).
    Returns (rows uint8 [..., row_bytes], aux or None):
      codebook: aux = fp16 norms [...];  int4_g32: aux = fp16 scales [..., d/32]."""
    d = x16.shape[-1]
    xr = rotate(np.asarray(x16, dtype=np.float64), s)
    if fmt == CODEBOOK:
        n = np.sqrt(np.sum(xr * xr, axis=-1))
        norm16 = formats.to_f16(n)
        with np.errstate(divide="ignore", invalid="ignore"):
            u = np.where(n[..., None] > 0, math.sqrt(d) * xr / n[..., None], 0.0)
        u32 = formats.to_f32(u)
        idx = np.sum(u32[..., None] > np.asarray(bounds32, dtype=np.float32), axis=-1)
        return formats.pack_bits(idx, bits), norm16
    if fmt == FP16:
        return formats.to_f16(xr).view(np.uint8).reshape(*xr.shape[:-1], 2 * d), None
    if fmt == FP8_E4M3:
        return formats.e4m3_encode(formats.to_f32(xr)), None
    if fmt == INT4_G32:
        nib, scales = formats.int4_g32_encode(formats.to_f32(xr))
        return formats.pack_bits(nib, 4), scales
    raise ValueError(fmt)


def decode_rotated(rows: np.ndarray, aux, fmt: str, d: int, bits: int = 0,
                   centroids32: Optional[np.ndarray] = None) -> np.ndarray:
    """Stored rows -> the dequantised vector in the rotated domain (float64 [..., d])."""
    rows = np.asarray(rows, dtype=np.uint8)
    if fmt == CODEBOOK:
        idx = formats.unpack_bits(rows, bits, d)
        c = np.asarray(centroids32, dtype=np.float32).astype(np.float64)
        return c[idx] * np.asarray(aux, dtype=np.float64)[..., None] / math.sqrt(d)
    if fmt == FP16:
        return np.ascontiguousarray(rows).view(np.float16).astype(np.float64)
    if fmt == FP8_E4M3:
        return formats.e4m3_decode(rows)
    if fmt == INT4_G32:
        return formats.int4_g32_decode(formats.unpack_bits(rows, 4, d), aux)
    raise ValueError(fmt)


def decode(rows, aux, fmt, s, d, bits=0, centroids32=None) -> np.ndarray:
    """Stored rows -> dequantised vector in the original domain (rotation undone)."""
    return unrotate(decode_rotated(rows, aux, fmt, d, bits, centroids32), s)


@dataclasses.dataclass
class Side:
    """One of K or V in a tier: format, code bits, codebook tables, signs, pool arrays."""

    fmt: str
    bits: int
    centroids32: Optional[np.ndarray]
    bounds32: Optional[np.ndarray]
    signs: np.ndarray  # int8 [Hkv, d]
    rows: np.ndarray  # uint8 [num_pages, Hkv, page_size, row_bytes]
    aux: Optional[np.ndarray]  # fp16 [num_pages, Hkv, page_size(, d/32)]


def new_side(fmt, bits, centroids32, bounds32, signs, num_pages, num_kv_heads, page_size, d) -> Side:
    rb = formats.row_bytes(fmt, bits, d)
    rows = np.zeros((num_pages, num_kv_heads, page_size, rb), dtype=np.uint8)
    aux = None
    if fmt == CODEBOOK:
        aux = np.zeros((num_pages, num_kv_heads, page_size), dtype=np.float16)
    elif fmt == INT4_G32:
        aux = np.zeros((num_pages, num_kv_heads, page_size, d // formats.GROUP), dtype=np.float16)
    return Side(fmt, bits, centroids32, bounds32, signs, rows, aux)


def write(side: Side, slots: np.ndarray, x16: np.ndarray, page_size: int) -> None:
    """Encode x16 [T, Hkv, d] and store token i at pool slot slots[i] (slot = page *
    page_size + offset); a negative slot skips the token."""
    slots = np.asarray(slots, dtype=np.int64)
    keep = slots >= 0
    page, off = slots[keep] // page_size, slots[keep] % page_size
    for h in range(x16.shape[1]):
        rows, aux = encode(x16[keep, h, :], side.signs[h], side.fmt, side.bits, side.bounds32)
        side.rows[page, h, off] = rows
        if side.aux is not None:
            side.aux[page, h, off] = aux


def gather(side: Side, block_row: np.ndarray, length: int, h: int, page_size: int):
    """Rows (and side data) of tokens 0..length-1 of one sequence, kv head h."""
    t = np.arange(length)
    page = np.asarray(block_row)[t // page_size]
    off = t % page_size
    rows = side.rows[page, h, off]
    aux = None if side.aux is None else side.aux[page, h, off]
    return rows, aux


def read(side: Side, block_row: np.ndarray, length: int, h: int, page_size: int) -> np.ndarray:
    """Dequantised vectors (original domain, float64 [length, d]) of one sequence's head h."""
    rows, aux = gather(side, block_row, length, h, page_size)
    d = side.signs.shape[-1]
    return decode(rows, aux, side.fmt, side.signs[h], d, side.bits, side.centroids32)
