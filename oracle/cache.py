"""Encode K/V vectors into a paged pool, and read them back (oracle; test infrastructure).

Sources:
  * VeloxQuant-MLX page, section "Stage 2: Lloyd-Max Scalar Quantization": after
    the rotation each vector is normalised to unit norm, the norm is kept as fp16,
    and every coordinate is replaced by the index of its nearest centroid.
  * VeloxQuant-MLX page, section "Memory Layout: What Actually Gets Stored": per
    token and head the record is the packed indices plus the fp16 norm.
  * FoveatedKV page, section "The VR headset thing": near tier fp16, far tier fp8
    E4M3 keys and INT4 values; every token still contributes to attention.
  * VeloxQuant-MLX page, section "Stage 3: QJL Residual Correction" (TurboQuantProd):
    the residual r = k - k^ of the codebook encode is not stored; only the signs
    z = sign(S r) of a random Johnson-Lindenstrauss projection (m = 128 rows) and the
    residual norm ||r|| as fp16; its "Memory Layout" table: for d = 128 and 3-bit codes
    48 B of codes + 16 B of signs + 2 B residual norm + 2 B norm = 68 B per key.
  * VeloxQuant-MLX page, section "Outlier Two-Stream Cache": calibrate per-channel
    variance over the first N tokens, pick the top-K channels, store them as int8 with a
    per-token scale and encode the rest (outliers zeroed) as usual; attend adds the
    outlier inner product to the inlier score.

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
    t % page_size;
  * residual sketch: taken in the rotated domain, z = sign(S r~) with r~ = x~ - x^~
    (x^~ the dequantised rotated vector, exactly what the decoder reconstructs) and S
    an m x d matrix of iid N(0,1) entries -- equal in distribution to sketching the
    unrotated residual, since the rotation is orthogonal; sign(0) = +1; the m sign
    bits follow the codes in the row, LSB-first like the codes; side data is
    (fp16 norm, fp16 ||r~||);
  * outlier two-stream (keys): K = 8 channels per kv head, chosen by population variance
    over the calibration tokens (ties to the lower channel); the channels are those of the
    unrotated vector, zeroed before the rotation; int8 q = clamp(rint(x / s), +-127) with
    s = fp16(max|x| / 127) per token; side data is fp16 norm, fp16 s, then the K int8
    values (12 bytes; the page counts 16 extra bytes per token for K = 8, "8 x 2", a
    layout it does not spell out -- here the values and their scale take 10).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

from . import formats
from .rotation import rotate, unrotate

CODEBOOK, FP16, FP8_E4M3, INT4_G32 = "codebook", "fp16", "fp8_e4m3", "int4_g32"
CODEBOOK_QJL = "codebook_qjl"
CODEBOOK_OUTLIER = "codebook_outlier"
QJL_DIM = formats.QJL_DIM
OUTLIER_CHANNELS = formats.OUTLIER_CHANNELS


def outlier_channels(k16: np.ndarray, count: int = OUTLIER_CHANNELS) -> np.ndarray:
    """Calibration of the outlier two-stream cache (VeloxQuant-MLX page, "Outlier Two-Stream
    Cache", steps 1-2): over the calibration tokens k16 [N, Hkv, d], the population variance
    of every channel of every kv head; per head the `count` channels of largest variance,
    largest first, ties to the lower channel.  Returns int32 [Hkv, count]."""
    x = np.asarray(k16, dtype=np.float64)
    var = x.var(axis=0)  # [Hkv, d]
    d = x.shape[-1]
    out = np.empty((x.shape[1], count), dtype=np.int32)
    for h in range(x.shape[1]):
        order = np.lexsort((np.arange(d), -var[h]))  # by variance descending, then index
        out[h] = order[:count]
    return out


def pack_outlier_aux(norm16, scale16, q) -> np.ndarray:
    """Side data of a codebook_outlier row, 4 + K bytes: fp16 norm, fp16 outlier scale (both
    little-endian), then the K int8 outlier values in the order of the channel list."""
    norm16 = np.asarray(norm16, dtype=np.float16)
    lead = norm16.shape
    out = np.empty(lead + (4 + OUTLIER_CHANNELS,), dtype=np.uint8)
    out[..., 0:2] = norm16[..., None].view(np.uint8).reshape(lead + (2,))
    out[..., 2:4] = np.asarray(scale16, dtype=np.float16)[..., None].view(np.uint8).reshape(lead + (2,))
    out[..., 4:] = np.asarray(q, dtype=np.int8).view(np.uint8)
    return out


def unpack_outlier_aux(aux):
    """(norm fp16 [...], scale fp16 [...], q int8 [..., K]) of codebook_outlier side data."""
    a = np.ascontiguousarray(aux, dtype=np.uint8)
    norm16 = a[..., 0:2].copy().view(np.float16)[..., 0]
    scale16 = a[..., 2:4].copy().view(np.float16)[..., 0]
    return norm16, scale16, a[..., 4:].copy().view(np.int8)


def encode(x16: np.ndarray, s: np.ndarray, fmt: str, bits: int = 0,
           bounds32: Optional[np.ndarray] = None, centroids32: Optional[np.ndarray] = None,
           proj: Optional[np.ndarray] = None, outliers: Optional[np.ndarray] = None):
    """Encode fp16 vectors x16 [..., d] rotated with signs s [d] (broadcastable).
    Returns (rows uint8 [..., row_bytes], aux or None):
      codebook: aux = fp16 norms [...];  int4_g32: aux = fp16 scales [..., d/32];
      codebook_qjl: aux = fp16 [..., 2] (norm, residual norm); needs centroids32 and
      the projection proj [m, d] (float32);
      codebook_outlier: aux = uint8 [..., 4 + K] (pack_outlier_aux); needs the head's K
      outlier channels `outliers` (original-domain indices)."""
    if fmt == CODEBOOK_OUTLIER:
        # VeloxQuant-MLX page, "Outlier Two-Stream Cache", step 3: the outlier channels go
        # to int8 with a per-token scale; the inlier vector, those channels zeroed in the
        # original domain, is encoded as usual (rotation, unit norm, codebook)
        x = np.asarray(x16, dtype=np.float64)
        idx = np.asarray(outliers, dtype=np.int64)
        x_in = x.copy()
        x_in[..., idx] = 0.0
        codes, norm16 = encode_rotated(rotate(x_in, s), CODEBOOK, bits, bounds32)
        q, scale16 = formats.outlier_int8_encode(x[..., idx])
        return codes, pack_outlier_aux(norm16, scale16, q)
    return encode_rotated(rotate(np.asarray(x16, dtype=np.float64), s), fmt, bits, bounds32, centroids32, proj)


def encode_rotated(xr: np.ndarray, fmt: str, bits: int = 0, bounds32: Optional[np.ndarray] = None,
                   centroids32: Optional[np.ndarray] = None, proj: Optional[np.ndarray] = None):
    """The encode of an already rotated vector x~ (float64 [..., d]): everything `encode`
    does after the rotation.  Same returns."""
    d = xr.shape[-1]
    if fmt == CODEBOOK_OUTLIER:
        raise ValueError("codebook_outlier splits channels of the unrotated vector: use encode")
    if fmt == CODEBOOK_QJL:
        # 1. the codebook encode of x~ (codes of `bits` bits, fp16 norm)
        codes, norm16 = encode_rotated(xr, CODEBOOK, bits, bounds32)
        # 2. the residual against what the decoder reconstructs
        r = xr - decode_rotated(codes, norm16, CODEBOOK, d, bits, centroids32)
        rnorm16 = formats.to_f16(np.sqrt(np.sum(r * r, axis=-1)))
        # 3. signs of the projection, decided on the float32 value: z_j = 1 <=> (S r)_j >= 0
        sr = formats.to_f32(r @ np.asarray(proj, dtype=np.float32).astype(np.float64).T)
        zbits = (sr >= 0).astype(np.int64)
        rows = np.concatenate([codes, formats.pack_bits(zbits, 1)], axis=-1)
        return rows, np.stack([norm16, rnorm16], axis=-1)
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
    if fmt == CODEBOOK_OUTLIER:  # the inlier part; decode() adds the outlier channels
        return decode_rotated(rows, unpack_outlier_aux(aux)[0], CODEBOOK, d, bits, centroids32)
    if fmt == CODEBOOK_QJL:  # the codebook part; qjl_correction() adds the sketch's term
        nb = (d * bits + 7) // 8
        return decode_rotated(rows[..., :nb], np.asarray(aux)[..., 0], CODEBOOK, d, bits, centroids32)
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


def qjl_correction(rows: np.ndarray, aux, q_rot: np.ndarray, proj: np.ndarray, d: int, bits: int) -> np.ndarray:
    """The sketch's estimate of <q~, r~> for stored codebook_qjl rows [..., row_bytes] and a
    rotated query q_rot [d]:  ||r~|| * sqrt(pi/2) / m * sum_j z_j <S_j, q~>,  z_j = +-1.

    VeloxQuant-MLX page, "Stage 3": the correction is unbiased.  For S_j ~ N(0, I),
    E[sign(<S_j, r>) <S_j, q>] = sqrt(2/pi) <q, r> / ||r||, so this is the unbiased
    estimator of that construction (the page's printed factor reads pi/(2m) and puts a
    sign on <S_j, q>; that form is neither unbiased nor proportional to ||q||)."""
    nb = (d * bits + 7) // 8
    z = 2.0 * formats.unpack_bits(np.asarray(rows, dtype=np.uint8)[..., nb:], 1, QJL_DIM).astype(np.float64) - 1.0
    sq = np.asarray(proj, dtype=np.float32).astype(np.float64) @ np.asarray(q_rot, dtype=np.float64)
    rnorm = np.asarray(aux, dtype=np.float64)[..., 1]
    return rnorm * math.sqrt(math.pi / 2.0) / QJL_DIM * (z @ sq)


def requantize(rows16: np.ndarray, fmt: str, bits: int = 0, bounds32: Optional[np.ndarray] = None,
               centroids32: Optional[np.ndarray] = None, proj: Optional[np.ndarray] = None):
    """Re-encode rows stored as fp16 (the rotated vector x~ in fp16, as an fp16 tier or a
    recent-token window holds it) into another format: the encode of the stored x~, with
    no second rotation (FoveatedKV page, "Making it fast": the unquantised decode buffer;
    AdapTQ page, "Hybrid Execution": tokens move to the quantised path once past the
    threshold).  Same returns as `encode`."""
    d = np.shape(rows16)[-1] // 2
    return encode_rotated(decode_rotated(rows16, None, FP16, d), fmt, bits, bounds32, centroids32, proj)


def decode(rows, aux, fmt, s, d, bits=0, centroids32=None, outliers=None) -> np.ndarray:
    """Stored rows -> dequantised vector in the original domain (rotation undone).  For
    codebook_outlier rows: the inlier part plus q_j * s at outlier channel j (the page's
    attend step adds <q[outliers], q_j> * s to the inlier score: the same inner product)."""
    x = unrotate(decode_rotated(rows, aux, fmt, d, bits, centroids32), s)
    if fmt == CODEBOOK_OUTLIER:
        _, scale16, q = unpack_outlier_aux(aux)
        x[..., np.asarray(outliers, dtype=np.int64)] += q.astype(np.float64) * scale16.astype(np.float64)[..., None]
    return x


@dataclasses.dataclass
class Side:
    """One of K or V in a tier: format, code bits, codebook tables, signs, pool arrays."""

    fmt: str
    bits: int
    centroids32: Optional[np.ndarray]
    bounds32: Optional[np.ndarray]
    signs: np.ndarray  # int8 [Hkv, d]
    rows: np.ndarray  # uint8 [num_pages, Hkv, page_size, row_bytes]
    aux: Optional[np.ndarray]  # fp16 [num_pages, Hkv, page_size(, d/32 | 2)]
    proj: Optional[np.ndarray] = None  # float32 [m, d], codebook_qjl keys only
    outliers: Optional[np.ndarray] = None  # int32 [Hkv, K] outlier channels, codebook_outlier keys only


def new_side(fmt, bits, centroids32, bounds32, signs, num_pages, num_kv_heads, page_size, d, proj=None,
             outliers=None) -> Side:
    rb = formats.row_bytes(fmt, bits, d)
    rows = np.zeros((num_pages, num_kv_heads, page_size, rb), dtype=np.uint8)
    aux = None
    if fmt == CODEBOOK:
        aux = np.zeros((num_pages, num_kv_heads, page_size), dtype=np.float16)
    elif fmt == CODEBOOK_QJL:
        aux = np.zeros((num_pages, num_kv_heads, page_size, 2), dtype=np.float16)
    elif fmt == CODEBOOK_OUTLIER:
        aux = np.zeros((num_pages, num_kv_heads, page_size, 4 + OUTLIER_CHANNELS), dtype=np.uint8)
    elif fmt == INT4_G32:
        aux = np.zeros((num_pages, num_kv_heads, page_size, d // formats.GROUP), dtype=np.float16)
    return Side(fmt, bits, centroids32, bounds32, signs, rows, aux, proj, outliers)


def write(side: Side, slots: np.ndarray, x16: np.ndarray, page_size: int) -> None:
    """Encode x16 [T, Hkv, d] and store token i at pool slot slots[i] (slot = page *
    page_size + offset); a negative slot skips the token."""
    slots = np.asarray(slots, dtype=np.int64)
    keep = slots >= 0
    page, off = slots[keep] // page_size, slots[keep] % page_size
    for h in range(x16.shape[1]):
        rows, aux = encode(x16[keep, h, :], side.signs[h], side.fmt, side.bits, side.bounds32, side.centroids32,
                           side.proj, None if side.outliers is None else side.outliers[h])
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
    return decode(rows, aux, side.fmt, side.signs[h], d, side.bits, side.centroids32,
                  None if side.outliers is None else side.outliers[h])
