"""Element formats and bit packing (oracle; test infrastructure only).

Sources:
  * VeloxQuant-MLX page, section "The Bit-Packing Problem": indices are packed
    into one little-endian bit stream; in the 3-bit example byte 0 holds index 0
    in bits 0-2, index 1 in bits 3-5 and the two low bits of index 2 in bits 6-7,
    and byte 1 holds the high bit of index 2 in bit 0 and index 3 in bits 1-3; the
    2-bit unpack shifts each byte by 0, 2, 4, 6.
  * VeloxQuant-MLX page, section "Memory Layout: What Actually Gets Stored": the
    per-vector norm is kept as fp16.
  * FoveatedKV page, section "The VR headset thing": the far tier holds fp8
    E4M3 keys and INT4 values; keys keep more precision than values.

Readings taken (the pages leave them open):
  * every row (one token's vector) starts on a byte boundary; bit k of the row's
    stream is bit (k mod 8) of byte floor(k / 8); element j occupies bits
    j*b .. j*b+b-1, least significant bit first;
  * fp8 is the OCP E4M3 format: bias 7, no infinities, S.1111.111 is NaN, largest
    finite value 448; encoding rounds to nearest, ties to the even code, and
    saturates finite values beyond 448 to +-448 (no per-vector scale);
  * INT4 values are symmetric: per group of 32 consecutive coordinates of one
    vector, scale s = fp16(max|x| / 7); level q = clamp(rint(x / s), -7, 7) with
    ties to even (s == 0 gives q = 0); the stored nibble is q + 8, packed with the
    same little-endian stream rule (even index in the low nibble).
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------- fp16 / fp32


def to_f32(x) -> np.ndarray:
    """Round float64 values to float32 (round to nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def to_f16(x) -> np.ndarray:
    """Round values to float32, then to float16 (each round to nearest even), the two
    roundings a kernel that holds float32 values and stores fp16 performs."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)


# ----------------------------------------------------------------------------- fp8 E4M3


def e4m3_decode(codes) -> np.ndarray:
    """Value (float64) of each fp8 E4M3 code 0..255 from the bit fields."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, subnormal, normal)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(0x7F, dtype=np.int64)  # 0x00..0x7E: all finite non-negative codes
_POS_VALUES = e4m3_decode(_POS_CODES)  # increasing


def e4m3_encode(x) -> np.ndarray:
    """fp8 E4M3 code (uint8) of each value: nearest finite value, ties to the even
    code, magnitudes beyond 448 saturate to 448.  The sign bit follows the sign of x
    (negative values that round to zero give 0x80).  NaN gives 0x7F."""
    v = np.asarray(x, dtype=np.float64)
    mag = np.abs(v)
    # index of the largest representable value <= mag
    lo = np.clip(np.searchsorted(_POS_VALUES, mag, side="right") - 1, 0, len(_POS_VALUES) - 1)
    hi = np.clip(lo + 1, 0, len(_POS_VALUES) - 1)
    dlo = mag - _POS_VALUES[lo]
    dhi = _POS_VALUES[hi] - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_POS_CODES[hi] % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    code = np.where(mag >= _POS_VALUES[-1], 0x7E, code)  # saturate
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------- INT4, 32-groups

GROUP = 32


def int4_g32_encode(x32: np.ndarray):
    """x32: float32 [..., d] (d a multiple of 32).  Returns (nibbles uint8 [..., d] in
    1..15, scales float16 [..., d/32])."""
    x = np.asarray(x32, dtype=np.float32)
    g = x.reshape(*x.shape[:-1], x.shape[-1] // GROUP, GROUP).astype(np.float64)
    amax = np.max(np.abs(g), axis=-1)
    scale16 = to_f16(to_f32(amax / 7.0))  # the kernel divides in fp32, then rounds to fp16
    s = scale16.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = to_f32(np.where(s > 0, g / np.where(s > 0, s, 1.0), 0.0))
    q = np.clip(np.rint(t.astype(np.float64)), -7, 7)
    q = np.where(s > 0, q, 0.0)
    nib = (q + 8).astype(np.uint8).reshape(x.shape)
    return nib, scale16


def int4_g32_decode(nibbles: np.ndarray, scales16: np.ndarray) -> np.ndarray:
    """(nibble - 8) * scale, float64 [..., d]."""
    n = np.asarray(nibbles, dtype=np.float64)
    d = n.shape[-1]
    q = (n - 8.0).reshape(*n.shape[:-1], d // GROUP, GROUP)
    return (q * np.asarray(scales16, dtype=np.float64)[..., None]).reshape(n.shape)


def symmetric_round(x: float, scale: float, qmax: int) -> int:
    """Plain symmetric rounding m = round(x / scale * qmax), ties to even.  The INT4
    encoder above is this with qmax = 7 and scale = the group's max |x|; the CacheQuant
    page's BFP8 worked example uses it with qmax = 127."""
    return int(np.rint(x / scale * qmax))


# ----------------------------------------------------------------------------- bit packing


def pack_bits(idx: np.ndarray, bits: int) -> np.ndarray:
    """Pack integers idx [..., n] (each < 2^bits) into a little-endian bit stream per row.
    Returns uint8 [..., ceil(n*bits/8)]."""
    idx = np.asarray(idx, dtype=np.int64)
    n = idx.shape[-1]
    bitplanes = (idx[..., None] >> np.arange(bits)) & 1  # [..., n, bits], LSB first
    stream = bitplanes.reshape(*idx.shape[:-1], n * bits).astype(np.uint8)
    return np.packbits(stream, axis=-1, bitorder="little")


def unpack_bits(rows: np.ndarray, bits: int, n: int) -> np.ndarray:
    """Inverse of pack_bits: uint8 [..., nbytes] -> int64 [..., n]."""
    stream = np.unpackbits(np.asarray(rows, dtype=np.uint8), axis=-1, bitorder="little")
    stream = stream[..., : n * bits].reshape(*rows.shape[:-1], n, bits).astype(np.int64)
    return np.sum(stream << np.arange(bits), axis=-1)


QJL_DIM = 128  # sign-sketch dimensions m of the residual correction


# ----------------------------------------------------------------------------- outlier stream

OUTLIER_CHANNELS = 8  # K of the outlier two-stream cache (VeloxQuant-MLX page: "at K=8")


def outlier_int8_encode(x: np.ndarray):
    """int8 with a per-token scale (VeloxQuant-MLX page, "Outlier Two-Stream Cache"): for
    the K outlier values x [..., K] of a token, s = fp16(max|x| / 127) (divided in float32,
    as a kernel does), q = clamp(rint(x / s), -127, 127) with the quotient rounded to
    float32 first; s = 0 gives q = 0.  Returns (q int8 [..., K], s float16 [...])."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.max(np.abs(x), axis=-1)
    s16 = to_f16(to_f32(amax / 127.0))
    sv = s16.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = to_f32(np.where(sv > 0, x / np.where(sv > 0, sv, 1.0), 0.0)).astype(np.float64)
    q = np.where(sv > 0, np.clip(np.rint(t), -127, 127), 0.0)
    return q.astype(np.int8), s16


def row_bytes(fmt: str, bits: int, d: int) -> int:
    """Bytes of one packed row (one token's vector) in the given format."""
    if fmt in ("codebook", "codebook_outlier"):  # outlier format: the inlier codes
        return (d * bits + 7) // 8
    if fmt == "codebook_qjl":  # codes, then the m sign bits of the residual sketch
        return (d * bits + 7) // 8 + QJL_DIM // 8
    if fmt == "fp16":
        return 2 * d
    if fmt == "fp8_e4m3":
        return d
    if fmt == "int4_g32":
        return d // 2
    raise ValueError(fmt)


def aux_bytes(fmt: str, d: int) -> int:
    """Bytes of per-row side data: fp16 norm (codebook), fp16 norm + fp16 residual norm
    (codebook with residual sketch), fp16 scale per 32-group (INT4)."""
    if fmt == "codebook":
        return 2
    if fmt == "codebook_qjl":  # fp16 norm, fp16 residual norm
        return 4
    if fmt == "codebook_outlier":  # fp16 norm, fp16 outlier scale, K int8 outlier values
        return 4 + OUTLIER_CHANNELS
    if fmt == "int4_g32":
        return 2 * (d // GROUP)
    return 0
