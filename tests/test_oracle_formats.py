"""Pins for oracle/formats.py: bit packing, fp8 E4M3, INT4 with 32-group scales.

Checked against the VeloxQuant-MLX page's packing example and unpack code, torch's
float8_e4m3fn conversion (a library routine), the OCP format's fixed points, brute
force, and the CacheQuant page's rounding example."""
import numpy as np
import pytest
import torch

from oracle import formats
from tests.conftest import read_golden


def test_page_3bit_example():
    g = read_golden("pack_3bit_example.txt")
    idx = np.array([int(v) for v in g["indices"]])
    want = [int(v, 16) for v in g["bytes"]]
    assert list(formats.pack_bits(idx, 3)) == want
    assert list(formats.unpack_bits(np.array(want, dtype=np.uint8), 3, 5)) == list(idx)


def test_2bit_matches_page_unpack_shifts():
    """The page's vectorised 2-bit unpack: ((packed[:, :, None] >> [0,2,4,6]) & 3)."""
    rng = np.random.default_rng(0)
    idx = rng.integers(0, 4, size=(7, 128))
    packed = formats.pack_bits(idx, 2)
    shifts = np.array([0, 2, 4, 6], dtype=np.uint8)
    vals = ((packed[:, :, None] >> shifts) & 0x3).reshape(7, -1)[:, :128]
    assert np.array_equal(vals, idx)


def test_4bit_even_index_in_low_nibble():
    idx = np.array([0x3, 0xA, 0xF, 0x1])
    assert list(formats.pack_bits(idx, 4)) == [0xA3, 0x1F]


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 8])
def test_pack_round_trip(bits):
    idx = np.random.default_rng(bits).integers(0, 2 ** bits, size=(9, 256))
    rows = formats.pack_bits(idx, bits)
    assert rows.shape == (9, 256 * bits // 8)
    assert np.array_equal(formats.unpack_bits(rows, bits, 256), idx)


def test_e4m3_fixed_points():
    dec = formats.e4m3_decode(np.arange(256))
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0
    assert dec[0x38] == 1.0
    assert dec[0x08] == 2.0 ** -6  # smallest normal
    assert dec[0x01] == 2.0 ** -9  # smallest subnormal
    assert dec[0x00] == 0.0 and np.signbit(dec[0x80])
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert np.sum(np.isnan(dec)) == 2
    assert np.all(np.diff(dec[:0x7F]) > 0)


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dec = formats.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(dec))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], dec[ok])


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(50000) * 3,
        rng.standard_normal(20000) * 100,
        rng.standard_normal(20000) * 0.01,
    ])
    # every exact midpoint between neighbouring values (ties) and every value itself
    pos = formats.e4m3_decode(np.arange(0x7F))
    mids = (pos[:-1] + pos[1:]) / 2
    vals = np.concatenate([vals, mids, -mids, pos, -pos]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = formats.e4m3_encode(vals)
    assert np.array_equal(got, ref)


def test_e4m3_saturates():
    got = formats.e4m3_encode(np.array([449.0, 464.0, 1e6, -500.0], dtype=np.float32))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0xFE]


def test_int4_g32_brute_force():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((40, 128)) * rng.uniform(0.01, 30, (40, 1))).astype(np.float32)
    x[3, 32:64] = 0.0  # an all-zero group
    nib, sc = formats.int4_g32_encode(x)
    assert nib.shape == x.shape and sc.shape == (40, 4) and sc.dtype == np.float16
    assert nib.min() >= 1 and nib.max() <= 15
    assert sc[3, 1] == 0 and np.all(nib[3, 32:64] == 8)
    levels = np.arange(-7, 8, dtype=np.float64)
    for r in range(40):
        for g in range(4):
            grp = x[r, 32 * g: 32 * g + 32].astype(np.float64)
            s = float(sc[r, g])
            assert s == float(np.float16(np.float32(np.max(np.abs(grp)) / 7)))
            if s == 0:
                continue
            q = nib[r, 32 * g: 32 * g + 32].astype(np.int64) - 8
            err = np.abs(grp[:, None] - levels[None, :] * s)
            best = err.min(axis=1)
            assert np.all(np.abs(grp - q * s) <= best + 1e-12 * np.abs(grp).max())
    dec = formats.int4_g32_decode(nib, sc)
    assert np.all(np.abs(dec - x) <= np.repeat(sc.astype(np.float64), 32, axis=1) * 0.5 + 1e-6)


def test_cachequant_rounding_example():
    g = read_golden("bfp8_rounding_example.txt")
    m = formats.symmetric_round(float(g["x"][0]), float(g["scale"][0]), int(g["qmax"][0]))
    assert m == int(g["m"][0])
    assert round(m * float(g["scale"][0]) / int(g["qmax"][0]), 3) == float(g["xhat"][0])


def test_row_bytes():
    assert formats.row_bytes("codebook", 4, 128) == 64
    assert formats.row_bytes("codebook", 3, 128) == 48
    assert formats.row_bytes("codebook", 2, 128) == 32
    assert formats.row_bytes("codebook", 4, 256) == 128
    assert formats.row_bytes("fp16", 0, 128) == 256
    assert formats.row_bytes("fp8_e4m3", 0, 128) == 128
    assert formats.row_bytes("int4_g32", 0, 128) == 64
    assert formats.aux_bytes("int4_g32", 128) == 8
