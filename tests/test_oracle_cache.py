"""Pins for oracle/cache.py: encode / decode of one vector and the paged pool."""
import functools
import math

import numpy as np
import pytest

from oracle import cache, codebook, formats
from tests.conftest import read_golden


@functools.lru_cache(maxsize=None)
def lm_tables(bits):
    return codebook.tables("lloyd_max", bits)


def test_hand_worked_d2_examples():
    g = read_golden("encode_d2_example.txt")
    c32, b32 = lm_tables(4)
    for case in ("A", "B"):
        x = np.array([float(v) for v in g[f"{case}_x"]], dtype=np.float16)
        s = np.array([int(v) for v in g[f"{case}_s"]])
        rows, norm = cache.encode(x, s, "codebook", 4, b32)
        assert list(rows) == [int(g[f"{case}_byte"][0], 16)]
        assert float(norm) == 1.0
        dec = cache.decode(rows, norm, "codebook", s, 2, 4, c32)
        np.testing.assert_allclose(dec, [float(v) for v in g[f"{case}_decoded"]], atol=5e-5)
    rows, norm = cache.encode(np.zeros(2, np.float16), np.ones(2), "codebook", 4, b32)
    assert list(rows) == [int(g["C_byte"][0], 16)] and float(norm) == 0.0


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_zero_vector_codes(bits):
    c32, b32 = lm_tables(bits)
    rows, norm = cache.encode(np.zeros((1, 128), np.float16), np.ones(128), "codebook", bits, b32)
    idx = formats.unpack_bits(rows, bits, 128)
    assert np.all(idx == 2 ** (bits - 1) - 1) and float(norm[0]) == 0.0
    dec = cache.decode(rows, norm, "codebook", np.ones(128), 128, bits, c32)
    assert np.all(dec == 0)


@pytest.mark.parametrize("bits,mse", [(2, 0.1175), (3, 0.03455), (4, 0.00950)])
def test_distortion_of_gaussian_vectors(bits, mse):
    """On iid N(0,1) vectors the rotated unit-norm coordinates are close to N(0,1)/sqrt(d);
    the per-coordinate distortion of u must then be near the Lloyd-Max MSE, and the
    cosine between a vector and its reconstruction near sqrt(1 - MSE)."""
    d = 128
    rng = np.random.default_rng(bits)
    s = np.where(rng.integers(0, 2, d) == 0, 1, -1)
    x = rng.standard_normal((3000, d)).astype(np.float16)
    c32, b32 = lm_tables(bits)
    rows, norm = cache.encode(x, s, "codebook", bits, b32)
    dec = cache.decode(rows, norm, "codebook", s, d, bits, c32)
    xf = x.astype(np.float64)
    cos = np.sum(xf * dec, axis=1) / (np.linalg.norm(xf, axis=1) * np.linalg.norm(dec, axis=1))
    # per coordinate of u = sqrt(d) x~ / ||x||: error^2 = d * ||x - xhat||^2 / ||x||^2 / d
    err = np.sum((xf - dec) ** 2, axis=1) / np.sum(xf * xf, axis=1)
    assert abs(np.mean(err) / mse - 1) < 0.06
    assert abs(np.mean(cos) - math.sqrt(1 - mse)) < 0.01


def test_fp16_tier_round_trip():
    rng = np.random.default_rng(2)
    s = np.where(rng.integers(0, 2, 128) == 0, 1, -1)
    x = (rng.standard_normal((50, 128)) * 3).astype(np.float16)
    rows, aux = cache.encode(x, s, "fp16", 0, None)
    assert rows.shape == (50, 256) and aux is None
    dec = cache.decode(rows, aux, "fp16", s, 128)
    np.testing.assert_allclose(dec, x.astype(np.float64), rtol=0, atol=3 * 2.0 ** -11 * 3 * 4)


def test_fp8_int4_tier_reconstruction():
    rng = np.random.default_rng(4)
    s = np.where(rng.integers(0, 2, 128) == 0, 1, -1)
    x = rng.standard_normal((500, 128)).astype(np.float16)
    xf = x.astype(np.float64)
    k_rows, _ = cache.encode(x, s, "fp8_e4m3")
    v_rows, v_sc = cache.encode(x, s, "int4_g32")
    assert k_rows.shape == (500, 128) and v_rows.shape == (500, 64) and v_sc.shape == (500, 4)
    k = cache.decode(k_rows, None, "fp8_e4m3", s, 128)
    v = cache.decode(v_rows, v_sc, "int4_g32", s, 128)
    rel_k = np.linalg.norm(k - xf) / np.linalg.norm(xf)
    rel_v = np.linalg.norm(v - xf) / np.linalg.norm(xf)
    assert rel_k < 0.04  # 3 mantissa bits: ~2^-4 / sqrt(3) relative per element
    assert 0.05 < rel_v < 0.2  # 15 levels over +-max of 32 Gaussians
    # FoveatedKV page, "The VR headset thing": keys kept at higher precision than values
    assert rel_k < rel_v


def test_pool_write_then_read_shuffled_pages():
    rng = np.random.default_rng(9)
    d, hkv, ps, n = 128, 2, 16, 53
    signs = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    c32, b32 = lm_tables(3)
    num_pages = 8
    pages = rng.permutation(num_pages)[:4]  # 4 pages hold 53 tokens
    block_row = pages.astype(np.int32)
    t = np.arange(n)
    slots = block_row[t // ps] * ps + t % ps
    x = rng.standard_normal((n, hkv, d)).astype(np.float16)
    side = cache.new_side("codebook", 3, c32, b32, signs, num_pages, hkv, ps, d)
    cache.write(side, slots, x, ps)
    for h in range(hkv):
        got = cache.read(side, block_row, n, h, ps)
        rows, norm = cache.encode(x[:, h], signs[h], "codebook", 3, b32)
        want = cache.decode(rows, norm, "codebook", signs[h], d, 3, c32)
        np.testing.assert_array_equal(got, want)
    # untouched pages stay zero
    unused = sorted(set(range(num_pages)) - set(pages.tolist()))
    assert not side.rows[unused].any()
