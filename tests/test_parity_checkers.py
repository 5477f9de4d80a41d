"""The GPU parity checkers accept rows the oracle itself wrote and reject rows with a
planted mistake (the mistakes are planted on the CPU, in oracle output)."""
import numpy as np
import pytest

from oracle import cache as oc
from oracle import formats as of
from tests import gpu_util as gu


@pytest.fixture(scope="module")
def data():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((40, 128)) * rng.uniform(0.01, 50, (40, 1))).astype(np.float16)
    s = np.where(rng.integers(0, 2, 128) == 0, 1, -1)
    return x, s


@pytest.mark.parametrize("fmt", ["fp16", "fp8_e4m3"])
def test_float_checker(data, fmt):
    x, s = data
    rows, _ = oc.encode(x, s, fmt)
    assert gu.check_float_rows(x, s, fmt, rows)[0] == 0
    bad = rows.copy()
    step = 2 if fmt == "fp16" else 1
    bad[3, 10 * step] ^= 0x04  # a wrong mantissa bit
    with pytest.raises(AssertionError):
        gu.check_float_rows(x, s, fmt, bad)
    rows_nosign, _ = oc.encode(x, np.ones_like(s), fmt)  # rotation without the signs
    with pytest.raises(AssertionError):
        gu.check_float_rows(x, s, fmt, rows_nosign)


def test_int4_checker(data):
    x, s = data
    rows, sc = oc.encode(x, s, "int4_g32")
    assert gu.check_int4_rows(x, s, rows, sc)[0] == 0
    nib = of.unpack_bits(rows, 4, 128)
    nib[5, 40] = np.clip(nib[5, 40] + 1, 1, 15) if nib[5, 40] < 15 else 14
    with pytest.raises(AssertionError):
        gu.check_int4_rows(x, s, of.pack_bits(nib, 4), sc)
    sc2 = sc.copy()
    sc2[2, 1] = np.float16(float(sc2[2, 1]) * 1.01)
    with pytest.raises(AssertionError):
        gu.check_int4_rows(x, s, rows, sc2)


def test_codebook_checker(data):
    x, s = data
    c32, b32 = gu.tables("lloyd_max", 4)
    rows, norm = oc.encode(x, s, "codebook", 4, b32)
    assert gu.check_codebook_codes(x, s, 4, rows, norm)[0] == 0
    idx = of.unpack_bits(rows, 4, 128)
    idx[7, 99] = (idx[7, 99] + 1) % 16
    with pytest.raises(AssertionError):
        gu.check_codebook_codes(x, s, 4, of.pack_bits(idx, 4), norm)
    norm2 = norm.copy()
    norm2[1] = np.float16(float(norm2[1]) * 1.002)
    with pytest.raises(AssertionError):
        gu.check_codebook_codes(x, s, 4, rows, norm2)
