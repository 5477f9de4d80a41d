"""Pins of the oracle's re-encode of stored fp16 rows (a recent-token window moving into a
quantised tier; FoveatedKV page, "Making it fast", and AdapTQ page, "Hybrid Execution").

What fixes it from outside the oracle: fp16 -> fp16 is the identity on the stored bytes;
a one-hot rotated vector has a hand-computable codebook row; fp8 of an fp16 value is
torch's float8_e4m3fn conversion; and re-encoding the fp16 window row of x gives the
codes of encoding x itself except where the fp16 rounding of x~ crosses a boundary."""
import math

import numpy as np
import pytest

from oracle import cache as oc
from oracle import codebook as ocb
from oracle import formats as ofmt


def tables(bits):
    c, _, _ = ocb.lloyd_max(bits)
    return ocb.float32_tables(c)


def fp16_rows(x16, s):
    rows, _ = oc.encode(x16, s, "fp16")
    return rows


def test_fp16_to_fp16_is_identity():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((50, 128)).astype(np.float16)
    s = np.where(rng.random(128) < 0.5, -1, 1).astype(np.int8)
    rows = fp16_rows(x, s)
    again, aux = oc.requantize(rows, "fp16")
    assert aux is None and np.array_equal(again, rows)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("d", [128, 256])
def test_one_hot_rotated_row(bits, d):
    c32, b32 = tables(bits)
    rows16 = np.zeros((1, d), np.float16)
    rows16[0, 5] = 2.0  # x~ = 2 e_5, exact in fp16
    rows, norm = oc.requantize(rows16.view(np.uint8), "codebook", bits, b32)
    assert norm[0] == np.float16(2.0)
    idx = ofmt.unpack_bits(rows, bits, d)[0]
    top = int(np.sum(math.sqrt(d) > b32.astype(np.float64)))  # u_5 = sqrt(d)
    mid = int(np.sum(0.0 > b32.astype(np.float64)))  # u = 0 elsewhere
    assert top == (1 << bits) - 1 and mid == (1 << (bits - 1)) - 1
    assert idx[5] == top and np.all(np.delete(idx, 5) == mid)


def test_fp8_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((40, 128)) * 30).astype(np.float16)
    s = np.where(rng.random(128) < 0.5, -1, 1).astype(np.int8)
    rows16 = fp16_rows(x, s)
    got, _ = oc.requantize(rows16, "fp8_e4m3")
    xr16 = rows16.view(np.float16)
    want = torch.from_numpy(xr16.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


@pytest.mark.parametrize("bits", [2, 4])
def test_codes_match_direct_encode_away_from_boundaries(bits):
    c32, b32 = tables(bits)
    rng = np.random.default_rng(3)
    d = 128
    x = rng.standard_normal((400, d)).astype(np.float16)
    s = np.where(rng.random(d) < 0.5, -1, 1).astype(np.int8)
    direct, n_direct = oc.encode(x, s, "codebook", bits, b32)
    moved, n_moved = oc.requantize(fp16_rows(x, s), "codebook", bits, b32)
    a, b = ofmt.unpack_bits(direct, bits, d), ofmt.unpack_bits(moved, bits, d)
    diff = a != b
    assert diff.mean() < 2e-2 and np.all(np.abs(a - b)[diff] == 1)
    # where they differ, the exact u sits within the fp16 rounding of x~ of a boundary
    from oracle.rotation import rotate
    xr = rotate(x.astype(np.float64), s)
    u = math.sqrt(d) * xr / np.linalg.norm(xr, axis=-1, keepdims=True)
    dist = np.min(np.abs(u[..., None] - b32.astype(np.float64)), axis=-1)
    assert np.all(dist[diff] < 2e-3 * math.sqrt(d))
    assert np.all(np.abs(n_direct.astype(np.float64) - n_moved.astype(np.float64)) <= 2e-3 * n_direct.astype(np.float64))
