"""Pins of the outlier two-stream cache in the oracle (VeloxQuant-MLX page, "Outlier
Two-Stream Cache").

What fixes it from outside the oracle: planted channel variances whose ranking is known by
construction (including a tie), hand-rounded int8 values, numpy's own variance for a
random case, the dequantised key's outlier channels against the int8 grid, and linearity
of the score: q . k^ = (R q) . x^~_inlier + sum_j q[c_j] q_j s, computed term by term."""
import math

import numpy as np

from oracle import cache as oc
from oracle import codebook as ocb
from oracle import formats as ofmt
from oracle.rotation import rotate, unrotate


def tables(bits):
    c, _, _ = ocb.lloyd_max(bits)
    return ocb.float32_tables(c)


def test_calibration_planted_variances():
    rng = np.random.default_rng(0)
    n, hkv, d = 512, 2, 128
    x = rng.standard_normal((n, hkv, d))
    want = [[90, 3, 77, 12, 100, 64, 5, 31], [7, 8, 127, 0, 55, 56, 90, 2]]
    for h in range(hkv):
        for r, c in enumerate(want[h]):
            x[:, h, c] *= 40.0 - 4 * r  # decreasing standard deviations 40, 36, ..., 12
    got = oc.outlier_channels(x.astype(np.float16))
    assert got.dtype == np.int32 and got.tolist() == want


def test_calibration_ties_go_to_the_lower_channel():
    x = np.zeros((4, 1, 128), np.float16)
    x[:, 0, [9, 4, 100]] = np.array([[1], [-1], [1], [-1]], np.float16)  # equal variance 1
    got = oc.outlier_channels(x)[0]
    assert got[:3].tolist() == [4, 9, 100]
    assert got[3:].tolist() == [0, 1, 2, 3, 5]  # then zero-variance channels by index


def test_calibration_matches_numpy_var():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((300, 3, 256)) * rng.uniform(0.1, 5, 256)).astype(np.float16)
    got = oc.outlier_channels(x)
    var = x.astype(np.float64).var(axis=0)
    for h in range(3):
        assert set(got[h]) == set(np.argsort(-var[h])[:8])


def test_int8_hand_values():
    x = np.array([[127.0, -63.5, 0.5, 1.5, -127.0, 2.25, 0.0, -0.49]])
    q, s = ofmt.outlier_int8_encode(x)
    assert s[0] == np.float16(1.0)
    assert q[0].tolist() == [127, -64, 0, 2, -127, 2, 0, 0]  # rint: ties to even
    q, s = ofmt.outlier_int8_encode(np.zeros((1, 8)))
    assert s[0] == 0 and not q.any()


def test_key_round_trip_and_score_linearity():
    bits = 4
    c32, b32 = tables(bits)
    rng = np.random.default_rng(2)
    d = 128
    x = rng.standard_normal((64, d))
    idx = np.array([3, 17, 40, 41, 80, 99, 120, 127])
    x[:, idx] *= 25
    x16 = x.astype(np.float16)
    s = np.where(rng.random(d) < 0.5, -1, 1).astype(np.int8)
    rows, aux = oc.encode(x16, s, "codebook_outlier", bits, b32, c32, outliers=idx)
    assert rows.shape == (64, ofmt.row_bytes("codebook_outlier", bits, d))
    assert aux.shape == (64, ofmt.aux_bytes("codebook_outlier", d))
    k_hat = oc.decode(rows, aux, "codebook_outlier", s, d, bits, c32, outliers=idx)
    norm16, scale16, q = oc.unpack_outlier_aux(aux)
    # the outlier stream: the int8 grid of the true values (error at most s/2)
    sv = scale16.astype(np.float64)[:, None]
    assert np.all(np.abs(q * sv - x16[:, idx].astype(np.float64)) <= sv / 2 + 1e-12)
    assert np.all(np.abs(q.astype(np.int64)).max(axis=1) == 127)
    # the inlier part: the plain codebook encode of the vector with those channels zeroed
    x_in = x16.copy()
    x_in[:, idx] = 0
    codes_in, n_in = oc.encode(x_in, s, "codebook", bits, b32)
    assert np.array_equal(codes_in, rows) and np.array_equal(n_in, norm16)
    # scores: term by term
    qv = rng.standard_normal(d)
    inl = oc.decode_rotated(rows, aux, "codebook_outlier", d, bits, c32)
    want = inl @ rotate(qv, s) + (q.astype(np.float64) * sv) @ qv[idx]
    np.testing.assert_allclose(k_hat @ qv, want, rtol=1e-12, atol=1e-9)
    # on the outlier channels the key is the inlier decode's (small) leftover plus q s
    assert np.allclose(unrotate(inl, s)[:, idx] + q * sv, k_hat[:, idx])
    assert np.all(np.abs(unrotate(inl, s)[:, idx]) < 0.5 * np.abs(x16[:, idx]).max())
