"""Pins of the residual sign sketch (codebook_qjl keys; VeloxQuant-MLX page, "Stage 3:
QJL Residual Correction" and "Memory Layout: What Actually Gets Stored").

What fixes it from outside the oracle: the page's byte table; the mathematics of the
estimator (for S with iid N(0,1) rows, E[sign(S_j r) S_j q] = sqrt(2/pi) <q, r> / ||r||,
so the correction is unbiased -- checked against the directly computed <q, r> over many
independent projections); the corrected score recovering the true inner product of the
unquantised vectors on average; and special cases (a zero residual, a sign flip of S)."""
import math

import numpy as np

from oracle import attention as oatt
from oracle import cache as oc
from oracle import codebook as ocb
from oracle import formats as ofmt
from oracle.rotation import rotate
from tests.conftest import read_golden


def tables(bits):
    c, _, _ = ocb.lloyd_max(bits)
    return ocb.float32_tables(c)


def test_key_layout_matches_page():
    g = read_golden("prod_key_layout.txt")
    d, bits, m = int(g["d"][0]), int(g["code_bits"][0]), int(g["sketch_dims"][0])
    assert m == oc.QJL_DIM
    rb, ab = ofmt.row_bytes("codebook_qjl", bits, d), ofmt.aux_bytes("codebook_qjl", d)
    assert rb == int(g["code_bytes"][0]) + int(g["sign_bytes"][0])
    assert rb + ab == int(g["key_bytes"][0])
    c32, b32 = tables(bits)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, d)).astype(np.float16)
    s = np.where(rng.random(d) < 0.5, -1, 1).astype(np.int8)
    proj = rng.standard_normal((m, d)).astype(np.float32)
    rows, aux = oc.encode(x, s, "codebook_qjl", bits, b32, c32, proj)
    assert rows.shape == (3, rb) and aux.shape == (3, 2) and aux.dtype == np.float16


def _rows_from_signs(z, d, bits):
    """A codebook_qjl row whose code part is zero and whose sign bits are z (0/1)."""
    codes = np.zeros((z.shape[0], (d * bits + 7) // 8), dtype=np.uint8)
    return np.concatenate([codes, ofmt.pack_bits(z.astype(np.int64), 1)], axis=-1)


def test_correction_is_unbiased():
    """Mean of the correction over many independent projections -> <q, r> (the page: the
    correction is unbiased).  A wrong constant, a flipped sign convention or a sign taken
    of <S_j, q> instead of using it fails this."""
    d, bits, m = 64, 3, oc.QJL_DIM
    rng = np.random.default_rng(1)
    q = rng.standard_normal(d)
    r = rng.standard_normal(d) * 0.3
    truth = float(q @ r)
    draws = 3000
    est = np.empty(draws)
    for i in range(draws):
        proj = rng.standard_normal((m, d)).astype(np.float32)
        z = (proj.astype(np.float64) @ r >= 0)
        rows = _rows_from_signs(z[None, :], d, bits)
        aux = np.array([[1.0, np.linalg.norm(r)]], dtype=np.float64)
        est[i] = oc.qjl_correction(rows, aux, q, proj, d, bits)[0]
    se = est.std() / math.sqrt(draws)
    assert abs(est.mean() - truth) < 4 * se, (est.mean(), truth, se)
    # and it is not trivially small: the per-draw spread is of the order of |q||r|/sqrt(m)
    assert 0.3 < est.std() / (np.linalg.norm(q) * np.linalg.norm(r) / math.sqrt(m)) < 3


def test_corrected_score_recovers_true_dot_on_average():
    """<q~, x^~> + correction, averaged over projections, estimates <q, x> of the stored
    fp16 vector itself (the codebook error is what the sketch corrects)."""
    d, bits, m = 128, 2, oc.QJL_DIM
    c32, b32 = tables(bits)
    rng = np.random.default_rng(2)
    x16 = rng.standard_normal(d).astype(np.float16)
    q = rng.standard_normal(d)
    s = np.where(rng.random(d) < 0.5, -1, 1).astype(np.int8)
    truth = float(q @ x16.astype(np.float64))
    q_rot = rotate(q, s)
    draws = 800
    est = np.empty(draws)
    for i in range(draws):
        proj = rng.standard_normal((m, d)).astype(np.float32)
        rows, aux = oc.encode(x16[None, :], s, "codebook_qjl", bits, b32, c32, proj)
        xhat = oc.decode_rotated(rows, aux, "codebook_qjl", d, bits, c32)[0]
        est[i] = q_rot @ xhat + oc.qjl_correction(rows, aux, q_rot, proj, d, bits)[0]
    xhat_only = float(q_rot @ xhat)
    se = est.std() / math.sqrt(draws)
    assert abs(est.mean() - truth) < 4 * se + 1e-3 * abs(truth)
    # the codebook part alone is off by much more than the averaged correction's error
    assert abs(xhat_only - truth) > 4 * se


def test_zero_residual_and_sign_symmetry():
    d, bits, m = 128, 4, oc.QJL_DIM
    rng = np.random.default_rng(3)
    proj = rng.standard_normal((m, d)).astype(np.float32)
    q = rng.standard_normal(d)
    z = rng.random(m) < 0.5
    rows = _rows_from_signs(z[None, :], d, bits)
    # zero residual norm: no correction whatever the signs
    assert oc.qjl_correction(rows, np.array([[1.0, 0.0]]), q, proj, d, bits)[0] == 0.0
    # complementing every sign bit negates the correction
    rows_c = _rows_from_signs(~z[None, :], d, bits)
    a = oc.qjl_correction(rows, np.array([[1.0, 2.0]]), q, proj, d, bits)[0]
    b = oc.qjl_correction(rows_c, np.array([[1.0, 2.0]]), q, proj, d, bits)[0]
    assert a == -b and a != 0.0
    # sign(0) = +1: a residual of zero sets every sign bit
    assert np.all(ofmt.unpack_bits(_rows_from_signs(np.ones((1, m), bool), d, bits)[:, d * bits // 8:], 1, m) == 1)


def test_sketch_tier_with_zero_residuals_is_plain_codebook_attention():
    """Attention over a codebook_qjl tier whose residual norms are zero equals attention
    over the same codes stored as a plain codebook tier."""
    d, bits, hkv, ps = 128, 3, 2, 16
    c32, b32 = tables(bits)
    rng = np.random.default_rng(4)
    n = 40
    x = rng.standard_normal((n, hkv, d)).astype(np.float16)
    v = rng.standard_normal((n, hkv, d)).astype(np.float16)
    signs = np.where(rng.random((hkv, d)) < 0.5, -1, 1).astype(np.int8)
    proj = rng.standard_normal((oc.QJL_DIM, d)).astype(np.float32)
    pages = (n + ps - 1) // ps
    slots = np.arange(n)
    kq = oc.new_side("codebook_qjl", bits, c32, b32, signs, pages, hkv, ps, d, proj)
    kp = oc.new_side("codebook", bits, c32, b32, signs, pages, hkv, ps, d)
    vs = oc.new_side("codebook", bits, c32, b32, signs, pages, hkv, ps, d)
    oc.write(kq, slots, x, ps)
    oc.write(kp, slots, x, ps)
    oc.write(vs, slots, v, ps)
    kq.aux[..., 1] = 0.0  # zero residual norms
    nb = d * bits // 8
    assert np.array_equal(kq.rows[..., :nb], kp.rows) and np.array_equal(kq.aux[..., 0], kp.aux)
    bt = np.arange(pages, dtype=np.int32)[None, :]
    lens = np.array([n])
    q = rng.standard_normal((1, hkv, d)).astype(np.float16)
    a = oatt.decode_attention(q, [oatt.TierState(kq, vs, bt, lens, ps)])
    b = oatt.decode_attention(q, [oatt.TierState(kp, vs, bt, lens, ps)])
    np.testing.assert_array_equal(a, b)
    # with the real residual norms the sketch moves the output
    oc.write(kq, slots, x, ps)
    c = oatt.decode_attention(q, [oatt.TierState(kq, vs, bt, lens, ps)])
    assert np.abs(c - b).max() > 0
