"""Pins for oracle/attention.py: plain decode attention over the dequantised cache."""
import math

import numpy as np
import pytest
import torch

from oracle import attention, cache, codebook


def test_attend_matches_torch_sdpa():
    rng = np.random.default_rng(0)
    for L, d in ((1, 128), (7, 128), (300, 256)):
        q = rng.standard_normal(d) * 2
        k = rng.standard_normal((L, d)) * 3
        v = rng.standard_normal((L, d))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, None, None], torch.from_numpy(k)[None, None],
            torch.from_numpy(v)[None, None])[0, 0, 0].numpy()
        np.testing.assert_allclose(attention.attend(q, k, v), ref, rtol=1e-12, atol=1e-12)


def test_attend_special_cases():
    rng = np.random.default_rng(1)
    k = rng.standard_normal((10, 128))
    v = rng.standard_normal((10, 128))
    np.testing.assert_allclose(attention.attend(np.zeros(128), k, v), v.mean(axis=0), atol=1e-14)
    np.testing.assert_allclose(attention.attend(rng.standard_normal(128), k[:1], v[:1]), v[0], atol=1e-14)
    q = 1000.0 * k[4] / np.linalg.norm(k[4])
    np.testing.assert_allclose(attention.attend(q, k, v), v[4], atol=1e-10)


def _fp16_tiers(x_k, x_v, signs_k, signs_v, split):
    """Build tiers holding the tokens of every (b, g) split at `split` into two fp16 tiers."""
    bsz, L, hkv, d = x_k.shape
    ps = 16
    tiers = []
    for lo, hi in ((0, split), (split, L)):
        n = hi - lo
        per = (n + ps - 1) // ps
        num_pages = max(1, per * bsz)
        k = cache.new_side("fp16", 0, None, None, signs_k, num_pages, hkv, ps, d)
        v = cache.new_side("fp16", 0, None, None, signs_v, num_pages, hkv, ps, d)
        bt = np.arange(bsz * max(per, 1), dtype=np.int32).reshape(bsz, max(per, 1))
        for b in range(bsz):
            t = np.arange(n)
            slots = bt[b, t // ps] * ps + t % ps
            cache.write(k, slots, x_k[b, lo:hi], ps)
            cache.write(v, slots, x_v[b, lo:hi], ps)
        tiers.append(attention.TierState(k, v, bt, np.full(bsz, n), ps))
    return tiers


def test_fp16_cache_equals_unquantised_attention():
    """With every token stored as fp16 (of the rotated vector), decode attention equals plain
    softmax(q K^T / sqrt(d)) V over the original fp16 keys/values up to fp16 rounding; and
    how tokens are split between tiers does not matter (every token contributes)."""
    rng = np.random.default_rng(3)
    bsz, L, hq, hkv, d = 2, 40, 4, 2, 128
    xk = rng.standard_normal((bsz, L, hkv, d)).astype(np.float16)
    xv = rng.standard_normal((bsz, L, hkv, d)).astype(np.float16)
    q = rng.standard_normal((bsz, hq, d)).astype(np.float16)
    sk = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    sv = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    outs = [attention.decode_attention(q, _fp16_tiers(xk, xv, sk, sv, split)) for split in (0, 13, 40)]
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=2e-6)
    g = hq // hkv
    for b in range(bsz):
        for h in range(hq):
            k = torch.from_numpy(xk[b, :, h // g].astype(np.float64))
            v = torch.from_numpy(xv[b, :, h // g].astype(np.float64))
            qq = torch.from_numpy(q[b, h].astype(np.float64))
            ref = torch.nn.functional.scaled_dot_product_attention(qq[None, None, None], k[None, None],
                                                                   v[None, None])[0, 0, 0].numpy()
            np.testing.assert_allclose(outs[0][b, h], ref, rtol=0, atol=5e-3)


def test_gqa_head_mapping_and_empty_sequence():
    """Query head h reads kv head h // (Hq / Hkv); a sequence with no tokens gives zeros."""
    bsz, L, hq, hkv, d = 2, 16, 8, 2, 128
    xk = np.zeros((bsz, L, hkv, d), np.float16)
    xv = np.zeros((bsz, L, hkv, d), np.float16)
    xv[:, :, 0, :] = 1.0
    xv[:, :, 1, :] = -2.0
    q = np.random.default_rng(0).standard_normal((bsz, hq, d)).astype(np.float16)
    sk = np.ones((hkv, d), np.int8)
    tiers = _fp16_tiers(xk, xv, sk, sk, 16)
    tiers[0].lens[1] = 0  # sequence 1 empty in both tiers
    tiers[1].lens[1] = 0
    out = attention.decode_attention(q, tiers)
    # the fp16 tier stores the rotated vector (sqrt(d) * e0 here): one fp16 rounding, 2^-11
    np.testing.assert_allclose(out[0, :4], 1.0, rtol=2.0 ** -11)
    np.testing.assert_allclose(out[0, 4:], -2.0, rtol=2.0 ** -11)
    assert np.all(out[1] == 0)


def test_brute_force_dequantise_then_attend_tiny():
    """Tiny codebook cache: decode_attention equals a direct loop that dequantises each
    token from its packed bits with the textbook formula and attends."""
    rng = np.random.default_rng(8)
    d, L, ps = 128, 21, 16
    c32, b32 = codebook.tables("lloyd_max", 4)
    s = np.where(rng.integers(0, 2, (1, d)) == 0, 1, -1).astype(np.int8)
    x = rng.standard_normal((L, 1, d)).astype(np.float16)
    kside = cache.new_side("codebook", 4, c32, b32, s, 2, 1, ps, d)
    vside = cache.new_side("codebook", 4, c32, b32, s, 2, 1, ps, d)
    bt = np.array([[1, 0]], dtype=np.int32)
    slots = bt[0, np.arange(L) // ps] * ps + np.arange(L) % ps
    cache.write(kside, slots, x, ps)
    cache.write(vside, slots, x[::-1].copy(), ps)
    q = rng.standard_normal((1, 1, d)).astype(np.float16)
    out = attention.decode_attention(q, [attention.TierState(kside, vside, bt, np.array([L]), ps)])
    # direct: nibble j of byte j//2 (low nibble for even j), value = C[idx] * norm / sqrt(d),
    # then x = s * H x~ / sqrt(d) with H from scipy
    import scipy.linalg
    H = scipy.linalg.hadamard(d).astype(np.float64)

    def deq(side, t):
        page, off = bt[0, t // ps], t % ps
        row = side.rows[page, 0, off]
        idx = [(row[j // 2] >> (4 * (j % 2))) & 0xF for j in range(d)]
        xr = np.array([float(c32[i]) for i in idx]) * float(side.aux[page, 0, off]) / math.sqrt(d)
        return s[0] * (H @ xr) / math.sqrt(d)

    K = np.stack([deq(kside, t) for t in range(L)])
    V = np.stack([deq(vside, t) for t in range(L)])
    sc = K @ q[0, 0].astype(np.float64) / math.sqrt(d)
    w = np.exp(sc - sc.max()); w /= w.sum()
    np.testing.assert_allclose(out[0, 0], w @ V, rtol=0, atol=1e-6)
