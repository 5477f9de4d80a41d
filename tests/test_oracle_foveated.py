"""Pins of the FoveatedKV kernel features in the oracle (FoveatedKV page, "Making it fast"):
spike flags (a far-tier token outscoring a near-tier one) and score-gated value loading
(tokens below exp(-16) of the largest weight add nothing to the value sum).

What fixes them from outside the oracle: hand-built caches whose scores are known by
construction (one-hot keys against a one-hot query), the closed form of a two-token
softmax, the gate at +inf reducing to plain attention, and a token-by-token running-max
implementation written here that must stay inside the oracle's bound."""
import math

import numpy as np

from oracle import attention as oatt
from oracle import cache as oc

D = 128


def one_hot_tiers(near, far, hkv=1):
    """Two fp16 tiers, one sequence; key t of a tier is a[t] * e_0 (so its score against
    q = sqrt(D) e_0 is a[t]), value t is (t + 1) * e_1."""
    signs = np.ones((hkv, D), dtype=np.int8)
    tiers = []
    for a in (near, far):
        n = len(a)
        pages = max(1, (n + 15) // 16)
        ks = oc.new_side("fp16", 0, None, None, signs, pages, hkv, 16, D)
        vs = oc.new_side("fp16", 0, None, None, signs, pages, hkv, 16, D)
        if n:
            k = np.zeros((n, hkv, D), np.float16)
            v = np.zeros((n, hkv, D), np.float16)
            k[:, :, 0] = np.asarray(a, np.float16)[:, None]
            v[:, :, 1] = np.arange(1, n + 1, dtype=np.float16)[:, None]
            oc.write(ks, np.arange(n), k, 16)
            oc.write(vs, np.arange(n), v, 16)
        tiers.append(oatt.TierState(ks, vs, np.arange(pages, dtype=np.int32)[None, :], np.array([n]), 16))
    return tiers


def query(scale=1.0):
    q = np.zeros((1, 1, D), np.float16)
    q[0, 0, 0] = math.sqrt(D) * scale
    return q


def test_spike_flag_by_construction():
    # near scores {3, 1, 2}; far {0.5, 1.5}: 1.5 outranks the near token scoring 1
    flags, margin = oatt.spike_flags(query(), one_hot_tiers([3, 1, 2], [0.5, 1.5]))
    assert flags[0, 0] == 1 and abs(margin[0, 0] - 0.5) < 2e-2
    flags, margin = oatt.spike_flags(query(), one_hot_tiers([3, 1, 2], [0.5, 0.875]))
    assert flags[0, 0] == 0 and abs(margin[0, 0] + 0.125) < 2e-2
    # a far token equal to the lowest near token does not outrank it
    flags, _ = oatt.spike_flags(query(), one_hot_tiers([3, 1, 2], [1.0]))
    assert flags[0, 0] == 0


def test_spike_flag_needs_both_tiers():
    for near, far in (([], [1, 2]), ([1, 2], []), ([], [])):
        flags, margin = oatt.spike_flags(query(), one_hot_tiers(near, far))
        assert flags[0, 0] == 0 and np.isnan(margin[0, 0])


def test_gate_two_token_closed_form():
    # scores 0 and -20 (nats): the second token is gated
    tiers = one_hot_tiers([0.0, -2.5], [])
    q = query(8.0)  # scores 0 and -20 (up to the fp16 rounding of the stored rows)
    gated, exact, bound = oatt.gated_attention(q, tiers)
    keys, values = oatt.dequantised_kv(tiers, 0, 0)  # what the cache holds
    s = keys @ q[0, 0].astype(np.float64) / math.sqrt(D)
    assert abs(s[0]) < 1e-2 and abs(s[1] + 20) < 5e-2
    w2 = 1.0 / (1.0 + math.exp(s[0] - s[1]))
    w1 = 1.0 - w2
    np.testing.assert_allclose(exact[0, 0], w1 * values[0] + w2 * values[1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gated[0, 0], w1 * values[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(bound[0, 0], w2 * np.abs(values[1]), rtol=0, atol=1e-18)


def test_gate_at_infinity_is_plain_attention():
    rng = np.random.default_rng(3)
    tiers = one_hot_tiers(list(rng.normal(0, 2, 40)), list(rng.normal(0, 2, 30)))
    q = query(4.0)
    gated, exact, bound = oatt.gated_attention(q, tiers, gate_nats=math.inf)
    assert np.array_equal(gated, exact) and not bound.any()
    np.testing.assert_allclose(exact[0, 0], oatt.decode_attention(q, tiers)[0, 0], rtol=1e-6, atol=1e-6)


def test_running_max_gate_stays_inside_the_bound():
    """A token-by-token online softmax that drops the value of a token more than 16 nats
    below its running maximum (which is never above the final one)."""
    rng = np.random.default_rng(5)
    a = list(rng.normal(0, 1.5, 200))
    a[150] = 6.0  # a late maximum: early tokens are judged against lower running maxima
    tiers = one_hot_tiers(a[:120], a[120:])
    q = query(6.0)
    gated, exact, bound = oatt.gated_attention(q, tiers)
    keys, values = oatt.dequantised_kv(tiers, 0, 0)
    s = keys @ q[0, 0].astype(np.float64) / math.sqrt(D)
    m, l, acc, dropped = -math.inf, 0.0, np.zeros(D), 0
    for t in range(len(s)):
        if s[t] > m:
            f = math.exp(m - s[t]) if m > -math.inf else 0.0
            l, acc, m = l * f, acc * f, s[t]
        p = math.exp(s[t] - m)
        l += p
        if s[t] < m - oatt.SCORE_GATE_NATS:
            dropped += 1
        else:
            acc = acc + p * values[t]
    online = acc / l
    assert dropped > 0 and bound[0, 0].max() > 0
    assert np.all(np.abs(online - exact[0, 0]) <= bound[0, 0] + 1e-12)
    assert np.all(np.abs(online - gated[0, 0]) <= bound[0, 0] + 1e-12)
