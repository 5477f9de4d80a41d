"""Decode attention over the compressed cache (oracle; test infrastructure only).

Sources:
  * XQuant page ("XQuant KV Cache Rematerialization"), step 4 "Implement On-the-Fly
    K, V Recomputation": scores = Q K^T / sqrt(head_dim), softmax over the keys,
    context = weights V.  That plain definition is what is computed here.
  * FoveatedKV page, section "The VR headset thing": every token of every tier
    contributes to one softmax, so its denominator stays correct.

Steps, in this order, all in float64:
  1. read every stored row of the sequence's kv head from each tier and dequantise
     it (codebook: fp16 norm * C[idx] / sqrt(d); fp16; fp8 E4M3; (nibble-8) * scale);
  2. undo the rotation, x = s * H x~ / sqrt(d), to get keys and values in the
     original domain;
  3. for every query head of the group (query head h reads kv head h // (Hq/Hkv)),
     plain softmax(q K^T / sqrt(d)) V over all tokens of all tiers.

Keys stored with a residual sketch (codebook_qjl, VeloxQuant-MLX page "Stage 3"): the
score of such a key is the page's corrected inner product, <q, k^> plus the sketch's
estimate of <q, r> (cache.qjl_correction, taken with the rotated query q~ = R q).

Readings taken: decode attends to the whole cache (no causal or window mask: the
query is the newest token); the output is float32; a sequence with no cached
token gives a zero output.  Score gating and spike flags (FoveatedKV "Making it
fast"): see the last section of this file.  The oracle does not use the rotated-domain scores, a
lookup table, split-K or an online softmax; that those give the same result is
what the GPU tests check.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence

import numpy as np

from . import cache
from .rotation import rotate


@dataclasses.dataclass
class TierState:
    """One precision tier: K and V sides, block tables and per-sequence lengths."""

    k: cache.Side
    v: cache.Side
    block_table: np.ndarray  # int32 [B, max_pages]
    lens: np.ndarray  # [B]
    page_size: int


def dequantised_kv(tiers: Sequence[TierState], b: int, g: int):
    """Keys and values (float64 [L_total, d], original domain) of sequence b, kv head g,
    concatenated over the tiers."""
    ks, vs = [], []
    for t in tiers:
        n = int(t.lens[b])
        if n == 0:
            continue
        ks.append(cache.read(t.k, t.block_table[b], n, g, t.page_size))
        vs.append(cache.read(t.v, t.block_table[b], n, g, t.page_size))
    if not ks:
        return None, None
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)


def sketch_terms(tiers: Sequence[TierState], b: int, g: int, q: np.ndarray) -> np.ndarray:
    """Per token of sequence b, kv head g (tier order, as dequantised_kv): the residual
    sketch's estimate of <q, r> for keys stored with one, else 0."""
    out = []
    for t in tiers:
        n = int(t.lens[b])
        if n == 0:
            continue
        if t.k.fmt != cache.CODEBOOK_QJL:
            out.append(np.zeros(n))
            continue
        rows, aux = cache.gather(t.k, t.block_table[b], n, g, t.page_size)
        q_rot = rotate(np.asarray(q, dtype=np.float64), t.k.signs[g])
        d = q.shape[-1]
        out.append(cache.qjl_correction(rows, aux, q_rot, t.k.proj, d, t.k.bits))
    return np.concatenate(out) if out else np.zeros(0)


def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray, extra=None) -> np.ndarray:
    """softmax(q K^T / sqrt(d)) V for one query vector q [d] (float64); `extra` [L] adds
    to each q.k before the 1/sqrt(d) scaling (the residual sketch's term)."""
    d = q.shape[-1]
    dots = keys @ np.asarray(q, dtype=np.float64)
    if extra is not None:
        dots = dots + extra
    scores = dots / math.sqrt(d)
    w = np.exp(scores - np.max(scores))  # the shift cancels in the normalisation
    w = w / np.sum(w)
    return w @ values


def decode_attention(q16: np.ndarray, tiers: Sequence[TierState],
                     heads: Sequence[tuple] | None = None) -> np.ndarray:
    """Decode attention for queries q16 [B, Hq, d] (fp16).  Returns float32 [B, Hq, d].
    heads: optional list of (b, h_q) to compute; the other outputs stay zero."""
    bsz, hq, d = q16.shape
    hkv = tiers[0].k.signs.shape[0]
    grp = hq // hkv
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    want = set(heads) if heads is not None else None
    for b in range(bsz):
        for g in range(hkv):
            todo = [h for h in range(g * grp, (g + 1) * grp) if want is None or (b, h) in want]
            if not todo:
                continue
            keys, values = dequantised_kv(tiers, b, g)
            if keys is None:
                continue
            sketched = any(t.k.fmt == cache.CODEBOOK_QJL for t in tiers)
            for h in todo:
                q = q16[b, h].astype(np.float64)
                out[b, h] = attend(q, keys, values, sketch_terms(tiers, b, g, q) if sketched else None)
    return out.astype(np.float32)


# ----------------------------------------------------------------------------- FoveatedKV
# Two kernel features of the FoveatedKV page, section "Making it fast": score-gated value
# loading (a token whose softmax weight is below exp(-16) of the largest contributes
# essentially nothing, so its value need not be dequantised) and spike detection (a
# far-tier token that scores above near-tier tokens), which the page reads off the softmax
# bookkeeping.  Tier 0 is the near tier; tiers 1.. are far.

SCORE_GATE_NATS = 16.0


def tier_scores(q: np.ndarray, tiers: Sequence[TierState], b: int, g: int) -> List[np.ndarray]:
    """Per tier, the scores (q.k + sketch term) / sqrt(d) of sequence b's tokens at kv head g
    (float64, natural-log units; empty arrays for empty tiers)."""
    d = q.shape[-1]
    out = []
    for i, t in enumerate(tiers):
        n = int(t.lens[b])
        if n == 0:
            out.append(np.zeros(0))
            continue
        keys = cache.read(t.k, t.block_table[b], n, g, t.page_size)
        dots = keys @ np.asarray(q, dtype=np.float64)
        if t.k.fmt == cache.CODEBOOK_QJL:
            rows, aux = cache.gather(t.k, t.block_table[b], n, g, t.page_size)
            q_rot = rotate(np.asarray(q, dtype=np.float64), t.k.signs[g])
            dots = dots + cache.qjl_correction(rows, aux, q_rot, t.k.proj, d, t.k.bits)
        out.append(dots / math.sqrt(d))
    return out


def spike_flags(q16: np.ndarray, tiers: Sequence[TierState]) -> np.ndarray:
    """int32 [B, Hq]: 1 where the highest score among the tokens of tiers 1.. exceeds the
    lowest score among the tokens of tier 0 (a far token outranks a near one), else 0; 0
    when tier 0 or the later tiers hold no token of the sequence.  Also returns the margin
    max_far - min_near (float64 [B, Hq], nan where undefined), which tells how close a
    decision was."""
    bsz, hq, _ = q16.shape
    hkv = tiers[0].k.signs.shape[0]
    grp = hq // hkv
    flags = np.zeros((bsz, hq), dtype=np.int32)
    margin = np.full((bsz, hq), np.nan)
    for b in range(bsz):
        for h in range(hq):
            s = tier_scores(q16[b, h].astype(np.float64), tiers, b, h // grp)
            near = s[0]
            far = np.concatenate(s[1:]) if len(s) > 1 else np.zeros(0)
            if near.size == 0 or far.size == 0:
                continue
            margin[b, h] = far.max() - near.min()
            flags[b, h] = int(far.max() > near.min())
    return flags, margin


def gated_attention(q16: np.ndarray, tiers: Sequence[TierState], gate_nats: float = SCORE_GATE_NATS):
    """Score-gated decode attention, with the gate taken against the largest score of the
    whole sequence: a token scoring more than gate_nats below it adds nothing to the value
    sum but still counts in the softmax denominator.  Returns (gated, exact, bound), each
    float64 [B, Hq, d]: bound[b, h, i] = sum over the gated tokens of w_t |v_t[i]| with the
    exact softmax weights w_t.  Any implementation that drops the value of a subset of
    the gated tokens -- for instance gating against a running maximum, which never
    exceeds the final one -- lies within `bound` of both `exact` and `gated`."""
    bsz, hq, d = q16.shape
    hkv = tiers[0].k.signs.shape[0]
    grp = hq // hkv
    gated = np.zeros((bsz, hq, d))
    exact = np.zeros((bsz, hq, d))
    bound = np.zeros((bsz, hq, d))
    for b in range(bsz):
        for g in range(hkv):
            keys, values = dequantised_kv(tiers, b, g)
            if keys is None:
                continue
            for h in range(g * grp, (g + 1) * grp):
                s = np.concatenate(tier_scores(q16[b, h].astype(np.float64), tiers, b, g))
                w = np.exp(s - s.max())
                w = w / w.sum()
                drop = s < s.max() - gate_nats
                exact[b, h] = w @ values
                gated[b, h] = (w * ~drop) @ values
                bound[b, h] = (w * drop) @ np.abs(values)
    return gated, exact, bound
