"""Rademacher sign vectors of the rotation (oracle; test infrastructure only).

Sources:
  * VeloxQuant-MLX page ("I Ported a Google Research Paper to Apple Silicon"),
    section "Stage 1: Random Rotation": the preconditioner multiplies every
    coordinate by an entry of a random Rademacher vector (+1 or -1) before the
    Walsh-Hadamard transform.
  * AdapTQ page ("Shrinking the LLM KV Cache by 8x on CPU"), section "The Math
    Fix: Hadamard Accelerated Rotation (HAR)": a random sign flip comes before
    the transform.

The pages do not say where the signs come from.  Reading taken: independent
signs per (layer, key or value side, kv head, coordinate), drawn from the
SplitMix64 generator (Steele, Lea and Flood, "Fast Splittable Pseudorandom
Number Generators", OOPSLA 2014; the 64-bit constants of Vigna's public
reference version): for the coordinate j of kv head h, side `kind` (0 keys,
1 values) and layer `layer`, the generator is seeded with

    state = seed XOR (layer * 2^40 + kind * 2^32 + h * 2^16 + j)

and its first output decides the sign: +1 when the output's lowest bit is 0,
-1 when it is 1.  Plain Python integers, modulo 2^64.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15  # the generator's state increment


def splitmix64_outputs(state: int, n: int) -> list:
    """The first n outputs of SplitMix64 started at `state`: each step adds the increment
    to the state and returns the state passed through the generator's mixing function
    (xor-shift 30, multiply, xor-shift 27, multiply, xor-shift 31)."""
    out = []
    s = state & MASK64
    for _ in range(n):
        s = (s + GOLDEN_GAMMA) & MASK64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        out.append(z ^ (z >> 31))
    return out


def sign_key(layer: int, kind: int, h: int, j: int) -> int:
    """The 64-bit key of one sign: layer in bits 40.., side in bits 32..39, kv head in bits
    16..31, coordinate in bits 0..15."""
    return (layer << 40) + (kind << 32) + (h << 16) + j


def make_signs(seed: int, layer: int, num_kv_heads: int, head_dim: int):
    """int8 [num_kv_heads, head_dim] +1/-1 sign vectors for keys and for values."""
    out = []
    for kind in (0, 1):
        s = np.empty((num_kv_heads, head_dim), dtype=np.int8)
        for h in range(num_kv_heads):
            for j in range(head_dim):
                first = splitmix64_outputs((seed ^ sign_key(layer, kind, h, j)) & MASK64, 1)[0]
                s[h, j] = 1 if (first & 1) == 0 else -1
        out.append(s)
    return out[0], out[1]
