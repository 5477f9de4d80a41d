"""Seeded synthetic inputs for the rotate-then-quantize KV-cache decode path.

This module is the one piece shared by the CPU oracle (``oracle/``), the CUDA
path's tests and ``bench.py``.  It holds NO arithmetic of the method itself:
no rotation, no quantisation, no attention.  It only draws random numbers and
lays out shapes, so that both sides receive byte-identical inputs.

Every random draw comes from a numpy PCG64 stream keyed by
``SeedSequence([config seed, stream id, *indices])``, so that the K/V of one
(sequence, kv head) can be regenerated on its own: the oracle recomputes a few
sampled heads of a multi-gigabyte workload without materialising the rest.
(Timing runs that never meet the oracle may instead fill a cache with draws of
the same distributions from a seeded torch generator on the GPU:
``GpuWorkload(cfg, fill="device")``.)

Workload shapes follow the pages' own workloads:
  * "Shrinking the LLM KV Cache by 8x on CPU: AdapTQ" (The Results): 4-bit
    rotated codes, 4096-token contexts.
  * "FoveatedKV" (Results table): 7B GQA shapes, H_kv=8, H_q=32, D=128,
    contexts 1K..32K, top 10% of tokens fp16 and the rest fp8-E4M3 keys plus
    INT4 values.
  * "I Ported a Google Research Paper to Apple Silicon" (VeloxQuant-MLX,
    Installing and Using It): fp16 keys/values ~ N(0,1), head_dim 128.
The pages' model activations are not available, so K/V are Gaussian (or
Student-t) with planted outlier channels, the property the pages' rotation is
meant to tame ("The Problem: The Tyranny of Outliers", AdapTQ page).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# Stream ids: one independent PCG64 stream family per kind of draw.
S_K, S_V, S_Q, S_OUTLIER, S_TIER, S_LENS, S_PAGES, S_SIGNS, S_SIGMA, S_NEWTOK, S_PROJ = range(11)

# Storage format names (the same four the C header enumerates).
CODEBOOK, FP16, FP8_E4M3, INT4_G32 = "codebook", "fp16", "fp8_e4m3", "int4_g32"
CODEBOOK_QJL = "codebook_qjl"  # keys: codebook codes + residual sign sketch
CODEBOOK_OUTLIER = "codebook_outlier"  # keys: codebook codes + int8 outlier channels
OUTLIER_CALIBRATION = 256  # calibration tokens of the outlier stream (the first of sequence 0)
QJL_DIM = 128


@dataclasses.dataclass(frozen=True)
class Tier:
    """One precision tier of the cache: how K and V rows of its tokens are stored."""

    k_format: str
    v_format: str
    k_bits: int = 0  # code bits, codebook format only
    v_bits: int = 0
    codebook: str = "lloyd_max"  # or "uniform"
    fraction: float = 1.0  # share of each (sequence, kv head)'s tokens held here
    window: int = 0  # > 0 (last tier only): the newest min(window, L) tokens, stored fp16


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seq_len: int  # every sequence's length (upper bound when ragged)
    tiers: Tuple[Tier, ...]
    seed: int
    ragged_min: int = 0  # >0: lengths uniform in [ragged_min, seq_len]
    kv_dist: str = "normal"  # "normal" | "student_t4" | "normal_channel_sigma"
    outlier_mode: str = "none"  # "fixed_channels" | "pairs" | "none"
    outlier_count: int = 0
    outlier_scale: float = 1.0
    page_size: int = 16
    shuffle_pages: bool = False
    prefill_chunk: int = 0  # tokens quantised-and-appended after the first seq_len
    decode_steps: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def scaled(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


LM4 = Tier(CODEBOOK, CODEBOOK, 4, 4)

CONFIGS: Dict[str, Config] = {
    # tiny: B1, 8/8 heads, D128, ctx 1024, 4 fixed outlier channels x20, 4-bit LM K and V, seed 0
    "tiny": Config("tiny", 1, 8, 8, 128, 1024, (LM4,), seed=0,
                   outlier_mode="fixed_channels", outlier_count=4, outlier_scale=20.0),
    # Llama-7B-shaped layer: B8, 32/32 heads, D128, ctx 8192, 1% outlier channels x50, 4-bit LM
    "llama7b": Config("llama7b", 8, 32, 32, 128, 8192, (LM4,), seed=1,
                      outlier_mode="pairs", outlier_count=41, outlier_scale=50.0),
    # the same layer with a recent-token window: the newest 256 tokens of every sequence in
    # fp16 (the hybrid threshold), the older ones 4-bit LM
    "llama7b_window": Config("llama7b_window", 8, 32, 32, 128, 8192, (LM4, Tier(FP16, FP16, window=256)), seed=1,
                             outlier_mode="pairs", outlier_count=41, outlier_scale=50.0),
    # the same layer with outlier two-stream keys: 8 channels per kv head (calibrated on the
    # first 256 tokens of sequence 0) as int8, the rest 4-bit LM; 4-bit LM values
    "llama7b_outlier": Config("llama7b_outlier", 8, 32, 32, 128, 8192, (Tier(CODEBOOK_OUTLIER, CODEBOOK, 4, 4),),
                              seed=1, outlier_mode="pairs", outlier_count=41, outlier_scale=50.0),
    # the same layer with product-quantised keys: 3-bit LM codes + 128-bit residual sign
    # sketch (4 bits per coordinate), 4-bit LM values
    "llama7b_prod": Config("llama7b_prod", 8, 32, 32, 128, 8192, (Tier(CODEBOOK_QJL, CODEBOOK, 3, 4),), seed=1,
                           outlier_mode="pairs", outlier_count=41, outlier_scale=50.0),
    # GQA long-context: B32, 32/8 heads, D128, ctx 32768; top 10% fp16, rest fp8 K + INT4-g32 V
    "gqa32k": Config("gqa32k", 32, 32, 8, 128, 32768,
                     (Tier(FP16, FP16, fraction=0.1), Tier(FP8_E4M3, INT4_G32, fraction=0.9)),
                     seed=2, outlier_mode="pairs", outlier_count=10, outlier_scale=30.0),
    # ragged: 64 sequences, lengths U[512, 65536], 32/8 heads, 3-bit LM K / 2-bit LM V,
    # 16-token pages in shuffled order, Student-t(4)/sqrt(2)
    "ragged": Config("ragged", 64, 32, 8, 128, 65536, (Tier(CODEBOOK, CODEBOOK, 3, 2),),
                     seed=3, ragged_min=512, kv_dist="student_t4", shuffle_pages=True),
    # append + decode: B4, 16/16 heads, D256, ctx 131072 + 16384-token chunk, 4-bit LM,
    # 128 decode steps, per-channel std log-uniform in [0.1, 10]
    "append": Config("append", 4, 16, 16, 256, 131072, (LM4,), seed=4,
                     kv_dist="normal_channel_sigma", prefill_chunk=16384, decode_steps=128),
}


def rng(cfg: Config, stream: int, *idx: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([cfg.seed, stream, *idx]))


# ----------------------------------------------------------------------------- lengths


def seq_lens(cfg: Config) -> np.ndarray:
    """Total context length of every sequence (int64 [B])."""
    if cfg.ragged_min > 0:
        return rng(cfg, S_LENS).integers(cfg.ragged_min, cfg.seq_len, size=cfg.batch,
                                         endpoint=True).astype(np.int64)
    return np.full(cfg.batch, cfg.seq_len, dtype=np.int64)


def window_len(cfg: Config, total: int) -> int:
    """Tokens in the recent-token window (a last tier with `window` > 0), else 0."""
    w = cfg.tiers[-1].window
    return min(w, total) if w > 0 else 0


def tier_lens(cfg: Config, total: int) -> List[int]:
    """Tokens per tier for one (sequence, kv head) of `total` tokens.  A window tier (last)
    takes the newest min(window, total); of the older ones the first tier gets
    round(fraction * older) and the last of the other tiers the rest."""
    w = window_len(cfg, total)
    base = cfg.tiers[:-1] if cfg.tiers[-1].window > 0 else cfg.tiers
    rest = total - w
    out, left = [], rest
    for i, t in enumerate(base):
        n = left if i == len(base) - 1 else min(left, int(round(t.fraction * rest)))
        out.append(n)
        left -= n
    if cfg.tiers[-1].window > 0:
        out.append(w)
    return out


# ----------------------------------------------------------------------------- values


def outlier_multipliers(cfg: Config) -> np.ndarray:
    """float32 [Hkv, D] channel multipliers (1 everywhere but the outlier channels).
    The same channels are applied to K and V."""
    m = np.ones((cfg.num_kv_heads, cfg.head_dim), dtype=np.float32)
    if cfg.outlier_mode == "fixed_channels":
        ch = rng(cfg, S_OUTLIER).permutation(cfg.head_dim)[: cfg.outlier_count]
        m[:, ch] = cfg.outlier_scale
    elif cfg.outlier_mode == "pairs":
        flat = rng(cfg, S_OUTLIER).choice(cfg.num_kv_heads * cfg.head_dim,
                                          size=cfg.outlier_count, replace=False)
        m.reshape(-1)[flat] = cfg.outlier_scale
    return m


def channel_sigma(cfg: Config, which: int) -> np.ndarray:
    """float32 [Hkv, D] per-channel std, log-uniform in [0.1, 10] (K and V drawn apart)."""
    r = rng(cfg, S_SIGMA, which)
    return np.exp(r.uniform(math.log(0.1), math.log(10.0),
                            size=(cfg.num_kv_heads, cfg.head_dim))).astype(np.float32)


def _draw(cfg: Config, r: np.random.Generator, n: int) -> np.ndarray:
    if cfg.kv_dist == "student_t4":
        return (r.standard_t(4.0, size=(n, cfg.head_dim)) / math.sqrt(2.0)).astype(np.float32)
    return r.standard_normal((n, cfg.head_dim), dtype=np.float32)


def kv_head(cfg: Config, which: int, b: int, h: int, n: int, stream: int = -1) -> np.ndarray:
    """fp16 [n, D] keys (which=0) or values (which=1) of sequence b, kv head h.
    `stream` selects a separate family (used for appended / decode-step tokens)."""
    key = (S_K if which == 0 else S_V)
    r = rng(cfg, key, b, h) if stream < 0 else rng(cfg, S_NEWTOK, which, stream, b, h)
    x = _draw(cfg, r, n)
    if cfg.kv_dist == "normal_channel_sigma":
        x *= channel_sigma(cfg, which)[h]
    x *= outlier_multipliers(cfg)[h]
    return x.astype(np.float16)


def queries(cfg: Config, step: int = 0) -> np.ndarray:
    """fp16 [B, Hq, D] decode queries, q ~ N(0, 1)."""
    r = rng(cfg, S_Q, step)
    return r.standard_normal((cfg.batch, cfg.num_q_heads, cfg.head_dim),
                             dtype=np.float32).astype(np.float16)


def signs(cfg: Config, which: int, layer: int = 0) -> np.ndarray:
    """int8 [Hkv, D] Rademacher signs (+1/-1) for K (which=0) or V (which=1), drawn
    independently per (layer, kv head, K|V).  They are an input of the method."""
    r = rng(cfg, S_SIGNS, layer, which)
    return np.where(r.integers(0, 2, size=(cfg.num_kv_heads, cfg.head_dim)) == 0,
                    1, -1).astype(np.int8)


def qjl_projection(cfg: Config, layer: int = 0) -> np.ndarray:
    """float32 [QJL_DIM, D] projection of the residual sign sketch, iid N(0,1) entries, one
    per layer.  Like the signs, it is an input of the method."""
    return rng(cfg, S_PROJ, layer).standard_normal((QJL_DIM, cfg.head_dim)).astype(np.float32)


def tier_members(cfg: Config, b: int, h: int, total: int) -> List[np.ndarray]:
    """Token positions (sorted) held by each tier for sequence b, kv head h.  With one
    tier all tokens are in it; otherwise the first tier takes the tokens with the highest
    seeded U(0,1) score (ties cannot occur with continuous draws) and the rest follow."""
    lens = tier_lens(cfg, total)
    w = window_len(cfg, total)
    rest = total - w
    tail = [np.arange(rest, total)] if cfg.tiers[-1].window > 0 else []  # the window: newest tokens
    base = lens[:-1] if tail else lens
    if len(base) == 1:
        return [np.arange(rest)] + tail
    score = rng(cfg, S_TIER, b, h).random(rest)
    order = np.argsort(-score, kind="stable")
    out, at = [], 0
    for n in base:
        out.append(np.sort(order[at: at + n]))
        at += n
    return out + tail


# ----------------------------------------------------------------------------- paging


@dataclasses.dataclass
class PageMap:
    """Block tables of one tier: physical page of logical page p of sequence b."""

    block_table: np.ndarray  # int32 [B, max_pages], -1 where unused
    lens: np.ndarray  # int64 [B] tokens held per sequence in this tier
    num_pages: int
    page_size: int

    def slots(self, b: int, positions: np.ndarray) -> np.ndarray:
        """Pool slot (physical page * page_size + offset) of token positions of seq b."""
        positions = np.asarray(positions, dtype=np.int64)
        page = self.block_table[b, positions // self.page_size].astype(np.int64)
        return (page * self.page_size + positions % self.page_size).astype(np.int32)


def page_map(cfg: Config, lens: np.ndarray, tier: int = 0, spare_pages: int = 0) -> PageMap:
    """Assign physical pages to every sequence.  Identity order unless the config shuffles
    pages (then a seeded permutation of the pool)."""
    ps = cfg.page_size
    per = [(int(n) + ps - 1) // ps for n in lens]
    total = sum(per) + spare_pages
    phys = np.arange(total, dtype=np.int32)
    if cfg.shuffle_pages:
        phys = rng(cfg, S_PAGES, tier).permutation(total).astype(np.int32)
    maxp = max(1, max(per) if per else 1)
    bt = np.full((len(lens), maxp), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(per):
        bt[b, :n] = phys[at: at + n]
        at += n
    return PageMap(bt, np.asarray(lens, dtype=np.int64), total, ps)


def kv_bytes_fp16(cfg: Config, total_tokens: int) -> int:
    """Bytes of an unquantised fp16 K+V cache holding `total_tokens` per kv head."""
    return total_tokens * cfg.num_kv_heads * cfg.head_dim * 2 * 2


# ----------------------------------------------------------------------------- assembly


def capacity(cfg: Config) -> int:
    """Largest number of tokens any sequence reaches (context + appended chunk + steps)."""
    return cfg.seq_len + cfg.prefill_chunk + cfg.decode_steps


_POOL = None


def _pool():
    """Threads for generation: every (sequence, head) has its own stream and numpy's bulk
    random fills release the GIL, so heads are drawn in parallel with identical results."""
    global _POOL
    if _POOL is None:
        import concurrent.futures
        import os
        _POOL = concurrent.futures.ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def sequence_kv(cfg: Config, b: int, total: int):
    """Per-head fp16 keys and values of sequence b's first `total` positions:
    two lists over kv heads of [total, D] arrays."""
    jobs = [(w, h) for w in (0, 1) for h in range(cfg.num_kv_heads)]
    out = list(_pool().map(lambda j: kv_head(cfg, j[0], b, j[1], total), jobs))
    return out[: cfg.num_kv_heads], out[cfg.num_kv_heads:]


def sequence_tiers(cfg: Config, b: int, total: int):
    """Token-major K/V of sequence b split into tiers: a list over tiers of
    (k [L_t, Hkv, D], v [L_t, Hkv, D]) fp16.  Slot t of a tier holds, for kv head h, the
    t-th (in position order) token of h that belongs to the tier."""
    ks, vs = sequence_kv(cfg, b, total)
    lens = tier_lens(cfg, total)
    out = [(np.empty((n, cfg.num_kv_heads, cfg.head_dim), np.float16),
            np.empty((n, cfg.num_kv_heads, cfg.head_dim), np.float16)) for n in lens]
    for h in range(cfg.num_kv_heads):
        for t, members in enumerate(tier_members(cfg, b, h, total)):
            out[t][0][:, h] = ks[h][members]
            out[t][1][:, h] = vs[h][members]
    return out


def calibration_keys(cfg: Config) -> np.ndarray:
    """fp16 keys [N, Hkv, D] of the first N = min(OUTLIER_CALIBRATION, L_0) tokens of sequence
    0, in position order: the calibration sample of the outlier stream."""
    n = min(OUTLIER_CALIBRATION, int(seq_lens(cfg)[0]))
    return np.stack([kv_head(cfg, 0, 0, h, n) for h in range(cfg.num_kv_heads)], axis=1)


def chunk_kv(cfg: Config, b: int, stream: int, n: int):
    """Token-major fp16 K/V [n, Hkv, D] of n appended tokens of sequence b, drawn from the
    appended-token stream `stream` (0 = prefill chunk, 1 + s = decode step s)."""
    k = np.stack([kv_head(cfg, 0, b, h, n, stream=stream) for h in range(cfg.num_kv_heads)], axis=1)
    v = np.stack([kv_head(cfg, 1, b, h, n, stream=stream) for h in range(cfg.num_kv_heads)], axis=1)
    return k, v


class GpuWorkload:
    """The cache of a config built on the GPU through the library's quantize-append, one
    sequence at a time (host fp16 -> device -> kvq_quantize_append).  Holds one PagedCache
    and block table per tier, sized for `capacity(cfg)` tokens per sequence."""

    def __init__(self, cfg: Config, device: str = "cuda", fill=True):
        """fill: True -- every sequence's K/V drawn on the host (the PCG64 streams above, the
        same values the oracle sees); "device" -- drawn on the GPU from a seeded torch
        generator with the same distributions (single-tier configs; for timing runs whose
        result is not compared with the oracle); False -- left empty."""
        import torch
        import quantized_decode_attention_rht_gb300 as kvq

        self.cfg = cfg
        self.lens = seq_lens(cfg)  # context length per sequence
        cap = np.array([min(capacity(cfg), int(n) + cfg.prefill_chunk + cfg.decode_steps)
                        for n in self.lens])
        ntier = len(cfg.tiers)
        # capacity per tier: every appended token goes to the last tier; with a window, the
        # window keeps its size and the tier before it gets one spare slot per sequence (the
        # token a decode step moves out of the window)
        cap_t = [np.array([tier_lens(cfg, int(n))[t] for n in self.lens]) for t in range(ntier)]
        if cfg.tiers[-1].window > 0:
            cap_t[-2] = cap_t[-2] + 1
        else:
            cap_t[-1] = cap_t[-1] + (cap - self.lens)
        self.maps = [page_map(cfg, cap_t[t], tier=t) for t in range(ntier)]
        self.tier_len = [np.array([tier_lens(cfg, int(n))[t] for n in self.lens]) for t in range(ntier)]
        ks, vs = signs(cfg, 0), signs(cfg, 1)
        self.k_signs = torch.from_numpy(ks).to(device)
        self.v_signs = torch.from_numpy(vs).to(device)
        self.k_qjl = (torch.from_numpy(qjl_projection(cfg)).to(device)
                      if any(t.k_format == CODEBOOK_QJL for t in cfg.tiers) else None)
        self.k_outliers = None
        if any(t.k_format == CODEBOOK_OUTLIER for t in cfg.tiers):
            # the library's calibration over the first tokens of sequence 0
            self.calib_tokens = calibration_keys(cfg)
            self.k_outliers = torch.empty((cfg.num_kv_heads, kvq.OUTLIER_CHANNELS), dtype=torch.int32,
                                          device=device)
            kvq.kvq_outlier_calibrate(torch.from_numpy(self.calib_tokens).to(device), self.k_outliers)
        self.caches = []
        for t, tier in enumerate(cfg.tiers):
            self.caches.append(kvq.PagedCache(cfg.head_dim, cfg.num_kv_heads, self.maps[t].num_pages,
                                              tier.k_format, tier.v_format, tier.k_bits, tier.v_bits,
                                              self.k_signs, self.v_signs, cfg.page_size, tier.codebook, device,
                                              k_qjl=self.k_qjl if tier.k_format == CODEBOOK_QJL else None,
                                              k_outliers=self.k_outliers if tier.k_format == CODEBOOK_OUTLIER
                                              else None))
        self.block_tables = [torch.from_numpy(np.maximum(m.block_table, 0)).to(device) for m in self.maps]
        self.seq_lens_dev = [torch.from_numpy(l.astype(np.int32)).to(device) for l in self.tier_len]
        self.device = device
        if fill == "device":
            self.fill_on_device()
        elif fill:
            for b in range(cfg.batch):
                for t, (k, v) in enumerate(sequence_tiers(cfg, b, int(self.lens[b]))):
                    self.append(t, b, np.arange(k.shape[0]), k, v)
            torch.cuda.synchronize()

    def device_draw(self, gen, which: int, h_count: int, n: int):
        """fp16 [n, Hkv, D] draws on the device with the config's distribution: N(0,1) or
        Student-t(4)/sqrt(2), times the per-channel std or the outlier multipliers."""
        import torch
        cfg = self.cfg
        shape = (n, h_count, cfg.head_dim)
        if cfg.kv_dist == "student_t4":  # t = z / sqrt(chi2_4 / 4), chi2_4 a sum of 4 squared normals
            z = torch.randn(shape, generator=gen, device=self.device)
            chi = sum(torch.randn(shape, generator=gen, device=self.device) ** 2 for _ in range(4))
            x = z / torch.sqrt(chi / 4.0) / math.sqrt(2.0)
        else:
            x = torch.randn(shape, generator=gen, device=self.device)
        if cfg.kv_dist == "normal_channel_sigma":
            x *= torch.from_numpy(channel_sigma(cfg, which)).to(self.device)
        x *= torch.from_numpy(outlier_multipliers(cfg)).to(self.device)
        return x.half()

    def fill_on_device(self, chunk: int = 16384):
        import torch
        cfg = self.cfg
        assert len(cfg.tiers) == 1, "device fill: single-tier configs"
        gen = torch.Generator(device=self.device)
        gen.manual_seed(1000003 * cfg.seed + 17)
        for b in range(cfg.batch):
            n = int(self.lens[b])
            for t0 in range(0, n, chunk):
                m = min(chunk, n - t0)
                k = self.device_draw(gen, 0, cfg.num_kv_heads, m)
                v = self.device_draw(gen, 1, cfg.num_kv_heads, m)
                slots = torch.from_numpy(self.maps[0].slots(b, np.arange(t0, t0 + m))).to(self.device)
                self.caches[0].append(k, v, slots)
        torch.cuda.synchronize()

    def append(self, tier: int, b: int, positions, k: np.ndarray, v: np.ndarray, stream=None):
        """Quantise-and-append host fp16 K/V [n, Hkv, D] at `positions` of sequence b."""
        import torch
        slots = torch.from_numpy(self.maps[tier].slots(b, positions)).to(self.device)
        kd = torch.from_numpy(np.ascontiguousarray(k)).to(self.device)
        vd = torch.from_numpy(np.ascontiguousarray(v)).to(self.device)
        self.caches[tier].append(kd, vd, slots, stream)

    def set_len(self, tier: int, lens: np.ndarray):
        import torch
        self.tier_len[tier] = np.asarray(lens)
        self.seq_lens_dev[tier].copy_(torch.from_numpy(self.tier_len[tier].astype(np.int32)))

    def views(self):
        import quantized_decode_attention_rht_gb300 as kvq
        return [kvq.TierView(c, bt, sl) for c, bt, sl in zip(self.caches, self.block_tables, self.seq_lens_dev)]

    def cache_bytes(self) -> int:
        """Algorithmic bytes of the cache rows + side data that one decode call reads."""
        total = 0
        import quantized_decode_attention_rht_gb300 as kvq
        for t, tier in enumerate(self.cfg.tiers):
            rk, ak = kvq.kvq_row_bytes(tier.k_format, tier.k_bits, self.cfg.head_dim)
            rv, av = kvq.kvq_row_bytes(tier.v_format, tier.v_bits, self.cfg.head_dim)
            total += int(self.tier_len[t].sum()) * self.cfg.num_kv_heads * (rk + ak + rv + av)
        return total
