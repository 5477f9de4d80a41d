"""GPU parity of kvq_decode_attention against the oracle.

Exact-bytes cases: the ORACLE encodes the cache; the same bytes are uploaded to the GPU;
GPU decode attention must match the oracle's dequantise-then-attend within 2e-3 max-abs.
Shapes follow each workload at sizes the oracle finishes in seconds, spanning several
pages and split-K chunks with ragged tails."""
import math

import numpy as np
import pytest

import workloads as W
from oracle import attention as oatt
from tests import gpu_util as gu


def seqs_for(cfg, lens):
    """Per tier, per sequence (k, v) for the given total lengths."""
    per_seq = [W.sequence_tiers(cfg, b, int(n)) for b, n in enumerate(lens)]
    return [[per_seq[b][t] for b in range(len(lens))] for t in range(len(cfg.tiers))]


def run_exact(cfg, lens, split_tokens=0, shuffle=None, q=None):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    tiers_kv = seqs_for(cfg, lens)
    built = gu.build_exact(kvq, torch, list(cfg.tiers), tiers_kv, W.signs(cfg, 0), W.signs(cfg, 1),
                           cfg.page_size, shuffle, k_qjl=W.qjl_projection(cfg))
    if q is None:
        q = W.queries(cfg.scaled(batch=len(lens)))
    got = gu.gpu_decode(kvq, torch, built.views, q, split_tokens)
    want = oatt.decode_attention(q, built.ora)
    return got, want, built, q


EXACT_CASES = {
    "tiny_full": (W.CONFIGS["tiny"], [1024]),
    "llama7b": (W.CONFIGS["llama7b"].scaled(batch=2, num_q_heads=4, num_kv_heads=4), [1000, 777]),
    "gqa32k": (W.CONFIGS["gqa32k"].scaled(batch=2, num_q_heads=8, num_kv_heads=2), [3000, 2111]),
    "ragged": (W.CONFIGS["ragged"].scaled(batch=5, num_q_heads=8, num_kv_heads=2, seq_len=2500, ragged_min=1), None),
    "append_d256": (W.CONFIGS["append"].scaled(batch=2, num_q_heads=4, num_kv_heads=4, seq_len=1500), [1500, 1499]),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(EXACT_CASES))
def test_decode_matches_oracle(name):
    cfg, lens = EXACT_CASES[name]
    if lens is None:
        lens = list(W.seq_lens(cfg))
    got, want, _, _ = run_exact(cfg, lens, shuffle=7 if cfg.shuffle_pages else None)
    err = np.abs(got - want)
    scale = np.abs(want).max()
    print(f"{name}: max-abs {err.max():.3e} (output max {scale:.3f})")
    assert np.all(np.isfinite(got))
    assert err.max() <= gu.ATOL_OUT
    assert err.max() <= 1e-4 * max(1.0, scale)  # fp32 accumulation: far inside the bound


@pytest.mark.gpu
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_decode_edge_lengths_and_groups(group):
    """Lengths 0, 1, 15, 16, 17 and a multi-chunk one in one batch, for every group size."""
    hkv = 2
    cfg = W.CONFIGS["llama7b"].scaled(batch=6, num_q_heads=hkv * group, num_kv_heads=hkv)
    lens = [0, 1, 15, 16, 17, 700]
    got, want, _, _ = run_exact(cfg, lens, split_tokens=64, shuffle=3)
    assert np.all(got[0] == 0)  # empty context
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


CODE_WIDTHS = [(128, 1, 3, 3), (128, 4, 3, 3), (128, 2, 2, 4), (128, 1, 4, 2), (128, 4, 2, 3),
               (256, 1, 3, 3), (256, 4, 4, 4), (256, 2, 2, 3), (256, 4, 3, 2), (256, 1, 2, 2),
               (128, 8, 3, 2), (128, 8, 4, 4), (256, 8, 3, 3),  # 8 heads: two 4-head items a chunk
               (64, 1, 4, 4), (64, 2, 3, 3), (64, 4, 3, 2), (64, 8, 2, 4)]  # D = 64: the generic kernel


@pytest.mark.gpu
@pytest.mark.parametrize("d,group,kb,vb", CODE_WIDTHS)
def test_decode_code_widths(d, group, kb, vb):
    """Every head_dim, code width (the runs of packed bits a lane reads differ for each) and
    group size of the codebook path, Lloyd-Max and uniform tables, ragged lengths."""
    hkv = 2
    codebook = "uniform" if (kb + vb) % 2 else "lloyd_max"
    cfg = W.CONFIGS["llama7b"].scaled(batch=4, num_q_heads=hkv * group, num_kv_heads=hkv, head_dim=d,
                                      tiers=(W.Tier("codebook", "codebook", k_bits=kb, v_bits=vb,
                                                    codebook=codebook),))
    lens = [1, 47, 300, 129]
    got, want, _, _ = run_exact(cfg, lens, split_tokens=96, shuffle=5)
    assert np.all(np.isfinite(got))
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


# (head_dim, query heads per kv head, page size, tiers): pools whose pages are not 16 tokens
# run on the generic kernel, whose warps step through a page TPS tokens at a time (16 at
# D = 64 with one head per kv head, 8 at D = 128, 4 at D = 128 with two heads or D = 256
# with one, 2 at D = 128 with four, 1 with eight); sizes that are no multiple of TPS leave
# the last step of a page part empty, a one-token page is all tail
_CB44 = (W.Tier("codebook", "codebook", 4, 4),)
_TWO_TIER = W.CONFIGS["gqa32k"].tiers
PAGE_SIZES = [(64, 1, 24, _CB44), (64, 1, 5, _CB44), (128, 1, 12, _CB44), (128, 2, 6, _CB44),
              (256, 1, 10, _CB44), (128, 4, 1, _CB44), (128, 8, 3, _CB44), (128, 4, 32, _CB44),
              (128, 4, 24, _TWO_TIER), (128, 1, 7, _TWO_TIER)]


@pytest.mark.gpu
@pytest.mark.parametrize("d,group,ps,tiers", PAGE_SIZES)
def test_decode_page_sizes(d, group, ps, tiers):
    """Pages of other sizes than 16 tokens (the generic kernel): lengths of one token, one
    page, a page and a token, and a ragged several-split one, on shuffled pages."""
    hkv = 2
    cfg = W.CONFIGS["llama7b"].scaled(batch=4, num_q_heads=hkv * group, num_kv_heads=hkv, head_dim=d,
                                      page_size=ps, tiers=tiers)
    lens = [1, ps, ps + 1, 333]
    got, want, _, _ = run_exact(cfg, lens, split_tokens=4 * ps, shuffle=5)
    assert np.all(np.isfinite(got))
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


# the most tiers one call attends (KVQ_MAX_TIERS): fp16 near and fp8 / INT4 far tiers (one
# launch of the fused fp16 / fp8 kernel, with the window below), a 4-bit codebook tier (the
# codebook kernel) and an fp16 recent-token window
FOUR_TIERS = (W.Tier("fp16", "fp16", fraction=0.1), W.Tier("fp8_e4m3", "int4_g32", fraction=0.4),
              W.Tier("codebook", "codebook", 4, 4), W.Tier("fp16", "fp16", window=64))


@pytest.mark.gpu
@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("group", [1, 4, 8])
def test_decode_four_tiers(group, split):
    """One softmax over four tiers of three kernel families, lengths from one token (the
    window alone) to several splits of every tier."""
    hkv = 2
    cfg = W.CONFIGS["gqa32k"].scaled(batch=4, num_q_heads=hkv * group, num_kv_heads=hkv, tiers=FOUR_TIERS)
    lens = [1, 63, 700, 2111]
    got, want, _, _ = run_exact(cfg, lens, split_tokens=split, shuffle=3)
    assert np.all(np.isfinite(got))
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


QJL_WIDTHS = [(1, 3, 4), (1, 2, 2), (2, 2, 3), (2, 4, 4), (4, 4, 4), (4, 3, 2)]


@pytest.mark.gpu
@pytest.mark.parametrize("group,kb,vb", QJL_WIDTHS)
def test_decode_qjl_keys(group, kb, vb):
    """Keys with a residual sign sketch (head_dim 128): the scores carry the sketch's
    correction ||r~|| sqrt(pi/2)/m sum_j z_j <S_j, q~>; both the one-query-head path and
    the grouped path, ragged lengths, several splits."""
    hkv = 2
    cfg = W.CONFIGS["llama7b"].scaled(batch=4, num_q_heads=hkv * group, num_kv_heads=hkv,
                                      tiers=(W.Tier("codebook_qjl", "codebook", k_bits=kb, v_bits=vb),))
    lens = [1, 47, 300, 129]
    got, want, built, q = run_exact(cfg, lens, split_tokens=96, shuffle=5)
    assert np.all(np.isfinite(got))
    err = np.abs(got - want).max()
    assert err <= 1e-4 * max(1.0, np.abs(want).max())
    # the correction is not negligible: leaving it out moves the output far past the error
    plain = np.zeros_like(want)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            keys, values = oatt.dequantised_kv(built.ora, b, h // group)
            plain[b, h] = oatt.attend(q[b, h].astype(np.float64), keys, values)
    assert np.abs(plain - want).max() > 100 * max(err, 1e-6)


@pytest.mark.gpu
def test_decode_qjl_near_tier_with_codebook_far_tier():
    """Two tiers in one call: sketched 4-bit keys (near) and plain 2-bit codebook (far)."""
    cfg = W.CONFIGS["llama7b"].scaled(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                                      tiers=(W.Tier("codebook_qjl", "codebook", k_bits=4, v_bits=4, fraction=0.25),
                                             W.Tier("codebook", "codebook", k_bits=2, v_bits=2)))
    lens = [5, 400, 1111]
    got, want, _, _ = run_exact(cfg, lens, split_tokens=64, shuffle=2)
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


@pytest.mark.gpu
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_decode_head_dim_64_two_tier(group):
    """head_dim 64 (the generic kernel): fp16 near tier + fp8 keys / INT4 values far tier,
    every group size, lengths spanning empty, sub-page and multi-chunk."""
    hkv = 2
    cfg = W.CONFIGS["gqa32k"].scaled(batch=5, num_q_heads=hkv * group, num_kv_heads=hkv, head_dim=64)
    lens = [0, 3, 16, 333, 1500]
    got, want, _, _ = run_exact(cfg, lens, split_tokens=64, shuffle=4)
    assert np.all(got[0] == 0)
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


@pytest.mark.gpu
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("split", [32, 0])
def test_decode_two_tier_edge_lengths(group, split):
    """fp16 near tier + fp8 / INT4 far tier at head_dim 128 on the fused kernel for every
    group size (a group of 8 runs as two items of four heads per chunk), short and
    multi-split lengths, small forced splits and the default plan."""
    cfg = W.CONFIGS["gqa32k"].scaled(batch=5, num_q_heads=2 * group, num_kv_heads=2)
    lens = [1, 9, 10, 11, 1234]  # near tier holds round(0.1 L): 0, 1, 1, 1, 123 tokens
    got, want, _, _ = run_exact(cfg, lens, split_tokens=split)
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


@pytest.mark.gpu
def test_two_tier_many_splits():
    """Split size 16 over long two-tier sequences (78 partials per sequence for the longest):
    same result as the default split."""
    cfg = W.CONFIGS["gqa32k"].scaled(batch=3, num_q_heads=8, num_kv_heads=2)
    lens = [1234, 700, 1]
    got16, want, _, _ = run_exact(cfg, lens, split_tokens=16)
    got0, _, _, _ = run_exact(cfg, lens)
    assert np.abs(got16 - want).max() <= 1e-4 * max(1.0, np.abs(want).max())
    np.testing.assert_allclose(got16, got0, rtol=0, atol=2e-6 * max(1.0, np.abs(got0).max()))


@pytest.mark.gpu
def test_split_invariance():
    """Split-K over 1, 2, 7 chunks and one chunk per page gives the same output."""
    cfg = W.CONFIGS["ragged"].scaled(batch=2, num_q_heads=8, num_kv_heads=2)
    lens = [1777, 1760]
    outs = []
    for split in (1792, 896, 256, 16):
        got, want, _, _ = run_exact(cfg, lens, split_tokens=split)
        outs.append(got)
        assert np.abs(got - want).max() <= gu.ATOL_OUT
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=2e-6 * max(1.0, np.abs(outs[0]).max()))


@pytest.mark.gpu
def test_fp16_cache_equals_plain_attention():
    """With the cache stored as fp16 (no codes), decode attention equals plain
    softmax(q K^T / sqrt(d)) V over the original fp16 keys/values, up to the fp16 rounding
    of the stored rotated vectors (relative 2^-11 per element)."""
    torch = gu.torch_cuda()
    cfg = W.CONFIGS["gqa32k"].scaled(batch=2, num_q_heads=8, num_kv_heads=2, tiers=(W.Tier("fp16", "fp16"),),
                                     outlier_mode="none")
    lens = [900, 533]
    got, _, _, q = run_exact(cfg, lens)
    g = cfg.group
    for b, n in enumerate(lens):
        ks, vs = W.sequence_kv(cfg, b, n)
        for h in range(cfg.num_q_heads):
            k = torch.from_numpy(ks[h // g].astype(np.float64))
            v = torch.from_numpy(vs[h // g].astype(np.float64))
            qq = torch.from_numpy(q[b, h].astype(np.float64))
            ref = torch.nn.functional.scaled_dot_product_attention(qq[None, None, None], k[None, None],
                                                                   v[None, None])[0, 0, 0].numpy()
            # fp16 rounding of rotated K shifts scores by <= 2^-11 * |q||k|/sqrt(d) ~ 5e-3 here
            assert np.abs(got[b, h] - ref).max() < 2e-2
            assert np.linalg.norm(got[b, h] - ref) / np.linalg.norm(ref) < 5e-3


# ----------------------------------------------------------------------------- full sizes


def head_tokens(cfg, b, g, total, with_chunk):
    """fp16 K and V [n, D] of every tier of sequence b, kv head g, in tier slot order,
    regenerated from the seeded inputs (plus the appended prefill chunk)."""
    k = W.kv_head(cfg, 0, b, g, total)
    v = W.kv_head(cfg, 1, b, g, total)
    members = W.tier_members(cfg, b, g, total)
    out = [[k[m], v[m]] for m in members]
    if with_chunk:
        out[-1][0] = np.concatenate([out[-1][0], W.kv_head(cfg, 0, b, g, cfg.prefill_chunk, stream=0)])
        out[-1][1] = np.concatenate([out[-1][1], W.kv_head(cfg, 1, b, g, cfg.prefill_chunk, stream=0)])
    return out


def pool_index(torch, wl, t, b, n):
    ps = wl.cfg.page_size
    pos = np.arange(n)
    pages = torch.from_numpy(wl.maps[t].block_table[b, pos // ps].astype(np.int64)).cuda()
    offs = torch.from_numpy((pos % ps).astype(np.int64)).cuda()
    return pages, offs


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "llama7b", "llama7b_prod", "llama7b_window", "llama7b_outlier", "gqa32k",
                                  "ragged", "append"])
def test_full_size_sampled_heads(name):
    """Every workload at its full size, built on the GPU by kvq_quantize_append and decoded with
    the split plan the benchmark uses.  For sampled (sequence, kv head) pairs:
      1. quantize parity at full length: the GPU's rows against the oracle's encoder;
      2. decode parity on identical bytes: the oracle's rows are written over the GPU's for
         those heads, and the GPU outputs of their query heads must match the oracle's
         dequantise-then-attend within 2e-3."""
    from oracle import cache as ocache
    from oracle import rotation as orot
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    cfg = W.CONFIGS[name]
    wl = W.GpuWorkload(cfg)
    last = len(cfg.tiers) - 1
    if cfg.prefill_chunk:
        for b in range(cfg.batch):
            k, v = W.chunk_kv(cfg, b, 0, cfg.prefill_chunk)
            wl.append(last, b, int(wl.tier_len[last][b]) + np.arange(cfg.prefill_chunk), k, v)
        wl.set_len(last, wl.tier_len[last] + cfg.prefill_chunk)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    picks = [(int(rng.integers(cfg.batch)), int(rng.integers(cfg.num_q_heads))) for _ in range(3)]
    picks.append((cfg.batch - 1, cfg.num_q_heads - 1))
    ks_all, vs_all = W.signs(cfg, 0), W.signs(cfg, 1)
    proj = W.qjl_projection(cfg)
    chans = None
    if any(t.k_format == "codebook_outlier" for t in cfg.tiers):
        chans = ocache.outlier_channels(W.calibration_keys(cfg))  # the oracle's calibration ...
        assert np.array_equal(wl.k_outliers.cpu().numpy(), chans)  # ... equals the library's
    kv_ref, sketch_rows = {}, {}
    near = total_el = 0
    for b, g in sorted({(b, h // cfg.group) for b, h in picks}):
        parts = head_tokens(cfg, b, g, int(wl.lens[b]), bool(cfg.prefill_chunk))
        K, V, SK = [], [], []
        for t, tier in enumerate(cfg.tiers):
            cache = wl.caches[t]
            n = int(wl.tier_len[t][b])
            assert parts[t][0].shape[0] == n
            pages, offs = pool_index(torch, wl, t, b, n)
            for side, x, sg in (("k", parts[t][0], ks_all[g]), ("v", parts[t][1], vs_all[g])):
                fmt = getattr(tier, f"{side}_format")
                bits = getattr(tier, f"{side}_bits")
                rows_t, aux_t = getattr(cache, f"{side}_rows"), getattr(cache, f"{side}_aux")
                rows_g = rows_t[pages, g, offs].cpu().numpy()
                aux_g = None if aux_t is None else aux_t[pages, g, offs].cpu().numpy()
                tab = gu.tables(tier.codebook, bits) if fmt.startswith("codebook") else (None, None)
                if fmt == "codebook_qjl":
                    gu.check_qjl_rows(x, sg, bits, proj, rows_g, aux_g, kind=tier.codebook)
                elif fmt == "codebook_outlier":
                    gu.check_outlier_rows(x, sg, bits, chans[g], rows_g, aux_g, kind=tier.codebook)
                elif fmt == "codebook":
                    st = gu.check_codebook_codes(x, sg, bits, rows_g, aux_g[:, 0], kind=tier.codebook)
                    near, total_el = near + st[1], total_el + st[2]
                elif fmt == "int4_g32":
                    gu.check_int4_rows(x, sg, rows_g, aux_g)
                else:
                    gu.check_float_rows(x, sg, fmt, rows_g)
                rows_o, aux_o = ocache.encode(x, sg, fmt, bits, tab[1], tab[0], proj,
                                              chans[g] if fmt == "codebook_outlier" else None)
                if side == "k":
                    SK.append((rows_o, aux_o) if fmt == "codebook_qjl" else n)
                rows_t[pages, g, offs] = torch.from_numpy(rows_o).cuda()
                if aux_t is not None:
                    aux_t[pages, g, offs] = torch.from_numpy(np.asarray(aux_o).reshape(n, -1)).cuda()
                dec = ocache.decode(rows_o, aux_o, fmt, sg, cfg.head_dim, bits, tab[0],
                                    chans[g] if fmt == "codebook_outlier" else None)
                (K if side == "k" else V).append(dec)
        kv_ref[(b, g)] = (np.concatenate(K), np.concatenate(V))
        sketch_rows[(b, g)] = SK
    if total_el:
        assert near < gu.MAX_BOUNDARY_FRACTION * total_el, (near, total_el)
    q = W.queries(cfg)
    got = gu.gpu_decode(kvq, torch, wl.views(), q)
    for b, h in picks:
        K, V = kv_ref[(b, h // cfg.group)]
        qh = q[b, h].astype(np.float64)
        extra = None
        if any(t.k_format == "codebook_qjl" for t in cfg.tiers):
            q_rot = orot.rotate(qh, ks_all[h // cfg.group])
            extra = np.concatenate([np.zeros(e) if isinstance(e, int) else
                                    ocache.qjl_correction(e[0], e[1], q_rot, proj, cfg.head_dim,
                                                          cfg.tiers[t].k_bits)
                                    for t, e in enumerate(sketch_rows[(b, h // cfg.group)])])
        want = oatt.attend(qh, K, V, extra)
        err = np.abs(got[b, h] - want).max()
        print(f"{name} b={b} h={h}: max-abs {err:.3e} (|out| max {np.abs(want).max():.2f})")
        assert err <= gu.ATOL_OUT


@pytest.mark.gpu
@pytest.mark.parametrize("group,kb,vb,width", [(8, 4, 4, 65536), (8, 3, 2, 131072), (4, 3, 2, 131072)])
def test_codebook_large_cache_instances(group, kb, vb, width):
    """The 16-warp tensor-core codebook instances, which the library picks for caches of 512 MB
    and more (sized by the block table's width), on short sequences: a block table `width`
    pages wide whose unused entries name page 0, 4096-token splits.  Eight query heads per kv
    head run as two 4-head items a chunk there too."""
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    hkv = 2
    cfg = W.CONFIGS["llama7b"].scaled(batch=2, num_q_heads=hkv * group, num_kv_heads=hkv,
                                      tiers=(W.Tier("codebook", "codebook", kb, vb),))
    lens = [3000, 1700]
    _, want, built, q = run_exact(cfg, lens)
    views = []
    for v in built.views:
        bt = torch.zeros((len(lens), width), dtype=torch.int32, device="cuda")
        bt[:, :v.block_table.shape[1]] = v.block_table
        views.append(kvq.TierView(v.cache, bt, v.seq_lens))
    got = gu.gpu_decode(kvq, torch, views, q, split_tokens=4096)
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())
