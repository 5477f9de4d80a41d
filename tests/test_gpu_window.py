"""GPU parity of the recent-token window (FoveatedKV page, "Making it fast": the unquantised
decode buffer in the same dispatch; AdapTQ page, "Hybrid Execution"): kvq_requantize moving
tokens out of an fp16 tier, and decode over a window tier next to quantised tiers (every
group size of the fused fp16 kernel, each tier on its own kernel family in one call).

Exact inputs: the oracle writes the window's fp16 rows; the same bytes are uploaded; the
GPU's re-encoded rows are checked against the oracle's re-encode of those rows (no
rotation error: the input is the stored x~ itself)."""
import numpy as np
import pytest

import workloads as W
from oracle import attention as oatt
from oracle import cache as ocache
from tests import gpu_util as gu

DEST = [("codebook", 2, "codebook", 2), ("codebook", 3, "codebook", 4), ("codebook", 4, "codebook", 4),
        ("codebook_qjl", 3, "codebook", 4), ("fp8_e4m3", 0, "int4_g32", 0), ("fp16", 0, "fp16", 0)]


def inputs(n, hkv, d, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, hkv, d)).astype(np.float32)
    x[:, :, rng.choice(d, 3, replace=False)] *= 30
    x[0] = 0.0
    x[1] = rng.standard_normal((hkv, d)) * 900
    return x.astype(np.float16)


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("kf,kb,vf,vb", DEST)
def test_requantize_matches_oracle(kf, kb, vf, vb, d):
    if kf == "codebook_qjl" and d == 64:
        pytest.skip("keys with a sketch need head_dim 128 or 256")
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    hkv, n, ps = 3, 150, 16
    rng = np.random.default_rng(d + kb)
    ks = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    vs = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    ks_d, vs_d = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    proj = rng.standard_normal((128, d)).astype(np.float32)
    k, v = inputs(n, hkv, d, d), inputs(n, hkv, d, d + 1)
    # the window, written by the oracle and uploaded byte for byte
    wpages = n // ps + 2
    wslots = rng.permutation(wpages * ps)[:n].astype(np.int32)
    win = kvq.PagedCache(d, hkv, wpages, "fp16", "fp16", 0, 0, ks_d, vs_d, ps)
    side_k = ocache.new_side("fp16", 0, None, None, ks, wpages, hkv, ps, d)
    side_v = ocache.new_side("fp16", 0, None, None, vs, wpages, hkv, ps, d)
    ocache.write(side_k, wslots, k, ps)
    ocache.write(side_v, wslots, v, ps)
    win.k_rows.copy_(torch.from_numpy(side_k.rows))
    win.v_rows.copy_(torch.from_numpy(side_v.rows))
    dpages = n // ps + 3
    dst = kvq.PagedCache(d, hkv, dpages, kf, vf, kb, vb, ks_d, vs_d, ps, k_qjl=proj if kf == "codebook_qjl" else None)
    dslots = rng.permutation(dpages * ps)[:n].astype(np.int32)
    src_slots = wslots.copy()
    src_slots[5] = -1  # skipped
    dslots[9] = dpages * ps + 1  # out of range: skipped
    kvq.kvq_requantize(win.struct, torch.from_numpy(src_slots).cuda(), dst.struct, torch.from_numpy(dslots).cuda())
    torch.cuda.synchronize()
    keep = np.setdiff1d(np.arange(n), [5, 9])
    for side, rows16, fmt, bits, rows_t, aux_t in (("k", side_k.rows, kf, kb, dst.k_rows, dst.k_aux),
                                                  ("v", side_v.rows, vf, vb, dst.v_rows, dst.v_aux)):
        rg = gu.pool_rows(rows_t, dslots[keep])
        ag = None if aux_t is None else gu.pool_rows(aux_t, dslots[keep])
        stored = rows16[wslots[keep] // ps, :, wslots[keep] % ps]  # [T, hkv, 2d] fp16 bytes of x~
        for h in range(hkv):
            xr = np.ascontiguousarray(stored[:, h]).view(np.float16).astype(np.float64)
            if fmt == "codebook":
                gu.check_codebook_codes(None, None, bits, rg[:, h], ag[:, h, 0], xr=xr)
            elif fmt == "codebook_qjl":
                gu.check_qjl_rows(None, None, bits, proj, rg[:, h], ag[:, h], xr=xr)
            elif fmt == "int4_g32":
                gu.check_int4_rows(None, None, rg[:, h], ag[:, h], xr=xr)
            else:
                bad, _ = gu.check_float_rows(None, None, fmt, rg[:, h], xr=xr)
                assert bad == 0  # exact input: the format's rounding of x~ itself
    # skipped tokens leave their destination rows untouched (zero)
    used = np.zeros(dpages * ps, bool)
    used[dslots[keep]] = True
    all_rows = dst.k_rows.cpu().numpy()
    free = np.flatnonzero(~used)
    assert not all_rows[free // ps, :, free % ps].any()


WINDOW_CASES = {
    # (tiers: main first, window last; group)
    "codebook_g1": ((W.Tier("codebook", "codebook", 4, 4), W.Tier("fp16", "fp16")), 1),
    "codebook_g2": ((W.Tier("codebook", "codebook", 3, 2), W.Tier("fp16", "fp16")), 2),
    "sketched_g4": ((W.Tier("codebook_qjl", "codebook", 3, 4), W.Tier("fp16", "fp16")), 4),
    "fp8_int4_g4": ((W.Tier("fp8_e4m3", "int4_g32"), W.Tier("fp16", "fp16")), 4),
    "fp8_int4_g1": ((W.Tier("fp8_e4m3", "int4_g32"), W.Tier("fp16", "fp16")), 1),
    "fp8_int4_g2": ((W.Tier("fp8_e4m3", "int4_g32"), W.Tier("fp16", "fp16")), 2),
    "three_tiers_g1": ((W.Tier("fp16", "fp16"), W.Tier("codebook", "codebook", 2, 2), W.Tier("fp16", "fp16")), 1),
    # head_dim 256: the window tier runs on the generic kernel next to the codebook one
    "codebook_d256_g2": ((W.Tier("codebook", "codebook", 4, 4), W.Tier("fp16", "fp16")), 2, 256),
    "outlier_d256_g1": ((W.Tier("codebook_outlier", "codebook", 3, 3), W.Tier("fp16", "fp16")), 1, 256),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(WINDOW_CASES))
def test_window_tier_decode(name):
    """A window tier (fp16, the newest min(L, 64) tokens) attended with quantised tiers in one
    call, each tier on its kernel family: exact bytes, oracle dequantise-then-attend."""
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    tiers, group, d = (WINDOW_CASES[name] + (128,))[:3]
    hkv = 2
    cfg = W.CONFIGS["llama7b"].scaled(batch=5, num_q_heads=hkv * group, num_kv_heads=hkv, tiers=tiers, head_dim=d)
    lens = [0, 40, 64, 65, 700]
    win = 64
    rng = np.random.default_rng(7)
    kv = [[] for _ in tiers]
    for b, n in enumerate(lens):
        kk = np.stack([W.kv_head(cfg, 0, b, h, n) for h in range(hkv)], axis=1).reshape(n, hkv, d)
        vv = np.stack([W.kv_head(cfg, 1, b, h, n) for h in range(hkv)], axis=1).reshape(n, hkv, d)
        body = n - min(n, win)  # the window holds the newest tokens; older ones are split
        inner = sorted(int(c) for c in rng.integers(0, body + 1, len(tiers) - 2))  # among the quantised tiers
        cuts = [0] + inner + [body, n]
        for t in range(len(tiers)):
            kv[t].append((kk[cuts[t]:cuts[t + 1]], vv[cuts[t]:cuts[t + 1]]))
    q = W.queries(cfg)
    chans = np.tile(np.arange(0, d, d // 8, dtype=np.int32), (hkv, 1))  # any valid outlier channel list
    built = gu.build_exact(kvq, torch, list(tiers), kv, W.signs(cfg, 0), W.signs(cfg, 1), 16, 4,
                           k_qjl=W.qjl_projection(cfg), k_outl=chans)
    got = gu.gpu_decode(kvq, torch, built.views, q)
    want = oatt.decode_attention(q, built.ora)
    assert np.all(got[0] == 0)
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


@pytest.mark.gpu
def test_fp8_encode_every_fp16_pattern():
    """The fp8 E4M3 encode (round to nearest even, saturating at +-448) on every one of the
    65,536 fp16 bit patterns, bit-exact against the oracle: the patterns are stored as the
    rows of an fp16 window tier and moved into an fp8-key tier with kvq_requantize, whose
    re-encode converts the stored value itself (no rotation in between).  NaN inputs must
    give a NaN code (0x7F or 0xFF, either sign)."""
    from oracle import formats as ofmt
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    d, hkv, ps = 128, 1, 16
    n = 65536 // d
    pages = n // ps
    pat = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ones = np.ones((hkv, d), dtype=np.int8)
    signs = torch.from_numpy(ones).cuda()
    win = kvq.PagedCache(d, hkv, pages, "fp16", "fp16", 0, 0, signs, signs, ps)
    win.k_rows.copy_(torch.from_numpy(pat.view(np.uint8).reshape(pages, hkv, ps, 2 * d)))
    win.v_rows.zero_()
    dst = kvq.PagedCache(d, hkv, pages, "fp8_e4m3", "fp16", 0, 0, signs, signs, ps)
    slots = torch.arange(n, dtype=torch.int32, device="cuda")
    kvq.kvq_requantize(win.struct, slots, dst.struct, slots)
    torch.cuda.synchronize()
    got = dst.k_rows.cpu().numpy().reshape(-1)
    with np.errstate(invalid="ignore"):  # NaN patterns
        vals = pat.view(np.float16).astype(np.float32)
        want = ofmt.e4m3_encode(vals)
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], want[~nan]), int(np.sum(got[~nan] != want[~nan]))
    assert np.all((got[nan] & 0x7F) == 0x7F)
    assert got[np.flatnonzero(vals == np.inf)[0]] == 0x7E and got[np.flatnonzero(vals == -np.inf)[0]] == 0xFE
