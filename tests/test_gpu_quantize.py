"""GPU parity of kvq_quantize_append against the oracle's encoder, row by row.

Inputs: ragged token counts, random (shuffled) pool slots with skipped (-1) and out-of-range
slots, Gaussian K/V with planted x30 outlier channels, plus degenerate vectors (zero,
one-hot, constant, values beyond the fp8 range)."""
import numpy as np
import pytest

from tests import gpu_util as gu

# rows 0..4 of make_inputs are degenerate on purpose (zero, one-hot, constant, huge, tiny):
# their codes are checked, but they sit exactly on boundaries and are left out of the
# boundary-fraction statistic, which describes workload-like data
DEGENERATE = 5

FORMATS = [("codebook", 2), ("codebook", 3), ("codebook", 4), ("fp16", 0), ("fp8_e4m3", 0), ("int4_g32", 0)]


def make_inputs(n, hkv, d, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, hkv, d)).astype(np.float32)
    ch = rng.choice(d, 3, replace=False)
    x[:, :, ch] *= 30
    x[0] = 0.0  # zero vector
    x[1] = 0.0
    x[1, :, 5] = 7.0  # one-hot
    x[2] = 1.5  # constant: the rotation puts everything in one coordinate
    x[3] = rng.standard_normal((hkv, d)) * 900  # rotated values beyond fp8's 448
    x[4] = rng.standard_normal((hkv, d)) * 1e-3  # tiny values (fp16 subnormals after rotation)
    return x.astype(np.float16)


def run_append(kvq, torch, fmt, bits, d, n=203, hkv=3, ps=16, seed=0, codebook="lloyd_max", k_only=False,
               v_fmt=None, k_qjl=None):
    rng = np.random.default_rng(seed + 100)
    k = make_inputs(n, hkv, d, seed)
    v = make_inputs(n, hkv, d, seed + 1)
    ks = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    vs = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    num_pages = (n + ps - 1) // ps + 3
    slots = rng.permutation(num_pages * ps)[:n].astype(np.int32)
    slots[7] = -1  # skipped
    slots[11] = num_pages * ps + 5  # out of range: skipped
    cache = kvq.PagedCache(d, hkv, num_pages, fmt, v_fmt or fmt, bits, bits, ks, vs, ps, codebook, k_qjl=k_qjl)
    cache.append(torch.from_numpy(k).cuda(), None if k_only else torch.from_numpy(v).cuda(),
                 torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    return k, v, ks, vs, slots, cache


# The library takes appends of at most 16384 vectors per side with one warp per vector
# (decode steps) and larger ones with the per-thread kernel (prefill chunks): 203 tokens x 3
# heads and 5600 x 3 cover both.
SIZES = [203, 5600]


@pytest.mark.gpu
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("fmt,bits", FORMATS)
def test_quantize_matches_oracle(fmt, bits, d, n):
    check_append(fmt, bits, d, n, 16)


@pytest.mark.gpu
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("fmt,bits,d,ps", [("codebook", 4, 128, 1), ("codebook", 3, 256, 12), ("int4_g32", 0, 128, 24),
                                           ("codebook", 2, 64, 32), ("fp8_e4m3", 0, 128, 7)])
def test_quantize_page_sizes(fmt, bits, d, ps, n):
    """Pools with pages of other sizes than 16 tokens: powers of two (the kernels shift the
    slot) and others (they divide it), on both append kernels."""
    check_append(fmt, bits, d, n, ps)


def check_append(fmt, bits, d, n, ps):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    k, v, ks, vs, slots, cache = run_append(kvq, torch, fmt, bits, d, n=n, ps=ps, seed=d + bits)
    keep = np.flatnonzero((slots >= 0) & (slots < cache.num_pages * cache.page_size))
    assert np.all(keep[:DEGENERATE] == np.arange(DEGENERATE))
    stats = []
    for x, signs, rows_t, aux_t in ((k, ks, cache.k_rows, cache.k_aux), (v, vs, cache.v_rows, cache.v_aux)):
        rows = gu.pool_rows(rows_t, slots[keep])
        aux = None if aux_t is None else gu.pool_rows(aux_t, slots[keep])
        for h in range(x.shape[1]):
            xh = x[keep, h]
            if fmt == "codebook":
                gu.check_codebook_codes(xh[:DEGENERATE], signs[h], bits, rows[:DEGENERATE, h],
                                        aux[:DEGENERATE, h, 0])
                stats.append(gu.check_codebook_codes(xh[DEGENERATE:], signs[h], bits, rows[DEGENERATE:, h],
                                                     aux[DEGENERATE:, h, 0]))
            elif fmt == "int4_g32":
                stats.append(gu.check_int4_rows(xh, signs[h], rows[:, h], aux[:, h]))
            else:
                stats.append(gu.check_float_rows(xh, signs[h], fmt, rows[:, h]))
    if fmt == "codebook":
        near = sum(s[1] for s in stats)
        total = sum(s[2] for s in stats)
        assert near < gu.MAX_BOUNDARY_FRACTION * total + 1, (near, total)
    # slots that were skipped stay zero
    used = np.zeros(cache.num_pages * cache.page_size, bool)
    used[slots[keep]] = True
    krows = cache.k_rows.cpu().numpy().reshape(cache.num_pages, -1, cache.page_size, cache.k_rows.shape[-1])
    unused = np.flatnonzero(~used)
    assert not krows[unused // cache.page_size, :, unused % cache.page_size].any()


@pytest.mark.gpu
@pytest.mark.parametrize("n", SIZES)
def test_quantize_uniform_codebook_and_k_only(n):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    k, v, ks, vs, slots, cache = run_append(kvq, torch, "codebook", 4, 128, n=n, seed=5, codebook="uniform",
                                            k_only=True)
    keep = np.flatnonzero((slots >= 0) & (slots < cache.num_pages * cache.page_size))
    rows = gu.pool_rows(cache.k_rows, slots[keep])
    aux = gu.pool_rows(cache.k_aux, slots[keep])
    for h in range(k.shape[1]):
        gu.check_codebook_codes(k[keep, h], ks[h], 4, rows[:, h], aux[:, h, 0], kind="uniform")
    assert not cache.v_rows.any().item()  # V untouched when only K is appended


@pytest.mark.gpu
def test_quantize_codes_on_a_large_sample():
    """North-star statistic on ~4M coordinates: differing codes only within 1e-6 of a
    boundary, and fewer than 1e-4 of the elements that close to one."""
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    import workloads as W
    cfg = W.CONFIGS["llama7b"]
    hkv, d, n = 8, 128, 2048
    x = np.stack([W.kv_head(cfg, 0, 0, h, n) for h in range(hkv)], axis=1)
    signs = W.signs(cfg, 0)[:hkv]
    ps = 16
    cache = kvq.PagedCache(d, hkv, n // ps, "codebook", "codebook", 4, 4, signs, signs, ps)
    slots = np.arange(n, dtype=np.int32)
    cache.append(torch.from_numpy(x).cuda(), None, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    rows = gu.pool_rows(cache.k_rows, slots)
    aux = gu.pool_rows(cache.k_aux, slots)
    bad = near = total = 0
    for h in range(hkv):
        b_, n_, t_, _ = gu.check_codebook_codes(x[:, h], signs[h], 4, rows[:, h], aux[:, h, 0])
        bad, near, total = bad + b_, near + n_, total + t_
    assert near < gu.MAX_BOUNDARY_FRACTION * total
    print(f"codes differing: {bad} of {total}; within 1e-6 of a boundary: {near}")


@pytest.mark.gpu
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("d,bits", [(128, 2), (128, 3), (128, 4), (256, 3)])
def test_quantize_qjl_keys_match_oracle(d, bits, n):
    """Keys with a residual sign sketch (codes, norm, residual norm, 128 sign bits) next to
    codebook values, on the degenerate and outlier rows of make_inputs."""
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    proj = np.random.default_rng(d * 7 + bits).standard_normal((128, d)).astype(np.float32)
    k, v, ks, vs, slots, cache = run_append(kvq, torch, "codebook_qjl", bits, d, n=n, seed=d + bits,
                                            v_fmt="codebook", k_qjl=proj)
    keep = np.flatnonzero((slots >= 0) & (slots < cache.num_pages * cache.page_size))
    assert cache.k_rows.shape[-1] == d * bits // 8 + 16 and cache.k_aux.shape[-1] == 2
    rows = gu.pool_rows(cache.k_rows, slots[keep])
    aux = gu.pool_rows(cache.k_aux, slots[keep])
    vrows = gu.pool_rows(cache.v_rows, slots[keep])
    vaux = gu.pool_rows(cache.v_aux, slots[keep])
    compared = bits_bad = rn_bad = 0
    for h in range(k.shape[1]):
        c, sb, rb = gu.check_qjl_rows(k[keep, h], ks[h], bits, proj, rows[:, h], aux[:, h])
        compared, bits_bad, rn_bad = compared + c, bits_bad + sb, rn_bad + rb
        gu.check_codebook_codes(v[keep, h], vs[h], bits, vrows[:, h], vaux[:, h, 0])
    assert compared >= 0.95 * len(keep) * k.shape[1]
    assert bits_bad <= 1e-3 * compared * 128 + 1
    # the zero vector: zero residual, every projection 0 -> every sign bit set
    z0 = rows[0, :, d * bits // 8:]
    assert np.all(z0 == 0xFF) and np.all(aux[0, :, 1] == 0)
    print(f"rows compared {compared}, sign bits differing {bits_bad}, residual norms differing {rn_bad}")
