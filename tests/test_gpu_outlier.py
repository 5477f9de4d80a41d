"""GPU parity of the outlier two-stream cache (VeloxQuant-MLX page, "Outlier Two-Stream
Cache"): calibration (kvq_outlier_calibrate), keys appended with an outlier stream
(inlier codes + int8 outlier channels with a per-token scale) and decode over them on the
codebook kernel (one query head per kv head and the tensor-core path, head_dim 128 and
256).  Decode inputs are exact bytes written by the oracle; the channel list comes from
the oracle's calibration of the same data."""
import numpy as np
import pytest

import workloads as W
from oracle import attention as oatt
from oracle import cache as ocache
from tests import gpu_util as gu
from tests.test_gpu_quantize import make_inputs


@pytest.mark.gpu
@pytest.mark.parametrize("d", [128, 256])
def test_calibrate_matches_oracle(d):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    rng = np.random.default_rng(d)
    n, hkv = 300, 4
    x = rng.standard_normal((n, hkv, d)) * rng.uniform(0.2, 3.0, (1, hkv, d))
    x[:, 0, [5, 77, 100]] *= 20  # planted outlier channels
    x[:, 3, :] = 0.0
    x[:, 3, [3, 9]] = np.where(np.arange(n) % 2, 1.0, -1.0)[:, None]  # a tie, then zero variances
    x16 = x.astype(np.float16)
    out = torch.full((hkv, 8), -1, dtype=torch.int32, device="cuda")
    kvq.kvq_outlier_calibrate(torch.from_numpy(x16).cuda(), out)
    torch.cuda.synchronize()
    want = ocache.outlier_channels(x16)
    assert np.array_equal(out.cpu().numpy(), want)
    assert set(want[0][:3]) == {5, 77, 100} and want[3].tolist() == [3, 9, 0, 1, 2, 4, 5, 6]


@pytest.mark.gpu
@pytest.mark.parametrize("n", [203, 5600])
@pytest.mark.parametrize("d,bits", [(128, 2), (128, 3), (128, 4), (256, 4)])
def test_quantize_outlier_keys(d, bits, n):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    hkv, ps = 3, 16
    rng = np.random.default_rng(d * 3 + bits)
    k = make_inputs(n, hkv, d, d + bits)
    v = make_inputs(n, hkv, d, d + bits + 1)
    ks = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    vs = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    chans = ocache.outlier_channels(k[:64])
    num_pages = (n + ps - 1) // ps + 3
    slots = rng.permutation(num_pages * ps)[:n].astype(np.int32)
    slots[7] = -1
    cache = kvq.PagedCache(d, hkv, num_pages, "codebook_outlier", "codebook", bits, bits, ks, vs, ps,
                           k_outliers=chans)
    cache.append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    keep = np.flatnonzero(slots >= 0)
    assert cache.k_aux.shape[-1] == 12 and cache.k_rows.shape[-1] == d * bits // 8
    rows = gu.pool_rows(cache.k_rows, slots[keep])
    aux = gu.pool_rows(cache.k_aux, slots[keep])
    vrows = gu.pool_rows(cache.v_rows, slots[keep])
    vaux = gu.pool_rows(cache.v_aux, slots[keep])
    for h in range(hkv):
        gu.check_outlier_rows(k[keep, h], ks[h], bits, chans[h], rows[:, h], aux[:, h])
        gu.check_codebook_codes(v[keep, h], vs[h], bits, vrows[:, h], vaux[:, h, 0])


OUTLIER_CASES = [(128, 1, 4, 4), (128, 1, 3, 2), (128, 2, 2, 3), (128, 4, 4, 4), (256, 1, 4, 4), (256, 4, 3, 3)]


@pytest.mark.gpu
@pytest.mark.parametrize("d,group,kb,vb", OUTLIER_CASES)
def test_decode_outlier_keys(d, group, kb, vb):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    hkv = 2
    cfg = W.CONFIGS["llama7b"].scaled(batch=4, num_q_heads=hkv * group, num_kv_heads=hkv, head_dim=d,
                                      tiers=(W.Tier("codebook_outlier", "codebook", kb, vb),))
    lens = [1, 47, 300, 129]
    per_seq = [W.sequence_tiers(cfg, b, n) for b, n in enumerate(lens)]
    kv = [[per_seq[b][0] for b in range(len(lens))]]
    chans = ocache.outlier_channels(kv[0][2][0][:64])  # calibrated on a sequence's first tokens
    built = gu.build_exact(kvq, torch, list(cfg.tiers), kv, W.signs(cfg, 0), W.signs(cfg, 1), cfg.page_size, 5,
                           k_outl=chans)
    q = W.queries(cfg)
    got = gu.gpu_decode(kvq, torch, built.views, q, 96)
    want = oatt.decode_attention(q, built.ora)
    assert np.all(np.isfinite(got))
    err = np.abs(got - want).max()
    assert err <= 1e-4 * max(1.0, np.abs(want).max())
    # the outlier stream matters: dropping it moves the output far past the error
    plain_tiers = []
    for t in built.ora:
        k_side = ocache.Side("codebook", t.k.bits, t.k.centroids32, t.k.bounds32, t.k.signs, t.k.rows,
                             ocache.unpack_outlier_aux(t.k.aux)[0], None, None)
        plain_tiers.append(oatt.TierState(k_side, t.v, t.block_table, t.lens, t.page_size))
    assert np.abs(oatt.decode_attention(q, plain_tiers) - want).max() > 100 * max(err, 1e-6)
