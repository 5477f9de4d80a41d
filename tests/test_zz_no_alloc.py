"""kvq_decode_attention_noalloc, the decode entry point for callers that may not allocate
device memory (plugins inside a framework that owns all device memory, serving loops with a
memory budget fixed at start-up): it uses the library's static device scratch instead of a
caller-provided workspace.  Its results must match kvq_decode_attention's on the same inputs,
on consecutive calls (the scratch keeps the previous call's contents)."""
import numpy as np
import pytest

import workloads as W
from tests import gpu_util as gu


def _two_tier_cache(kvq, torch, cfg, lens):
    ks, vs = W.signs(cfg, 0), W.signs(cfg, 1)
    ks_d, vs_d = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    per_seq = [W.sequence_tiers(cfg, b, n) for b, n in enumerate(lens)]
    views = []
    for t, tier in enumerate(cfg.tiers):
        tl = np.array([per_seq[b][t][0].shape[0] for b in range(len(lens))])
        pm = W.page_map(cfg, tl, tier=t)
        cache = kvq.PagedCache(cfg.head_dim, cfg.num_kv_heads, max(1, pm.num_pages), tier.k_format, tier.v_format,
                               tier.k_bits, tier.v_bits, ks_d, vs_d, cfg.page_size)
        for b in range(len(lens)):
            k, v = per_seq[b][t]
            slots = pm.slots(b, np.arange(k.shape[0]))
            cache.append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda())
        views.append(kvq.TierView(cache, torch.from_numpy(np.maximum(pm.block_table, 0)).cuda(),
                                  torch.from_numpy(tl.astype(np.int32)).cuda()))
    return views


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point():
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    lens = [2100, 999, 16]
    cfg = W.CONFIGS["gqa32k"].scaled(batch=len(lens), num_q_heads=8, num_kv_heads=2)
    views = _two_tier_cache(kvq, torch, cfg, lens)
    for step in range(2):  # two calls in a row, different queries
        q = torch.from_numpy(W.queries(cfg, step=step)).cuda()
        ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        ws = torch.empty(kvq.kvq_decode_workspace_size(views, len(lens), cfg.num_q_heads), dtype=torch.uint8,
                         device="cuda")
        kvq.kvq_decode_attention(views, q, ref, ws)
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        kvq.kvq_decode_attention_noalloc(views, q, out)
        torch.cuda.synchronize()
        err = (out - ref).abs().max().item()
        assert torch.isfinite(out).all().item()
        assert err <= gu.ATOL_OUT, err


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_its_scratch():
    """A shape whose split-K scratch exceeds the static array is refused before any launch.
    Every pointer handed over is a real allocation (a 4-page cache, a zeroed block table,
    zero lengths, real queries and outputs), so even a launch could read nothing invalid."""
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    ks = torch.ones((8, 128), dtype=torch.int8, device="cuda")
    cache = kvq.PagedCache(128, 8, 4, "codebook", "codebook", 4, 4, ks, ks)
    batch, hq, max_pages = 64, 32, 1 << 16  # 1M tokens in 1024-token splits: 1024 splits per
    # output, within the split limit but ~1 GB of partials, far more scratch than it has
    bt = torch.zeros((batch, max_pages), dtype=torch.int32, device="cuda")
    lens = torch.zeros(batch, dtype=torch.int32, device="cuda")
    q = torch.zeros((batch, hq, 128), dtype=torch.float16, device="cuda")
    out = torch.full((batch, hq, 128), 7.0, dtype=torch.float32, device="cuda")
    views = [kvq.TierView(cache, bt, lens)]
    assert kvq.kvq_decode_workspace_size(views, batch, hq, 1024) > kvq.NOALLOC_SCRATCH_BYTES
    launches = kvq.kvq_kernel_launches()
    st = kvq.lib().kvq_decode_attention_noalloc(kvq._views(views), 1, q.data_ptr(), batch, hq, 1024,
                                                out.data_ptr(), None)
    torch.cuda.synchronize()
    assert st == 3  # KVQ_ERR_WORKSPACE_TOO_SMALL
    assert kvq.kvq_kernel_launches() == launches  # nothing was launched
    assert (out == 7.0).all().item()  # nothing was written
