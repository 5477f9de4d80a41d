"""Host logic of the benchmark that needs no GPU: the clock record kept beside every
number (samples of nvidia-smi inside the timed region only, median SM clock, the throttle
reasons that were active), the layer reshaping options and the traffic record's guard."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _stamp(t):
    return time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".%03d" % int(round((t % 1) * 1000) % 1000)


def _line(t, mhz, reasons=()):
    flags = ["Active" if n in reasons else "Not Active" for n in bench.REASON_NAMES]
    return ", ".join([_stamp(t), "0", str(mhz), "2070", "900.00", "0x0"] + flags)


def test_clock_samples_inside_the_timed_region_only():
    t = 1_800_000_000.25
    lines = [_line(t - 2.0, 300, ("hw_slowdown",)),  # before the region: idle clock, a slowdown
             _line(t + 0.1, 2070), _line(t + 0.2, 2060, ("sw_power_cap",)), _line(t + 0.3, 2070),
             _line(t + 3.0, 1200, ("sw_thermal_slowdown",)),  # after it
             "garbage, line", ""]
    got = bench.parse_clock_samples(lines, t, t + 1.0)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    every = bench.parse_clock_samples(lines)
    assert every["samples"] == 5 and every["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert bench.parse_clock_samples(lines, t + 5, t + 6)["samples"] == 0


def test_layer_reshaping_keeps_the_workload_and_changes_only_its_shape():
    """--head-dim / --num-kv-heads reshape a workload (to time the shapes the fused kernels
    leave to the generic one); every other field and the per-rank seeds stay as they were."""
    base = bench.rank_config("llama7b", 0)
    d64 = bench.rank_config("llama7b", 0, head_dim=64)
    g8 = bench.rank_config("llama7b", 0, num_kv_heads=4)
    assert (d64.head_dim, d64.num_q_heads, d64.num_kv_heads) == (64, base.num_q_heads, base.num_kv_heads)
    assert (g8.head_dim, g8.num_q_heads, g8.num_kv_heads) == (base.head_dim, 32, 4) and g8.group == 8
    assert d64.seed == base.seed and d64.tiers == base.tiers and d64.seq_len == base.seq_len
    assert bench.rank_config("llama7b", 1, num_kv_heads=4).seed == base.seed + 1000


def test_kernel_traffic_only_for_the_captured_source_and_batch():
    """The DRAM traffic of the dominant kernel is reported only for the batch it was captured
    at (its split-K partial writes do not grow with the batch) and only while the kernel
    source is the captured one."""
    t = bench.TRAFFIC["gqa32k"]
    assert bench.kernel_traffic("gqa32k", t["captured_batch"]) in (None, t["bytes"])
    assert bench.kernel_traffic("gqa32k", t["captured_batch"] // 2) is None
    assert bench.kernel_traffic("llama7b", 8) is None


def test_quality_sample_covers_every_kv_head_whatever_the_batch():
    """The quality record samples the first and last query head of every kv head in the first
    and last sequence, so the kv heads with outlier channels are always in it, and it splits
    the error between kv heads with and without them."""
    import types
    import numpy as np
    import workloads as W
    from oracle.attention import attend

    for batch in (1, 4, 32):
        cfg = W.CONFIGS["gqa32k"].scaled(batch=batch)
        pairs = bench.quality_pairs(cfg)
        assert {h // cfg.group for _, h in pairs} == set(range(cfg.num_kv_heads))
        assert {b for b, _ in pairs} == {0, batch - 1}
        assert len(pairs) == len(set(pairs)) == len({0, batch - 1}) * cfg.num_kv_heads * 2

    cfg = W.CONFIGS["gqa32k"].scaled(batch=2, seq_len=96)
    wl = types.SimpleNamespace(lens=W.seq_lens(cfg))
    q = W.queries(cfg)
    k_new = np.stack([[W.kv_head(cfg, 0, b, g, 1, stream=7)[0] for g in range(cfg.num_kv_heads)]
                      for b in range(cfg.batch)])
    v_new = np.stack([[W.kv_head(cfg, 1, b, g, 1, stream=7)[0] for g in range(cfg.num_kv_heads)]
                      for b in range(cfg.batch)])
    out = np.zeros((cfg.batch, cfg.num_q_heads, cfg.head_dim))
    for b in range(cfg.batch):  # exact attention over the fp16 cache with the step's token in place
        for g in range(cfg.num_kv_heads):
            n = int(wl.lens[b])
            k = W.kv_head(cfg, 0, b, g, n).astype(np.float64)
            v = W.kv_head(cfg, 1, b, g, n).astype(np.float64)
            i = W.tier_members(cfg, b, g, n)[-1][-1]
            k[i], v[i] = k_new[b, g], v_new[b, g]
            for h in range(g * cfg.group, (g + 1) * cfg.group):
                out[b, h] = attend(q[b, h].astype(np.float64), k, v)
    got = bench.output_error_vs_fp16(cfg, wl, q, out, k_new, v_new, window=False)
    assert got["rel_err_vs_fp16_cache"]["max"] < 1e-12 and got["cosine_vs_fp16_cache"]["min"] > 1 - 1e-12
    with_out = {g for g in range(cfg.num_kv_heads) if (W.outlier_multipliers(cfg)[g] != 1).any()}
    assert 0 < len(with_out) < cfg.num_kv_heads
    assert got["kv_heads_with_outlier_channels"]["pairs"] == 2 * 2 * len(with_out)
    assert got["kv_heads_without_outlier_channels"]["pairs"] == 2 * 2 * (cfg.num_kv_heads - len(with_out))

    # a wrong output on one kv head with outlier channels shows in that bucket only
    g = min(with_out)
    bad = out.copy()
    bad[0, g * cfg.group] *= -1.0
    got = bench.output_error_vs_fp16(cfg, wl, q, bad, k_new, v_new, window=False)
    assert abs(got["kv_heads_with_outlier_channels"]["cosine_min"] + 1.0) < 1e-9
    assert got["kv_heads_without_outlier_channels"]["cosine_min"] > 1 - 1e-12
