"""Host logic of the seeded workloads: tier membership, including the recent-token window
(the newest min(W, L) tokens of every sequence; AdapTQ page, "Hybrid Execution": a short
context stays entirely unquantised)."""
import numpy as np

import workloads as W


def test_window_holds_the_newest_tokens():
    cfg = W.CONFIGS["llama7b_window"]
    for total in (0, 1, 100, 256, 257, 8192):
        lens = W.tier_lens(cfg, total)
        members = W.tier_members(cfg, 0, 3, total)
        assert sum(lens) == total and [len(m) for m in members] == lens
        w = min(256, total)
        assert lens[-1] == w
        assert np.array_equal(members[-1], np.arange(total - w, total))
        assert np.array_equal(np.sort(np.concatenate(members)), np.arange(total))


def test_short_context_is_all_window():
    cfg = W.CONFIGS["llama7b_window"]
    assert W.tier_lens(cfg, 200) == [0, 200]


def test_fraction_tiers_unchanged():
    cfg = W.CONFIGS["gqa32k"]
    for total in (0, 9, 10, 1234, 32768):
        lens = W.tier_lens(cfg, total)
        assert lens[0] == min(total, int(round(0.1 * total))) and sum(lens) == total
        members = W.tier_members(cfg, 1, 2, total)
        assert np.array_equal(np.sort(np.concatenate(members)), np.arange(total))
