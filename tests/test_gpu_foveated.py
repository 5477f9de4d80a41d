"""GPU parity of the FoveatedKV kernel features (FoveatedKV page, "Making it fast") through
kvq_decode_attention_ex, on every decode kernel family: the fused fp16 / fp8 + INT4 kernel,
the codebook kernel (one query head per kv head, and the tensor-core path for 2 and 4),
keys with a residual sketch or an outlier stream, and the generic kernel.

Spike flags: caches built so that, per (sequence, query head), the near tier's scores sit
well above or well below the far tier's (margins of several nats), so the float32
decision must equal the oracle's.  Score gate: a sink token at position 0 scores ~20 and a
crowd of tokens ~17 nats below it; the output must lie within the oracle's bound of both
the exact and the gated result, and differ from the ungated output (something was
skipped)."""
import numpy as np
import pytest

import workloads as W
from oracle import attention as oatt
from tests import gpu_util as gu

D = 128

# (name, tiers, group): which kernel family the call lands on
PATHS = {
    "fused_fp16_fp8": ((W.Tier("fp16", "fp16"), W.Tier("fp8_e4m3", "int4_g32")), 4),
    "codebook_g1": ((W.Tier("codebook", "codebook", 4, 4), W.Tier("codebook", "codebook", 2, 2)), 1),
    "codebook_g4": ((W.Tier("codebook", "codebook", 4, 4), W.Tier("codebook", "codebook", 3, 2)), 4),
    "sketched_g2": ((W.Tier("codebook_qjl", "codebook", 3, 4), W.Tier("codebook", "codebook", 2, 2)), 2),
    "generic_g2": ((W.Tier("fp16", "fp16"), W.Tier("codebook", "codebook", 4, 4)), 2),
    "outlier_g1": ((W.Tier("codebook_outlier", "codebook", 4, 4), W.Tier("codebook", "codebook", 2, 2)), 1),
    "outlier_g4": ((W.Tier("codebook_outlier", "codebook", 3, 2), W.Tier("fp8_e4m3", "int4_g32")), 4),
}
# any valid channel list serves exact-bytes parity (oracle and kernel read the same one)
OUTLIER_LIST = np.tile(np.array([0, 5, 17, 40, 64, 99, 100, 127], dtype=np.int32), (2, 1))


def decode_ex(kvq, torch, views, q16, split_tokens=0, score_gate=False, spikes=False):
    q = torch.from_numpy(q16).cuda()
    b, hq, d = q16.shape
    out_buf, out = gu.guarded_empty(torch, (b, hq, d), torch.float32)
    ws_buf, ws = gu.guarded_empty(torch, (max(1, kvq.kvq_decode_workspace_size(views, b, hq, split_tokens)),),
                                  torch.uint8)
    flags = torch.full((b, hq), -1, dtype=torch.int32, device="cuda") if spikes else None
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvq.kvq_decode_attention(views, q, out, ws, split_tokens, score_gate=score_gate, spike_flags=flags,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gu.assert_guards(out_buf, out)
    gu.assert_guards(ws_buf, ws)
    return out.cpu().numpy(), (flags.cpu().numpy() if spikes else None)


def unit(rng, n):
    u = rng.standard_normal((n, D))
    return u / np.linalg.norm(u, axis=-1, keepdims=True)


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(PATHS))
def test_spike_flags(name):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    tiers, group = PATHS[name]
    hkv, rng = 2, np.random.default_rng(17)
    hq = hkv * group
    near_len, far_len = [10, 0, 40, 7, 33], [100, 50, 0, 300, 1]
    u = unit(rng, hkv)  # one direction per kv head
    kv = [[], []]
    for nl, fl in zip(near_len, far_len):
        kn = rng.standard_normal((nl, hkv, D)) + 3.0 * np.sqrt(D) * u[None]  # near: large along u
        kf = rng.standard_normal((fl, hkv, D))
        kv[0].append((kn.astype(np.float16), rng.standard_normal((nl, hkv, D)).astype(np.float16)))
        kv[1].append((kf.astype(np.float16), rng.standard_normal((fl, hkv, D)).astype(np.float16)))
    sign = np.where(rng.random((len(near_len), hq)) < 0.5, -1.0, 1.0)
    q16 = (4.0 * sign[..., None] * u[np.arange(hq) // group][None]).astype(np.float16)
    cfg = W.CONFIGS["llama7b"].scaled(num_q_heads=hq, num_kv_heads=hkv)
    built = gu.build_exact(kvq, torch, list(tiers), kv, W.signs(cfg, 0), W.signs(cfg, 1), 16, 3,
                           k_qjl=W.qjl_projection(cfg), k_outl=OUTLIER_LIST)
    got, flags = decode_ex(kvq, torch, built.views, q16, split_tokens=32, spikes=True)
    want_flags, margin = oatt.spike_flags(q16, built.ora)
    defined = ~np.isnan(margin)
    assert np.all(np.abs(margin[defined]) > 1.0)  # decisions far from a tie
    assert np.array_equal(flags, want_flags), (flags, want_flags)
    assert flags[defined].min() == 0 and flags[defined].max() == 1  # both outcomes occur
    want = oatt.decode_attention(q16, built.ora)
    assert np.abs(got - want).max() <= 1e-4 * max(1.0, np.abs(want).max())


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(PATHS))
def test_score_gate_within_bound(name):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    tiers, group = PATHS[name]
    hkv, rng = 2, np.random.default_rng(23)
    hq = hkv * group
    lens = [700, 1100, 257]
    u = unit(rng, hkv)
    kv = [[] for _ in tiers]
    for n in lens:
        for t in range(len(tiers)):
            m = n // 4 if t == 0 else n - n // 4
            a = np.full((m, hkv), 3.0)  # 17 nats below the sink: gated
            a[: m // 3] = rng.normal(0.0, 1.0, (m // 3, hkv))  # far below: gated, negligible
            a[m // 3: m // 3 + 5] = 12.0  # inside the window: kept
            if t == 0:
                a[0] = 20.0  # the sink token, first of the sequence's first tier
            k = rng.standard_normal((m, hkv, D)) * 0.2 + a[..., None] * u[None]
            v = 1.0 + 0.1 * rng.standard_normal((m, hkv, D))  # the crowd's values add up
            kv[t].append((k.astype(np.float16), v.astype(np.float16)))
    q16 = np.ascontiguousarray(np.broadcast_to((np.sqrt(D) * u[np.arange(hq) // group])[None], (len(lens), hq, D)),
                               dtype=np.float16)
    cfg = W.CONFIGS["llama7b"].scaled(num_q_heads=hq, num_kv_heads=hkv)
    built = gu.build_exact(kvq, torch, list(tiers), kv, W.signs(cfg, 0), W.signs(cfg, 1), 16, None,
                           k_qjl=W.qjl_projection(cfg), k_outl=OUTLIER_LIST)
    split = 1024  # one chunk per tier and sequence: the sink sets the running maximum early
    gated_gpu, _ = decode_ex(kvq, torch, built.views, q16, split, score_gate=True)
    plain_gpu, _ = decode_ex(kvq, torch, built.views, q16, split)
    gated, exact, bound = oatt.gated_attention(q16, built.ora)
    tol = 1e-4 * max(1.0, np.abs(exact).max())
    assert np.abs(plain_gpu - exact).max() <= tol
    assert np.all(np.abs(gated_gpu - exact) <= bound + tol)
    assert np.all(np.abs(gated_gpu - gated) <= bound + tol)
    assert bound.max() > 1e-5  # the crowd below the gate carries visible weight
    assert np.abs(gated_gpu - plain_gpu).max() > 1e-6  # and the kernel did leave it out
