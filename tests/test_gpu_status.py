"""The decode call's device error report (kvq_decode_options.status) on the GPU.

* A valid call reports 0 on every kernel family, and leaves the guard bands around its
  output and workspace untouched.
* The codebook kernel's bounded wait for its own bulk copies: a TEST-ONLY build of the
  library (``build(variant="spintest")``) polls a slot twice with the non-blocking
  test_wait before giving up, so on valid data the give-up path runs: the call must report
  KVQ_DEVERR_COPY_TIMEOUT, return normally and leave finite outputs (the abandoned work items
  contribute nothing), and the production library must keep working afterwards.
* Queries that are 4-byte but not 16-byte aligned move tiers to other kernel families and
  another split plan; a workspace of kvq_decode_workspace_size() bytes must still do.
Out-of-range lengths and block-table entries are not fed to a GPU: the index checks that
handle them are exercised on the host (tests/test_index_checks.py)."""
import ctypes

import numpy as np
import pytest

import workloads as W
from oracle import attention as oatt
from tests import gpu_util as gu

FAMILIES = {
    "fused_fp16_fp8_g4": ((W.Tier("fp16", "fp16"), W.Tier("fp8_e4m3", "int4_g32")), 4, 128),
    "fused_fp16_fp8_g8": ((W.Tier("fp16", "fp16"), W.Tier("fp8_e4m3", "int4_g32")), 8, 128),
    "codebook_g1": ((W.Tier("codebook", "codebook", 4, 4),), 1, 128),
    "codebook_g1_d256": ((W.Tier("codebook", "codebook", 4, 4),), 1, 256),
    "codebook_g4": ((W.Tier("codebook", "codebook", 3, 2),), 4, 128),
    "codebook_g8": ((W.Tier("codebook", "codebook", 4, 4),), 8, 128),
    "generic_d64": ((W.Tier("fp16", "fp16"), W.Tier("fp8_e4m3", "int4_g32")), 2, 64),
    "generic_d64_codebook": ((W.Tier("codebook", "codebook", 4, 4),), 8, 64),
}


def _cache(kvq, torch, tiers, group, d, lens, seed=3):
    hkv = 2
    rng = np.random.default_rng(seed)
    ks = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    vs = np.where(rng.integers(0, 2, (hkv, d)) == 0, 1, -1).astype(np.int8)
    tier_kv = [[(rng.standard_normal((n, hkv, d)).astype(np.float16), rng.standard_normal((n, hkv, d)).astype(np.float16))
                for n in lens] for _ in tiers]
    built = gu.build_exact(kvq, torch, list(tiers), tier_kv, ks, vs, shuffle_seed=seed)
    q = rng.standard_normal((len(lens), hkv * group, d)).astype(np.float16)
    return built, q


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(FAMILIES))
def test_valid_call_reports_no_error_and_keeps_guards(name):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    tiers, group, d = FAMILIES[name]
    lens = [700, 33, 0, 129]
    built, q16 = _cache(kvq, torch, tiers, group, d, lens)
    b, hq, _ = q16.shape
    q = torch.from_numpy(q16).cuda()
    out_buf, out = gu.guarded_empty(torch, (b, hq, d), torch.float32)
    ws_buf, ws = gu.guarded_empty(torch, (max(1, kvq.kvq_decode_workspace_size(built.views, b, hq)),), torch.uint8)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvq.kvq_decode_attention(built.views, q, out, ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gu.assert_guards(out_buf, out)
    gu.assert_guards(ws_buf, ws)
    want = oatt.decode_attention(q16, built.ora)
    assert float(np.abs(out.cpu().numpy() - want).max()) <= gu.ATOL_OUT


@pytest.mark.gpu
def test_misaligned_queries_fit_the_reported_workspace():
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    tiers, group, d = FAMILIES["fused_fp16_fp8_g4"]
    lens = [2100, 999, 16]
    built, q16 = _cache(kvq, torch, tiers, group, d, lens, seed=5)
    b, hq, _ = q16.shape
    base = torch.zeros(q16.size + 8, dtype=torch.float16, device="cuda")
    q = base[2:2 + q16.size].view(q16.shape)  # 4 bytes past a 16-byte boundary
    q.copy_(torch.from_numpy(q16))
    assert q.data_ptr() % 16 == 4
    need = kvq.kvq_decode_workspace_size(built.views, b, hq)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")  # exactly the reported size
    out = torch.empty((b, hq, d), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_attention(built.views, q, out, ws)
    torch.cuda.synchronize()
    want = oatt.decode_attention(q16, built.ora)
    assert float(np.abs(out.cpu().numpy() - want).max()) <= gu.ATOL_OUT


def _spintest_lib(kvq):
    from quantized_decode_attention_rht_gb300 import build
    path = build.build(variant="spintest")
    lib = ctypes.CDLL(path)
    i32, vp, sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    lib.kvq_decode_attention_ex.argtypes = [ctypes.POINTER(kvq.KvqTierView), i32, vp, i32, i32, i32, vp, vp, sz,
                                            ctypes.POINTER(kvq.KvqDecodeOptions), vp]
    lib.kvq_decode_attention_ex.restype = ctypes.c_int
    return lib


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["codebook_g1", "codebook_g1_d256", "codebook_g4", "codebook_g8"])
def test_copy_wait_give_up_is_reported(name):
    torch = gu.torch_cuda()
    kvq = gu.kvq_module()
    spin = _spintest_lib(kvq)
    tiers, group, d = FAMILIES[name]
    lens = [3000, 1700, 64, 1]
    built, q16 = _cache(kvq, torch, tiers, group, d, lens, seed=9)
    b, hq, _ = q16.shape
    q = torch.from_numpy(q16).cuda()
    out = torch.full((b, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_decode_workspace_size(built.views, b, hq), dtype=torch.uint8, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    arr = kvq._views(built.views)
    opts = kvq.KvqDecodeOptions(0, None, status.data_ptr())
    st = spin.kvq_decode_attention_ex(arr, len(built.views), q.data_ptr(), b, hq, 0, out.data_ptr(), ws.data_ptr(),
                                      ws.numel(), ctypes.byref(opts), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    assert int(status.item()) & kvq.DEVERR_COPY_TIMEOUT
    assert torch.isfinite(out).all().item()  # abandoned items contribute nothing, nothing stale is read
    # the production library on the same inputs: no error, the oracle's result
    status.fill_(-1)
    kvq.kvq_decode_attention(built.views, q, out, ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = oatt.decode_attention(q16, built.ora)
    assert float(np.abs(out.cpu().numpy() - want).max()) <= gu.ATOL_OUT
