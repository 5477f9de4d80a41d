"""Helpers shared by the GPU parity tests: building the library, building oracle pools
and uploading them byte for byte, and the decision-boundary allowances.

The allowances follow from where the two sides may legitimately differ.  The oracle
rotates in float64 and takes every rounding decision on the exact value rounded to
float32; the kernel rotates in float32.  The kernel's Walsh-Hadamard result carries an
absolute error of at most (log2(D) + 2) * 2^-24 * sum|x| / sqrt(D) per coordinate (one
rounding per butterfly stage on partial sums bounded by sum|x|, plus the final scale), so
a stored value may differ from the oracle's only where the exact value lies within that
distance of a rounding boundary.  For codebook indices the criterion is the one fixed for
this method: a differing index is allowed only where the exact u is within 1e-6 of a
decision boundary, and such elements must be fewer than 1e-4 of all."""
from __future__ import annotations

import math

import numpy as np
import pytest

from oracle import attention as oatt
from oracle import cache as ocache
from oracle import codebook as ocb
from oracle import formats as ofmt
from oracle import rotation as orot

U_BOUNDARY = 1e-6
MAX_BOUNDARY_FRACTION = 1e-4
ATOL_OUT = 2e-3


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


_built = False


def kvq_module():
    global _built
    torch_cuda()
    import quantized_decode_attention_rht_gb300 as kvq
    if not _built:
        from quantized_decode_attention_rht_gb300 import build
        build.build()
        _built = True
    kvq.lib()
    return kvq


_TABLES = {}


def tables(kind, bits):
    if (kind, bits) not in _TABLES:
        _TABLES[(kind, bits)] = ocb.tables(kind, bits)
    return _TABLES[(kind, bits)]


def fwht_error_bound(x16: np.ndarray) -> np.ndarray:
    """Per-vector bound on the absolute error of the kernel's float32 rotated coordinates."""
    d = x16.shape[-1]
    return (math.log2(d) + 2) * 2.0 ** -24 * np.sum(np.abs(x16.astype(np.float64)), axis=-1) / math.sqrt(d)


def pool_rows(tensor, slots):
    """Rows of a device pool tensor [P, Hkv, ps, ...] at the given slots -> numpy [T, Hkv, ...]."""
    a = tensor.cpu().numpy()
    ps = a.shape[2]
    slots = np.asarray(slots)
    return a[slots // ps, :, slots % ps]


# ----------------------------------------------------------------------------- codes


def rotated(x16, signs, xr):
    """The exact rotated vectors: of x16 with signs, or xr as given (a re-encode of stored
    rows, whose input is already rotated)."""
    return orot.rotate(x16.astype(np.float64), signs) if xr is None else np.asarray(xr, dtype=np.float64)


def check_codebook_codes(x16, signs, bits, rows_gpu, norms_gpu, kind="lloyd_max", xr=None):
    """x16 [T, d] of one head, signs [d] (or xr: the exact rotated vectors); rows_gpu
    [T, row_bytes]; norms_gpu fp16 [T].  Returns (mismatches, near-boundary count, elements)."""
    c32, b32 = tables(kind, bits)
    xr = rotated(x16, signs, xr)
    d = xr.shape[-1]
    rows_o, norm_o = ocache.encode_rotated(xr, "codebook", bits, b32)
    idx_o = ofmt.unpack_bits(rows_o, bits, d)
    idx_g = ofmt.unpack_bits(rows_gpu, bits, d)
    n = np.sqrt(np.sum(xr * xr, axis=-1))
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(n[:, None] > 0, math.sqrt(d) * xr / n[:, None], 0.0)
    dist = np.min(np.abs(u[..., None] - b32.astype(np.float64)), axis=-1)
    near = dist < U_BOUNDARY
    bad = idx_o != idx_g
    assert not np.any(bad & ~near), f"{int(np.sum(bad & ~near))} codes differ away from a boundary"
    assert np.all(np.abs(idx_o - idx_g)[bad] == 1)
    # norms: equal, or one fp16 ulp apart where the exact norm sits on a rounding midpoint
    ng = np.asarray(norms_gpu, dtype=np.float16)
    diff = ng != norm_o
    if np.any(diff):
        a, b = ng[diff].astype(np.float64), norm_o[diff].astype(np.float64)
        assert np.all(np.abs(np.asarray(ng[diff]).view(np.uint16).astype(np.int64) -
                             np.asarray(norm_o[diff]).view(np.uint16).astype(np.int64)) == 1)
        mid = (a + b) / 2
        assert np.all(np.abs(n[diff] - mid) <= 1.2e-5 * n[diff]), "norm differs away from a midpoint"
    return int(np.sum(bad)), int(np.sum(near)), idx_o.size, int(np.sum(diff))


def check_qjl_rows(x16, signs, bits, proj, rows_gpu, aux_gpu, kind="lloyd_max", xr=None):
    """Keys with a residual sign sketch: x16 [T, d] of one head, proj float32 [m, d];
    rows_gpu [T, row_bytes]; aux_gpu fp16 [T, 2].

    The codes and the norm follow the codebook criteria.  Where both agree with the
    oracle, the residual is the same vector up to float32 rounding, so the residual norm
    may differ by at most one fp16 ulp and a sign bit only where |<S_j, r~>| lies within
    the float32 error of the kernel's residual and dot product:
    1e-5 * sum_i |S_ji| (|r~_i| + |x~_i|), far above (log2 d + 4) 2^-24 of that sum.
    Rows whose codes or norm differ carry a different residual and are checked only for
    their codes.  Returns (rows compared, sign bits differing, residual norms differing)."""
    c32, b32 = tables(kind, bits)
    xr = rotated(x16, signs, xr)
    d = xr.shape[-1]
    nb = d * bits // 8
    aux_gpu = np.asarray(aux_gpu, dtype=np.float16)
    check_codebook_codes(None, None, bits, rows_gpu[:, :nb], aux_gpu[:, 0], kind, xr=xr)
    rows_o, aux_o = ocache.encode_rotated(xr, "codebook_qjl", bits, b32, c32, proj)
    same = np.all(rows_gpu[:, :nb] == rows_o[:, :nb], axis=-1) & (aux_gpu[:, 0] == aux_o[:, 0])
    r = xr - ocache.decode_rotated(rows_o, aux_o, "codebook_qjl", d, bits, c32)
    s64 = np.asarray(proj, dtype=np.float32).astype(np.float64)
    sr = r @ s64.T
    tol = 1e-5 * (np.abs(r) + np.abs(xr)) @ np.abs(s64).T
    z_o = ofmt.unpack_bits(rows_o[:, nb:], 1, ocache.QJL_DIM)
    z_g = ofmt.unpack_bits(rows_gpu[:, nb:], 1, ocache.QJL_DIM)
    bad = (z_o != z_g) & same[:, None]
    assert not np.any(bad & (np.abs(sr) > tol)), "sign bits differ away from zero"
    ug = aux_gpu[:, 1].view(np.uint16).astype(np.int64)
    uo = np.asarray(aux_o[:, 1], dtype=np.float16).view(np.uint16).astype(np.int64)
    rdiff = (ug != uo) & same
    assert np.all(np.abs(ug - uo)[rdiff] == 1), "residual norms differ by more than one fp16 ulp"
    return int(np.sum(same)), int(np.sum(bad)), int(np.sum(rdiff))


def check_outlier_rows(x16, signs, bits, channels, rows_gpu, aux_gpu, kind="lloyd_max"):
    """Keys with an outlier stream: x16 [T, d] of one head, channels [K].  The inlier codes
    and norm follow the codebook criteria on the rotated inlier vector (outlier channels
    zeroed); the outlier scale and the int8 values must equal the oracle's exactly (both
    come from exact fp16 inputs through one float32 division and one rounding each)."""
    c32, b32 = tables(kind, bits)
    x_in = np.array(x16, dtype=np.float16)
    x_in[:, np.asarray(channels)] = 0
    norm_g, scale_g, q_g = ocache.unpack_outlier_aux(aux_gpu)
    stats = check_codebook_codes(x_in, signs, bits, rows_gpu, norm_g)
    _, aux_o = ocache.encode(x16, signs, "codebook_outlier", bits, b32, c32, outliers=channels)
    _, scale_o, q_o = ocache.unpack_outlier_aux(aux_o)
    assert np.array_equal(scale_g.view(np.uint16), scale_o.view(np.uint16)), "outlier scales differ"
    assert np.array_equal(q_g, q_o), "int8 outlier values differ"
    return stats


def check_float_rows(x16, signs, fmt, rows_gpu, xr=None):
    """fp16 / fp8 rows: every stored value must be the format's rounding of SOME value within
    the kernel's rotation error tau of the exact rotated coordinate, i.e. lie between the
    roundings of x~ - tau and x~ + tau (rounding is monotone; +0 and -0 compare equal).
    Returns (values differing from the oracle's, values)."""
    tau = fwht_error_bound(x16)[:, None] if xr is None else np.zeros((len(xr), 1))  # stored rows: exact input
    xr = rotated(x16, signs, xr)
    rows_o, _ = ocache.encode_rotated(xr, fmt)
    if fmt == "fp16":
        def rnd(z):
            return ofmt.to_f16(z).astype(np.float64)
        vo = np.ascontiguousarray(rows_o).view(np.float16).astype(np.float64)
        vg = np.ascontiguousarray(rows_gpu).view(np.float16).astype(np.float64)
    else:
        def rnd(z):
            return ofmt.e4m3_decode(ofmt.e4m3_encode(ofmt.to_f32(z)))
        vo, vg = ofmt.e4m3_decode(rows_o), ofmt.e4m3_decode(rows_gpu)
    lo, hi = rnd(xr - tau), rnd(xr + tau)
    ok = (vg >= lo) & (vg <= hi)
    if not np.all(ok):
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"{int(np.sum(~ok))} {fmt} values outside [RN(x-tau), RN(x+tau)]; first at {tuple(i)}: "
                             f"gpu {vg[tuple(i)]!r} oracle {vo[tuple(i)]!r} exact {xr[tuple(i)]!r} tau {tau[i[0], 0]!r}")
    return int(np.sum(vo != vg)), vo.size


def check_int4_rows(x16, signs, rows_gpu, scales_gpu, xr=None):
    """INT4-g32 rows: each stored scale must be the rounding of max|x~|/7 for some max within
    tau of the exact one, and each level the rounding of (x~ +- tau) / s with the scale the
    GPU stored (plus one float32 rounding of the quotient).  Returns (levels differing from the
    oracle's, scales differing, levels)."""
    tau = fwht_error_bound(x16)[:, None] if xr is None else np.zeros((len(xr), 1))
    xr = rotated(x16, signs, xr)
    n, d = xr.shape
    rows_o, sc_o = ocache.encode_rotated(xr, "int4_g32")
    g = xr.reshape(n, d // 32, 32)
    amax = np.max(np.abs(g), axis=-1)
    s_lo = ofmt.to_f16(ofmt.to_f32(np.maximum(amax - tau, 0) / 7)).astype(np.float64)
    s_hi = ofmt.to_f16(ofmt.to_f32((amax + tau) / 7)).astype(np.float64)
    sg = np.asarray(scales_gpu, dtype=np.float16).astype(np.float64)
    assert np.all((sg >= s_lo) & (sg <= s_hi)), "group scale outside the rounding interval"
    q_g = ofmt.unpack_bits(rows_gpu, 4, d).reshape(n, d // 32, 32).astype(np.int64) - 8
    q_o = ofmt.unpack_bits(rows_o, 4, d).reshape(n, d // 32, 32).astype(np.int64) - 8
    s = sg[..., None]
    t3 = tau[..., None] + 8 * 2.0 ** -24 * s
    with np.errstate(divide="ignore", invalid="ignore"):
        lo = np.where(s > 0, np.clip(np.rint(ofmt.to_f32((g - t3) / np.where(s > 0, s, 1)).astype(np.float64)), -7, 7), 0)
        hi = np.where(s > 0, np.clip(np.rint(ofmt.to_f32((g + t3) / np.where(s > 0, s, 1)).astype(np.float64)), -7, 7), 0)
    ok = (q_g >= lo) & (q_g <= hi)
    assert np.all(ok), f"{int(np.sum(~ok))} INT4 levels outside the rounding interval"
    return int(np.sum(q_g != q_o)), int(np.sum(sg != sc_o.astype(np.float64))), q_g.size


# ----------------------------------------------------------------------------- exact-bytes decode setup


class Built:
    """An oracle pool and the GPU cache holding the same bytes."""

    def __init__(self, ora_tiers, gpu_caches, views, k_signs, v_signs):
        self.ora, self.gpu, self.views, self.k_signs, self.v_signs = ora_tiers, gpu_caches, views, k_signs, v_signs


def build_exact(kvq, torch, tier_specs, tier_kv, k_signs, v_signs, page_size=16, shuffle_seed=None, k_qjl=None,
                k_outl=None):
    """tier_specs: list of workloads.Tier; tier_kv: per tier, per sequence, (k [L, Hkv, D], v)
    fp16.  The ORACLE encodes every row into numpy pools; those bytes are uploaded into the
    GPU caches unchanged.  Returns Built."""
    hkv, d = k_signs.shape
    batch = len(tier_kv[0])
    rng = np.random.default_rng(shuffle_seed)
    ora_tiers, gpu, views = [], [], []
    ks_dev = torch.from_numpy(k_signs).cuda()
    vs_dev = torch.from_numpy(v_signs).cuda()
    for spec, seqs in zip(tier_specs, tier_kv):
        lens = np.array([k.shape[0] for k, _ in seqs])
        per = [(int(n) + page_size - 1) // page_size for n in lens]
        num_pages = max(1, sum(per) + 2)
        phys = rng.permutation(num_pages) if shuffle_seed is not None else np.arange(num_pages)
        maxp = max(1, max(per))
        bt = np.zeros((batch, maxp), dtype=np.int32)
        at = 0
        for b, n in enumerate(per):
            bt[b, :n] = phys[at: at + n]
            at += n
        kc = tables(spec.codebook, spec.k_bits) if spec.k_format.startswith("codebook") else (None, None)
        vc = tables(spec.codebook, spec.v_bits) if spec.v_format == "codebook" else (None, None)
        proj = k_qjl if spec.k_format == "codebook_qjl" else None
        outl = k_outl if spec.k_format == "codebook_outlier" else None
        ks = ocache.new_side(spec.k_format, spec.k_bits, kc[0], kc[1], k_signs, num_pages, hkv, page_size, d, proj,
                             outl)
        vs = ocache.new_side(spec.v_format, spec.v_bits, vc[0], vc[1], v_signs, num_pages, hkv, page_size, d)
        for b, (k, v) in enumerate(seqs):
            t = np.arange(k.shape[0])
            slots = bt[b, t // page_size] * page_size + t % page_size
            ocache.write(ks, slots, k, page_size)
            ocache.write(vs, slots, v, page_size)
        ora_tiers.append(oatt.TierState(ks, vs, bt, lens, page_size))
        c = kvq.PagedCache(d, hkv, num_pages, spec.k_format, spec.v_format, spec.k_bits, spec.v_bits,
                           ks_dev, vs_dev, page_size, spec.codebook, k_qjl=proj, k_outliers=outl)
        c.k_rows.copy_(torch.from_numpy(ks.rows))
        c.v_rows.copy_(torch.from_numpy(vs.rows))
        if ks.aux is not None:
            c.k_aux.copy_(torch.from_numpy(ks.aux.reshape(c.k_aux.shape)))
        if vs.aux is not None:
            c.v_aux.copy_(torch.from_numpy(vs.aux.reshape(c.v_aux.shape)))
        gpu.append(c)
        views.append(kvq.TierView(c, torch.from_numpy(bt).cuda(), torch.from_numpy(lens.astype(np.int32)).cuda()))
    return Built(ora_tiers, gpu, views, k_signs, v_signs)


# ----------------------------------------------------------------------------- guard bands

GUARD_BYTES = 4096  # canary bytes before and after a guarded buffer (keeps 256-byte alignment)
GUARD_FRONT, GUARD_BACK = 0xA5, 0x5A


def guarded_empty(torch, shape, dtype):
    """(backing uint8 buffer, view of `shape` / `dtype` inside it) with GUARD_BYTES of canary
    pattern on each side, for checking that a kernel writes nothing outside its buffer."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.empty(n + 2 * GUARD_BYTES, dtype=torch.uint8, device="cuda")
    buf[:GUARD_BYTES].fill_(GUARD_FRONT)
    buf[GUARD_BYTES + n:].fill_(GUARD_BACK)
    view = buf[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)
    return buf, view


def assert_guards(buf, view):
    n = view.numel() * view.element_size()
    front, back = buf[:GUARD_BYTES].cpu().numpy(), buf[GUARD_BYTES + n:].cpu().numpy()
    assert (front == GUARD_FRONT).all(), "write before the buffer"
    assert (back == GUARD_BACK).all(), "write after the buffer"


def gpu_decode(kvq, torch, views, q16, split_tokens=0):
    """Decode through the C ABI with guard bands around the output and the workspace and the
    device error report on; both are checked after the call."""
    q = torch.from_numpy(q16).cuda()
    b, hq, d = q16.shape
    out_buf, out = guarded_empty(torch, (b, hq, d), torch.float32)
    ws_buf, ws = guarded_empty(torch, (max(1, kvq.kvq_decode_workspace_size(views, b, hq, split_tokens)),),
                               torch.uint8)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvq.kvq_decode_attention(views, q, out, ws, split_tokens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device error bits {int(status.item())}"
    assert_guards(out_buf, out)
    assert_guards(ws_buf, ws)
    return out.cpu().numpy()
