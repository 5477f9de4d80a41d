"""The C ABI without a GPU: the library builds and loads, exports exactly the entry points
include/kvq.h declares, its host-side codebooks agree with the oracle's, and argument
checks fail before anything is launched."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import codebook as ocb
from oracle import formats as ofmt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    from quantized_decode_attention_rht_gb300 import build
    build.build()
    import quantized_decode_attention_rht_gb300 as m
    m.lib()
    return m


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", text)))


def test_exports_match_header(kvq):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(kvq.lib(), n), n
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == names


def test_launch_counter_is_host_side(kvq):
    n = kvq.kvq_kernel_launches()
    assert isinstance(n, int) and n >= 0
    assert kvq.kvq_quantize_append is not None  # argument checks below launch nothing
    assert kvq.kvq_kernel_launches() == n


def test_status_strings(kvq):
    for s, name in kvq.STATUS.items():
        assert kvq.kvq_status_string(s) == name
    assert kvq.kvq_status_string(99) == "KVQ_ERR_UNKNOWN"


@pytest.mark.parametrize("d", [64, 128, 256])
def test_row_bytes_match_oracle(kvq, d):
    for fmt in ("codebook", "codebook_qjl", "codebook_outlier", "fp16", "fp8_e4m3", "int4_g32"):
        for bits in ((2, 3, 4) if fmt.startswith("codebook") else (0,)):
            if d == 64 and fmt in ("codebook_qjl", "codebook_outlier"):  # codebook kernel only: D 128, 256
                with pytest.raises(kvq.KvqError):
                    kvq.kvq_row_bytes(fmt, bits, d)
                continue
            assert kvq.kvq_row_bytes(fmt, bits, d) == (ofmt.row_bytes(fmt, bits, d), ofmt.aux_bytes(fmt, d))
    with pytest.raises(kvq.KvqError):
        kvq.kvq_row_bytes("codebook", 5, d)
    for bad in (32, 96, 512):
        with pytest.raises(kvq.KvqError):
            kvq.kvq_row_bytes("fp16", 0, bad)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_lloyd_max_library_matches_oracle(kvq, bits):
    c, b = kvq.kvq_lloyd_max_codebook(bits)
    oc, ob, _ = ocb.lloyd_max(bits)
    np.testing.assert_allclose(c, oc, rtol=0, atol=1e-9)
    np.testing.assert_allclose(b, ob, rtol=0, atol=1e-9)
    c32, b32 = kvq.kvq_codebook_tables(bits, c)
    oc32, ob32 = ocb.float32_tables(oc)
    assert np.array_equal(c32, oc32) and np.array_equal(b32, ob32)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_uniform_library_matches_oracle(kvq, bits):
    c, b = kvq.kvq_uniform_codebook(bits)
    oc, ob, _ = ocb.uniform_codebook(bits)
    np.testing.assert_allclose(c, oc, rtol=0, atol=1e-9)
    c32, b32 = kvq.kvq_codebook_tables(bits, c)
    oc32, ob32 = ocb.float32_tables(oc)
    assert np.array_equal(c32, oc32) and np.array_equal(b32, ob32)


def _fake_cache(kvq, **kw):
    """A cache struct with aligned, never-dereferenced fake device addresses."""
    s = kvq.KvqCache()
    s.head_dim, s.num_kv_heads, s.page_size, s.num_pages = 128, 2, 16, 4
    s.k_format = s.v_format = kvq.FMT_CODEBOOK
    s.k_bits = s.v_bits = 4
    base = 1 << 40
    for i, f in enumerate(("k_rows", "v_rows", "k_aux", "v_aux", "k_centroids", "k_bounds", "v_centroids",
                           "v_bounds", "k_signs", "v_signs")):
        setattr(s, f, base + 4096 * i)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


@pytest.fixture(autouse=True)
def _no_gpu_for_fabricated_addresses():
    """The argument checks below hand the library made-up device addresses, relying on the
    host-side check to refuse the call first; they only run where no GPU exists, so a check
    that someday came too late could not reach a device."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("host-only checks with fabricated device addresses")
    except ImportError:
        pass


def _quant(kvq, cache, k=1 << 41, v=1 << 41, n=3, slots=1 << 42):
    return kvq.lib().kvq_quantize_append(ctypes.byref(cache), k, v, n, slots, None)


def test_quantize_argument_checks(kvq):
    L = kvq.lib()
    assert L.kvq_quantize_append(None, 1 << 41, None, 3, 1 << 42, None) == 1
    assert _quant(kvq, _fake_cache(kvq, head_dim=96)) == 2
    assert _quant(kvq, _fake_cache(kvq, head_dim=512)) == 2
    assert _quant(kvq, _fake_cache(kvq, k_bits=5)) == 2
    assert _quant(kvq, _fake_cache(kvq, k_format=7)) == 1
    assert _quant(kvq, _fake_cache(kvq, k_rows=None)) == 1
    assert _quant(kvq, _fake_cache(kvq, k_rows=(1 << 40) + 8)) == 1  # rows not 16-byte aligned
    assert _quant(kvq, _fake_cache(kvq, k_bounds=None)) == 1
    assert _quant(kvq, _fake_cache(kvq), k=None, v=None) == 1
    assert _quant(kvq, _fake_cache(kvq), n=-1) == 1
    assert _quant(kvq, _fake_cache(kvq), slots=None) == 1
    assert _quant(kvq, _fake_cache(kvq), k=(1 << 41) + 2) == 1  # input not 16-byte aligned
    assert _quant(kvq, _fake_cache(kvq), n=0) == 0  # nothing to do
    assert _quant(kvq, _fake_cache(kvq), k=None, v=None, n=0, slots=None) == 0  # empty tensors may have no address


def _views(kvq, caches, max_pages=8):
    arr = (kvq.KvqTierView * len(caches))()
    for i, c in enumerate(caches):
        arr[i].cache = ctypes.pointer(c)
        arr[i].block_table = 1 << 43
        arr[i].seq_lens = 1 << 44
        arr[i].max_pages = max_pages
    return arr


def _ws(kvq, caches, batch=2, hq=4, split=0, max_pages=8):
    n = ctypes.c_size_t()
    st = kvq.lib().kvq_decode_workspace_size(_views(kvq, caches, max_pages), len(caches), batch, hq, split,
                                             ctypes.byref(n))
    return st, n.value


def test_decode_argument_checks(kvq):
    c = _fake_cache(kvq)
    assert _ws(kvq, [c])[0] == 0
    for hq in (2, 4, 8, 16):  # head_dim 64: the generic kernel, every group size
        assert _ws(kvq, [_fake_cache(kvq, head_dim=64)], hq=hq)[0] == 0
    assert _ws(kvq, [_fake_cache(kvq, head_dim=96)])[0] == 2
    assert _ws(kvq, [c], hq=6)[0] == 2  # Hq/Hkv = 3 is not built
    assert _ws(kvq, [c], hq=3)[0] == 1  # Hq not a multiple of Hkv
    assert _ws(kvq, [c] * 5)[0] == 1  # more tiers than KVQ_MAX_TIERS
    assert _ws(kvq, [c, _fake_cache(kvq, k_signs=(1 << 40) + 4096 * 20)])[0] == 1  # tiers disagree on signs
    assert _ws(kvq, [c, _fake_cache(kvq, num_kv_heads=4)])[0] == 1
    assert _ws(kvq, [c], split=24)[0] == 1  # split not a multiple of the page size
    assert _ws(kvq, [c], split=16, max_pages=2000)[0] == 2  # more than KVQ_MAX_SPLITS chunks
    assert _ws(kvq, [c], split=32, max_pages=2000)[0] == 0
    assert _ws(kvq, [_fake_cache(kvq, k_format=kvq.FMT_FP16, v_format=kvq.FMT_CODEBOOK)])[0] == 2
    # decode with too small a workspace fails before any launch
    L = kvq.lib()
    st = L.kvq_decode_attention(_views(kvq, [c]), 1, 1 << 45, 2, 4, 0, 1 << 46, 1 << 47, 16, None)
    assert st == 3


def test_workspace_size_formula(kvq):
    c = _fake_cache(kvq)
    # 2 sequences, 4 query heads, 8 pages of 16 tokens, 32-token splits -> 4 splits
    st, n = _ws(kvq, [c], batch=2, hq=4, split=32, max_pages=8)
    parts = 2 * 4 * 4
    # partial accumulators + (max, sum) pairs + lowest scores, each rounded up to 256 B,
    # + 256 B work counter
    want = -(-parts * 128 * 4 // 256) * 256 + -(-parts * 2 * 4 // 256) * 256 + -(-parts * 4 // 256) * 256 + 256
    assert st == 0 and n == want


def _qjl_cache(kvq, **kw):
    args = dict(k_format=kvq.FMT_CODEBOOK_QJL, k_qjl=(1 << 40) + 4096 * 30)
    args.update(kw)
    return _fake_cache(kvq, **args)


def test_qjl_key_checks(kvq):
    """Keys with a residual sketch need the projection (16-byte aligned) and 16-byte
    aligned (norm, residual norm) pairs; values may not carry a sketch."""
    assert kvq.kvq_row_bytes("codebook_qjl", 3, 128) == (128 * 3 // 8 + 16, 4)
    assert _quant(kvq, _qjl_cache(kvq), n=0) == 0  # arguments accepted (nothing to launch)
    assert _quant(kvq, _qjl_cache(kvq, k_qjl=None)) == 1
    assert _quant(kvq, _qjl_cache(kvq, k_qjl=(1 << 40) + 4096 * 30 + 4)) == 1
    assert _quant(kvq, _qjl_cache(kvq, k_aux=(1 << 40) + 4096 * 2 + 2)) == 1
    assert _quant(kvq, _qjl_cache(kvq, v_format=kvq.FMT_CODEBOOK_QJL)) == 1
    assert _ws(kvq, [_qjl_cache(kvq)])[0] == 0
    assert _ws(kvq, [_qjl_cache(kvq)], hq=4 * 2)[0] == 0  # 4 query heads per kv head
    assert _ws(kvq, [_qjl_cache(kvq, head_dim=256)])[0] == 2  # the sketched decode is built for D=128
    assert _quant(kvq, _qjl_cache(kvq, head_dim=64)) == 2 and _ws(kvq, [_qjl_cache(kvq, head_dim=64)])[0] == 2
    assert _ws(kvq, [_qjl_cache(kvq, v_format=kvq.FMT_FP16, v_bits=0)])[0] == 2
    assert _ws(kvq, [_qjl_cache(kvq), _fake_cache(kvq)])[0] == 0  # with a plain codebook tier
    # a tier of another kernel family runs on its own kernel in the same call
    assert _ws(kvq, [_qjl_cache(kvq), _fake_cache(kvq, k_format=kvq.FMT_FP8_E4M3, k_bits=0,
                                                    v_format=kvq.FMT_INT4_G32, v_bits=0)])[0] == 0
    assert _ws(kvq, [_qjl_cache(kvq), _qjl_cache(kvq, k_qjl=(1 << 40) + 4096 * 31)])[0] == 1
    assert _ws(kvq, [_qjl_cache(kvq, page_size=32)])[0] == 2
    assert _ws(kvq, [_qjl_cache(kvq)], hq=2 * 8)[0] == 2  # 8 query heads per kv head


def test_requantize_checks(kvq):
    """Moving tokens out of an fp16 window: argument checks before any launch."""
    L = kvq.lib()
    win = _fake_cache(kvq, k_format=kvq.FMT_FP16, v_format=kvq.FMT_FP16, k_bits=0, v_bits=0)
    dst = _fake_cache(kvq)

    def rq(src, d, n=3, ss=1 << 42, ds=1 << 43):
        return L.kvq_requantize(ctypes.byref(src), ss, ctypes.byref(d), ds, n, None)

    assert rq(win, dst, n=0) == 0  # nothing to move
    assert rq(win, dst, n=-1) == 1
    assert rq(dst, dst, n=0) == 2  # the source must be an fp16 tier
    assert rq(win, _fake_cache(kvq, head_dim=256), n=0) == 1
    assert rq(win, _fake_cache(kvq, num_kv_heads=4), n=0) == 1
    assert rq(win, _fake_cache(kvq, k_signs=(1 << 40) + 4096 * 20), n=0) == 1  # another rotation
    assert rq(win, _fake_cache(kvq, k_bounds=None), n=0) == 1
    assert rq(win, dst, n=2, ss=None) == 1
    assert rq(win, dst, n=2, ds=(1 << 43) + 2) == 1
    assert rq(win, dst, n=(1 << 28) // win.num_kv_heads + 1) == 1  # past 2^28 vectors: split the move
    assert rq(_fake_cache(kvq, k_format=kvq.FMT_FP16, v_format=kvq.FMT_FP16, k_rows=(1 << 40) + 8), dst, n=0) == 1


def _outl_cache(kvq, **kw):
    args = dict(k_format=kvq.FMT_CODEBOOK_OUTLIER, k_outliers=(1 << 40) + 4096 * 32)
    args.update(kw)
    return _fake_cache(kvq, **args)


def test_outlier_key_checks(kvq):
    """Keys with an outlier stream need the channel list (16-byte aligned) and 16-byte
    aligned side data; values may not carry one; decode runs on the codebook kernel
    (head_dim 128 or 256, groups 1, 2, 4); a re-encode into it is not offered."""
    assert kvq.kvq_row_bytes("codebook_outlier", 4, 128) == (64, 12)
    assert _quant(kvq, _outl_cache(kvq), n=0) == 0
    assert _quant(kvq, _outl_cache(kvq, k_outliers=None)) == 1
    assert _quant(kvq, _outl_cache(kvq, k_outliers=(1 << 40) + 4096 * 32 + 4)) == 1
    assert _quant(kvq, _outl_cache(kvq, k_aux=(1 << 40) + 4096 * 2 + 4)) == 1
    assert _quant(kvq, _outl_cache(kvq, v_format=kvq.FMT_CODEBOOK_OUTLIER)) == 1
    assert _ws(kvq, [_outl_cache(kvq)])[0] == 0
    assert _ws(kvq, [_outl_cache(kvq, head_dim=256)])[0] == 0
    assert _ws(kvq, [_outl_cache(kvq)], hq=2 * 4)[0] == 0
    assert _ws(kvq, [_outl_cache(kvq)], hq=2 * 8)[0] == 2
    assert _ws(kvq, [_outl_cache(kvq, v_format=kvq.FMT_FP16, v_bits=0)])[0] == 2
    win = _fake_cache(kvq, k_format=kvq.FMT_FP16, v_format=kvq.FMT_FP16, k_bits=0, v_bits=0)
    assert kvq.lib().kvq_requantize(ctypes.byref(win), 1 << 42, ctypes.byref(_outl_cache(kvq)), 1 << 43, 0,
                                    None) == 2


def test_outlier_calibrate_checks(kvq):
    L = kvq.lib()
    assert L.kvq_outlier_calibrate(None, 10, 2, 128, 1 << 42, None) == 1
    assert L.kvq_outlier_calibrate(1 << 41, 0, 2, 128, 1 << 42, None) == 1
    assert L.kvq_outlier_calibrate(1 << 41, 10, 0, 128, 1 << 42, None) == 1
    assert L.kvq_outlier_calibrate(1 << 41, 10, 2, 64, 1 << 42, None) == 2
    assert L.kvq_outlier_calibrate(1 << 41, 10, 2, 128, (1 << 42) + 2, None) == 1


@pytest.mark.parametrize("seed,layer,hkv,d", [(0, 0, 1, 64), (12345, 3, 8, 128), ((1 << 64) - 1, 31, 2, 256),
                                              (0x9E3779B97F4A7C15, 1000, 16, 128)])
def test_make_signs_matches_oracle(kvq, seed, layer, hkv, d):
    from oracle import signs as osg
    k, v = kvq.kvq_make_signs(seed, layer, hkv, d)
    ok, ov = osg.make_signs(seed, layer, hkv, d)
    assert np.array_equal(k, ok) and np.array_equal(v, ov)


def test_make_signs_argument_checks(kvq):
    lib = kvq.lib()
    buf = np.zeros(256, dtype=np.int8)
    assert lib.kvq_make_signs(0, 0, 1, 128, None, buf.ctypes.data) == 1
    assert lib.kvq_make_signs(0, -1, 1, 128, buf.ctypes.data, buf.ctypes.data) == 1
    assert lib.kvq_make_signs(0, 1 << 24, 1, 128, buf.ctypes.data, buf.ctypes.data) == 1
    assert lib.kvq_make_signs(0, 0, 0, 128, buf.ctypes.data, buf.ctypes.data) == 1
    assert lib.kvq_make_signs(0, 0, 1, 96, buf.ctypes.data, buf.ctypes.data) == 2


def test_eight_query_heads_per_kv_head(kvq):
    """Eight query heads per kv head: plain codebook tiers (D 128, 256), fp16 and fp8 / INT4
    tiers (D 128) and the generic kernel (D 64) accept the call; keys with a residual sketch or
    an outlier stream, which only the codebook kernel's 1/2/4-head instances read, refuse it
    before any launch."""
    hq = 8 * 2  # the fake caches have 2 kv heads
    assert _ws(kvq, [_fake_cache(kvq)], hq=hq)[0] == 0
    assert _ws(kvq, [_fake_cache(kvq, head_dim=256)], hq=hq)[0] == 0
    assert _ws(kvq, [_fake_cache(kvq, head_dim=64)], hq=hq)[0] == 0
    assert _ws(kvq, [_fake_cache(kvq, k_format=kvq.FMT_FP16, v_format=kvq.FMT_FP16, k_bits=0, v_bits=0),
                     _fake_cache(kvq, k_format=kvq.FMT_FP8_E4M3, k_bits=0, v_format=kvq.FMT_INT4_G32, v_bits=0)],
               hq=hq)[0] == 0
    assert _ws(kvq, [_qjl_cache(kvq)], hq=hq)[0] == 2
    assert _ws(kvq, [_outl_cache(kvq)], hq=hq)[0] == 2
    assert _ws(kvq, [_qjl_cache(kvq)], hq=4 * 2)[0] == 0 and _ws(kvq, [_outl_cache(kvq)], hq=4 * 2)[0] == 0


def test_library_chosen_chunks_fit_long_block_tables(kvq):
    """With split_tokens = 0 the chunks sized for the GPU's item count lengthen where one
    long sequence would need more splits than KVQ_MAX_SPLITS (few sequences at long
    context); the fused fp16 / fp8 kernel's chunks stop at 2048 tokens, so its tiers refuse
    block tables of more than KVQ_MAX_SPLITS x 2048 tokens in total.  An explicit split size
    is taken as given."""
    def fp16(**kw):
        return _fake_cache(kvq, k_format=kvq.FMT_FP16, v_format=kvq.FMT_FP16, k_bits=0, v_bits=0,
                           num_pages=1 << 20, **kw)

    for hkv, hq in ((2, 4), (8, 32)):
        for c in (fp16(num_kv_heads=hkv), _fake_cache(kvq, num_kv_heads=hkv, num_pages=1 << 20),
                  _fake_cache(kvq, num_kv_heads=hkv, num_pages=1 << 20, page_size=8)):
            for mp in (4096, 65536, 131072):  # up to 2,097,152 tokens (1,048,576 at page size 8)
                assert _ws(kvq, [c], batch=1, hq=hq, max_pages=mp)[0] == 0, (hkv, c.k_format, c.page_size, mp)
    assert _ws(kvq, [fp16()], batch=1, hq=4, max_pages=1024 * 128)[0] == 0
    assert _ws(kvq, [fp16()], batch=1, hq=4, max_pages=1024 * 128 + 1)[0] == 2
    assert _ws(kvq, [fp16(), fp16()], batch=1, hq=4, max_pages=512 * 128)[0] == 0
    assert _ws(kvq, [fp16(), fp16()], batch=1, hq=4, max_pages=512 * 128 + 1)[0] == 2
    assert _ws(kvq, [fp16()], batch=1, hq=4, split=16, max_pages=1025)[0] == 2


def test_generic_kernel_batch_limit(kvq):
    """The generic kernel's grid holds the sequences in its z extent: a tier on it takes at
    most 65535 sequences a call, refused before any launch beyond; the fused kernels, which
    are persistent, take any batch."""
    generic = _fake_cache(kvq, page_size=8)
    assert _ws(kvq, [generic], batch=65535, hq=4, max_pages=2)[0] == 0
    assert _ws(kvq, [generic], batch=65536, hq=4, max_pages=2)[0] == 2
    assert _ws(kvq, [_fake_cache(kvq)], batch=65536, hq=4, max_pages=2)[0] == 0
