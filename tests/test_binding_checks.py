"""The Python binding's argument checks, on the CPU: a host tensor, another dtype, a shape
that disagrees with the call or too few elements are refused before the library sees a
pointer.  The stand-in below reports itself as a CUDA tensor but raises if its address is
taken, so a check that let a call through would fail the test instead of reaching a device."""
import numpy as np
import pytest
import torch

import quantized_decode_attention_rht_gb300 as kvq


class Dev:
    """A CPU tensor that answers like a CUDA one; taking its address is an error."""

    is_cuda = True

    def __init__(self, t):
        self.t = t

    dtype = property(lambda self: self.t.dtype)
    shape = property(lambda self: self.t.shape)

    def dim(self):
        return self.t.dim()

    def numel(self):
        return self.t.numel()

    def is_contiguous(self):
        return True

    def data_ptr(self):
        raise AssertionError("the checks let the call reach the library")


def dev(shape, dtype):
    return Dev(torch.zeros(shape, dtype=dtype))


D, HKV, HQ, B = 128, 2, 8, 3


@pytest.fixture(scope="module")
def cache():
    signs = np.ones((HKV, D), dtype=np.int8)
    return kvq.PagedCache(D, HKV, 4, "codebook", "codebook", 4, 4, signs, signs, device="cpu")


def tiers(cache, rows=B, lens=B, bt_dtype=torch.int32):
    return [kvq.TierView(cache, dev((rows, 4), bt_dtype), dev((lens,), torch.int32))]


def decode(cache, q=None, out=None, ws=None, views=None, **kw):
    q = q if q is not None else dev((B, HQ, D), torch.float16)
    out = out if out is not None else dev((B, HQ, D), torch.float32)
    ws = ws if ws is not None else dev((1024,), torch.uint8)
    kvq.kvq_decode_attention(views if views is not None else tiers(cache), q, out, ws, **kw)


def test_decode_arguments(cache):
    with pytest.raises(AssertionError):  # everything valid: the call goes as far as the pointers
        decode(cache)
    with pytest.raises(ValueError, match="CUDA"):
        decode(cache, q=torch.zeros((B, HQ, D), dtype=torch.float16))
    with pytest.raises(TypeError):
        decode(cache, q=dev((B, HQ, D), torch.float32))
    with pytest.raises(ValueError, match="shape"):
        decode(cache, q=dev((B, HQ, 64), torch.float16))  # not the tiers' head_dim
    with pytest.raises(TypeError):
        decode(cache, out=dev((B, HQ, D), torch.float16))
    with pytest.raises(ValueError, match="shape"):
        decode(cache, out=dev((B, HQ - 1, D), torch.float32))
    with pytest.raises(ValueError, match="CUDA"):
        decode(cache, ws=torch.zeros(1024, dtype=torch.uint8))
    with pytest.raises(ValueError, match="shape"):
        decode(cache, spike_flags=dev((B * HQ,), torch.int32))
    with pytest.raises(TypeError):
        decode(cache, status=dev((1,), torch.int64))
    with pytest.raises(ValueError, match="elements"):
        decode(cache, status=dev((0,), torch.int32))
    with pytest.raises(TypeError):
        decode(cache, views=tiers(cache, bt_dtype=torch.int64))
    with pytest.raises(ValueError, match="rows"):
        decode(cache, views=tiers(cache, rows=B - 1))
    with pytest.raises(ValueError, match="elements"):
        decode(cache, views=tiers(cache, lens=B - 1))
    with pytest.raises(ValueError, match="tier"):
        decode(cache, views=[])
    with pytest.raises(TypeError):
        kvq.kvq_decode_attention_noalloc(tiers(cache), dev((B, HQ, D), torch.float32),
                                         dev((B, HQ, D), torch.float32))
    with pytest.raises(AssertionError):
        kvq.kvq_decode_attention_noalloc(tiers(cache), dev((B, HQ, D), torch.float16),
                                         dev((B, HQ, D), torch.float32))


def test_append_requantize_calibrate_arguments(cache):
    s = cache.struct
    k = dev((5, HKV, D), torch.float16)
    slots = dev((5,), torch.int32)
    with pytest.raises(AssertionError):
        kvq.kvq_quantize_append(s, k, k, slots)
    with pytest.raises(AssertionError):  # keys only
        kvq.kvq_quantize_append(s, k, None, slots)
    with pytest.raises(ValueError):
        kvq.kvq_quantize_append(s, None, None, slots)
    with pytest.raises(TypeError):
        kvq.kvq_quantize_append(s, dev((5, HKV, D), torch.float32), None, slots)
    with pytest.raises(ValueError, match="shape"):
        kvq.kvq_quantize_append(s, dev((5, HKV + 1, D), torch.float16), None, slots)
    with pytest.raises(ValueError, match="shape"):
        kvq.kvq_quantize_append(s, k, dev((4, HKV, D), torch.float16), slots)  # v of another length
    with pytest.raises(ValueError, match="elements"):
        kvq.kvq_quantize_append(s, k, k, dev((4,), torch.int32))
    with pytest.raises(TypeError):
        kvq.kvq_quantize_append(s, k, k, dev((5,), torch.int64))
    with pytest.raises(ValueError, match="CUDA"):
        kvq.kvq_quantize_append(s, torch.zeros((5, HKV, D), dtype=torch.float16), None, slots)

    with pytest.raises(AssertionError):
        kvq.kvq_requantize(s, slots, s, slots)
    with pytest.raises(ValueError, match="elements"):
        kvq.kvq_requantize(s, slots, s, dev((4,), torch.int32))

    out_idx = dev((HKV, kvq.OUTLIER_CHANNELS), torch.int32)
    with pytest.raises(AssertionError):
        kvq.kvq_outlier_calibrate(k, out_idx)
    with pytest.raises(ValueError, match="shape"):
        kvq.kvq_outlier_calibrate(k, dev((HKV + 1, kvq.OUTLIER_CHANNELS), torch.int32))
    with pytest.raises(TypeError):
        kvq.kvq_outlier_calibrate(dev((5, HKV, D), torch.float32), out_idx)
