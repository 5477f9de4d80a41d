"""CPU oracle for rotate-then-quantize KV-cache compression and decode attention.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` / reference arm
may import or call anything in this package.  The CUDA path never does, and
this package never imports the CUDA path: the two share no code.  The only
module both sides use is ``workloads`` (seeded inputs, no method arithmetic).

Everything here is plain numpy in float64 and follows the pages step by step,
in their order and notation, so that it can be checked against them by eye:

  signs.py      the Rademacher sign vectors (SplitMix64, one draw per sign)
  rotation.py   random signs + Sylvester Walsh-Hadamard, orthonormal scaling
  codebook.py   Lloyd-Max for N(0,1) by trapezoidal quadrature; uniform codebook
  formats.py    fp16 / fp8-E4M3 rounding, INT4 with per-32-group scale, bit packing
  cache.py      encode one vector per format; paged pool write and read
  attention.py  dequantise, undo the rotation, then plain softmax(q K^T / sqrt(d)) V

Where floating point decides an integer (a code index, an INT4 level, an fp16 /
fp8 rounding) the oracle first computes the exact value in float64, rounds it
to float32 -- the precision the CUDA kernels hold their values in -- and takes
the decision on that float32 value.

Every function is pinned by ``tests/test_oracle_*.py`` to facts that do not
come from the oracle itself (closed forms, library routines, the pages' worked
examples, brute force on tiny inputs).  No function here is "parity unpinned".
"""
from . import signs, rotation, codebook, formats, cache, attention  # noqa: F401
