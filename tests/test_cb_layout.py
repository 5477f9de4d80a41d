"""The codebook decode kernel's shared-memory placement, checked on the host: the layout
code (`Layout::place` / `Layout::area` in csrc/decode_cb.cuh, the functions the kernel
itself calls) is compiled for the CPU with nvcc and run over every kernel instance and
every 16-byte-aligned start of the dynamic shared-memory window (tables aligned to their
size, warp areas disjoint and clear of the tables, everything inside the launch's window
of at most 227 KB)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_codebook_kernel_shared_memory_placement(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "cb_layout_check")
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"),
                        os.path.join(HERE, "cb_layout_check.cu"), "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-3000:]
    lines = r.stdout.splitlines()
    assert lines[-1] == "0 failures"
    assert "planted mistake caught" in lines  # the checker does reject a window that is too small
    assert sum(l.startswith("ok ") for l in lines) == 9 * (3 * 2 + 2 + 3 + 3 * 2)
    # the quad table (2-bit values on the tensor-core path) is placed where it fits
    assert any(" quad 65536 " in l and "V2" in l and "PathM" in l for l in lines)
