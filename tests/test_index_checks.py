"""The decode kernels' device-side index checks, exercised on the host: the functions in
csrc/kvq_internal.cuh that every decode kernel applies to the lengths and block-table
entries it reads (clamp a length into [0, max_pages * page_size], skip a page outside the
pool, never read more splits than the plan made), each raising its KVQ_DEVERR_* bit, are
compiled for the CPU with nvcc and fed out-of-range values -- on the CPU only.  The same
program walks the generic decode kernel's page loop with its slot test for every page size
up to 40 and every warp step width: each token of a chunk once, no lane past its page."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_device_index_checks_on_host(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "index_check")
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"),
                        os.path.join(HERE, "index_check.cu"), "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout[-3000:]
    assert r.stdout.splitlines()[-1] == "0 failures"
