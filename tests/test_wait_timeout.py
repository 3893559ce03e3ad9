"""The bounded-wait path: a wait that nothing completes gives up, raises the
status bit and lets the kernel return.

Every mbarrier wait of the replay kernels is bounded by %globaltimer (2 s in
the library).  tests/csrc/wait_timeout.cu is built here with a 5 ms limit and
waits, through the library's own wait functions, on an mbarrier that no
thread ever arrives at.  The CPU test only builds it (nvcc cross-compiles);
the GPU test runs it and checks that each wait gave up after the limit, that
the status word carries RS_DEV_TIMEOUT, and that the context stays usable.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "csrc", "wait_timeout.cu")
OUT = os.path.join(ROOT, "tests", "_build", "libwait_timeout.so")
LIMIT_NS = 5_000_000


def _build() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    tmp = OUT + f".tmp{os.getpid()}"
    cmd = [nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-Xcompiler",
           "-fPIC", f"-DRS_WAIT_LIMIT_NS={LIMIT_NS}ull", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(ROOT, "rs_decode_gb300", "csrc"), SRC, "-o", tmp, "--cudart=shared"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    os.replace(tmp, OUT)
    return OUT


def test_wait_timeout_kernel_builds():
    assert os.path.getsize(_build()) > 0


@pytest.mark.gpu
def test_wait_gives_up_and_reports_timeout():
    import torch
    from rs_decode_gb300 import binding as rb
    lib = ctypes.CDLL(_build())
    lib.rs_test_wait_timeout.argtypes = [ctypes.c_void_p] * 4
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ns = torch.zeros(4, dtype=torch.int64, device="cuda")
    res = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    assert lib.rs_test_wait_timeout(status.data_ptr(), ns.data_ptr(), res.data_ptr(), stream.cuda_stream) == 0
    torch.cuda.synchronize()
    w1, w2, w3, flag = res.tolist()
    t1, t2, t3, limit = ns.tolist()
    assert limit == LIMIT_NS
    assert (w1, w2, w3, flag) == (0, 0, 0, 1)
    assert LIMIT_NS <= t1 < 50 * LIMIT_NS
    # the second wait ends at the limit of whichever thread started it first
    # (its flag then releases the others, thread 0 among them)
    assert LIMIT_NS // 2 <= t2 < 50 * LIMIT_NS
    assert t3 < LIMIT_NS  # the raised flag ends a later wait at once
    assert status.item() & 0x8  # RS_DEV_TIMEOUT
    # the context is still usable: a library call runs normally afterwards
    x = torch.arange(8, device="cuda", dtype=torch.float32)
    assert float((x * 2).sum()) == 56.0
    assert "sm_103a" in rb.rs_version()
