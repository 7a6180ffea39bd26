"""Bounded device waits give up instead of hanging (-m gpu).

Every mbarrier wait in the library's kernels polls for at most a fixed
number of SM clock cycles (about one second), then records
DQ_ERR_DEVICE_TIMEOUT in a device status word and returns.  This test builds
the library's wait helpers with a limit of about one millisecond into a small
test library, runs one kernel whose barrier nothing ever arrives on (CTA and
cluster scope, no bulk copy in flight), and checks that every thread returned
from the wait with a failure and that the status word holds the timeout.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
DQ_ERR_DEVICE_TIMEOUT = -6


@pytest.fixture(scope="module")
def wt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    out = os.path.join(tempfile.mkdtemp(prefix="dq_wait_"), "libwt.so")
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-rdc=true", "-shared", "-Xcompiler", "-fPIC", "-DDQ_WAIT_LIMIT_CYCLES=2000000LL",
                    "-I", os.path.join(os.path.dirname(HERE), "include"),
                    os.path.join(HERE, "csrc", "wait_timeout.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.wt_run.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
    lib.wt_status.argtypes = [ctypes.c_void_p]
    return lib


@pytest.mark.parametrize("cluster", [0, 1])
def test_wait_gives_up_and_reports(wt, cluster):
    st = ctypes.c_int(99)
    assert wt.wt_status(ctypes.byref(st)) == 0
    assert st.value == 0
    n = 64
    out = np.zeros(n, dtype=np.int32)
    assert wt.wt_run(cluster, out.ctypes.data_as(ctypes.c_void_p), n) == 0
    assert (out == 2).all(), out                # every thread left its wait, unsatisfied
    assert wt.wt_status(ctypes.byref(st)) == 0
    assert st.value == DQ_ERR_DEVICE_TIMEOUT
    # read-and-clear: the next read is clean, and the context still works
    assert wt.wt_status(ctypes.byref(st)) == 0
    assert st.value == 0
    assert float(torch.ones(4, device="cuda").sum()) == 4.0
