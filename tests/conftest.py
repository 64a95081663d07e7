import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs through the C ABI)")

_PROBE_SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "probes", "gpu_probes.cu")
_PROBE_OUT = os.path.join(os.path.dirname(_PROBE_SRC), "_build", "libgpu_probes.so")


def _build_probe_lib():
    """The test-only probe library (tests/probes/gpu_probes.cu), compiled for sm_103a on first
    use and again when its sources are newer than the build."""
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_quantize_gb300", "csrc")
    deps = [_PROBE_SRC, os.path.join(csrc, "nvfp4_device.cuh")]
    out = _PROBE_OUT
    if not os.path.exists(out) or any(os.path.getmtime(d) > os.path.getmtime(out) for d in deps):
        os.makedirs(os.path.dirname(out), exist_ok=True)
        tmp = out + ".%d" % os.getpid()
        cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
               "-fmad=false", "-shared", "-Xcompiler", "-fPIC", "-I", csrc, _PROBE_SRC, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stdout + r.stderr
        os.replace(tmp, out)
    L = ctypes.CDLL(out)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    L.probe_cvt_rs_e2m1x4.argtypes = [vp, vp, i64, vp]
    L.probe_cvt_rn_e2m1x2.argtypes = [vp, vp, i64, vp]
    L.probe_div6.argtypes = [ctypes.c_uint32, ctypes.c_uint32, vp, vp]
    L.probe_busy_launch.argtypes = [ctypes.c_int, ctypes.c_uint64, vp, vp]
    return L


@pytest.fixture(scope="session")
def probe_lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    return _build_probe_lib()
