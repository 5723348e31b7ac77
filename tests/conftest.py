import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and libcsa2")


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def pins_lib():
    """The brute-force codec checkers (tests/pins/pins.c), built on first use."""
    src = os.path.join(ROOT, "tests", "pins", "pins.c")
    so = os.path.join(ROOT, "tests", "pins", "libpins.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-o", so, src, "-lm"])
    L = ctypes.CDLL(so)
    i64 = ctypes.c_int64
    L.pin_e2m1_sweep.restype = i64
    L.pin_e2m1_sweep.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_double), ctypes.c_int,
                                 ctypes.POINTER(ctypes.c_uint32)]
    L.pin_e4m3_sweep.restype = i64
    L.pin_e4m3_sweep.argtypes = L.pin_e2m1_sweep.argtypes
    L.pin_e4m3_brute.restype = i64
    L.pin_e4m3_brute.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_uint32), i64, ctypes.POINTER(ctypes.c_uint32)]
    return L


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle
