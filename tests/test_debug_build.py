"""The library's debug variant, without a GPU: built with device-side index
checks (-DSV_DEVICE_CHECKS) for sm_103a, it exports exactly the product
library's names and reports its checks; the product library reports none.
The library a process loads follows SV_LIBRARY (debug: the checked variant)."""
import ctypes
import os
import shutil
import subprocess

import pytest

from test_lib_abi import declared_functions


def _nvcc_or_skip():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")


def _exports(path):
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    return sorted(line.split()[-1] for line in out.splitlines() if " T " in line)


def test_debug_variant_builds_with_checks():
    _nvcc_or_skip()
    from speculative_decoding_verification_66_gb300 import _build
    path = _build.build(debug=True)
    assert path == _build.DEBUG_LIB_PATH and os.path.exists(path)
    lib = ctypes.CDLL(path)
    lib.sv_device_checks.restype = ctypes.c_int
    assert lib.sv_device_checks() == 1
    assert _exports(path) == declared_functions()


def test_product_library_has_no_checks():
    _nvcc_or_skip()
    from speculative_decoding_verification_66_gb300 import _build
    lib = ctypes.CDLL(_build.build())
    lib.sv_device_checks.restype = ctypes.c_int
    assert lib.sv_device_checks() == 0


def test_loaded_variant_follows_the_environment():
    _nvcc_or_skip()
    import speculative_decoding_verification_66_gb300 as sv
    from speculative_decoding_verification_66_gb300 import _build, _lib
    want_debug = os.environ.get("SV_LIBRARY", "") == "debug"
    _build.build(debug=want_debug)
    assert _lib.LIB_PATH == (_build.DEBUG_LIB_PATH if want_debug else _build.LIB_PATH)
    assert sv.sv_device_checks() == want_debug
