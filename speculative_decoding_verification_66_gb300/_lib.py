"""ctypes loader for libspecverify.so (argument types only; no logic)."""
from __future__ import annotations

import ctypes
import os
import threading

# The product library, or with SV_LIBRARY=debug in the environment the variant
# built with device-side index checks (_build.build(debug=True)).
_DIR = os.path.dirname(os.path.abspath(__file__))
PRODUCT_PATH = os.path.join(_DIR, "libspecverify.so")
DEBUG_PATH = os.path.join(_DIR, "libspecverify_debug.so")
LIB_PATH = DEBUG_PATH if os.environ.get("SV_LIBRARY", "") == "debug" else PRODUCT_PATH

# Exported names and their C signatures, as declared in include/spec_verify.h.
_vp, _i64, _i32, _f32, _u64, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t)
SIGNATURES = {
    "sv_workspace_bytes": (_i32, [_i64, _i64, _i64, _i32, _i32, ctypes.POINTER(_sz)]),
    "spec_verify": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _u64, _i32, _vp, _vp,
                           _vp, _sz, _vp]),
    "spec_verify_debug": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _u64, _i32, _vp,
                                 _vp, _vp, _sz, _vp, _vp, _vp, _vp, _vp]),
    "spec_verify_timed": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _u64, _i32, _vp,
                                 _vp, _vp, _sz, _vp, _vp, _i32]),
    "sv_host_staging_bytes": (_i32, [_i64, _i64, _i64, _i32, _i32, ctypes.POINTER(_sz)]),
    "spec_verify_host": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _u64, _i32, _vp,
                                _vp, _vp, _sz, _vp]),
    "spec_verify_static": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _u64, _i32, _vp,
                                  _vp, _vp]),
    "sv_early_exit_workspace_bytes": (_i32, [_i64, _i64, _i64, _i32, _i32, ctypes.POINTER(_sz)]),
    "spec_verify_early_exit": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _u64, _i32,
                                      _vp, _vp, _vp, _sz, _vp]),
    "sv_sharded_workspace_bytes": (_i32, [_i64, _i64, _i64, _i32, _i32, _i32,
                                          ctypes.POINTER(_sz)]),
    "spec_verify_sharded": (_i32, [_vp, _vp, _i32, _vp, _i64, _i64, _i64, _i32, _f32, _u64, _i32,
                                   _vp, _vp, _vp, _sz, _vp]),
    "sv_filtered_workspace_bytes": (_i32, [_i64, _i64, _i64, _i32, _i32, ctypes.POINTER(_sz)]),
    "spec_verify_filtered": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _i64, _f32,
                                    _u64, _i32, _vp, _vp, _vp, _sz, _vp]),
    "spec_verify_filtered_debug": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _i64, _f32,
                                          _u64, _i32, _vp, _vp, _vp, _sz, _vp, _vp, _vp, _vp, _vp,
                                          _vp]),
    "spec_verify_filtered_timed": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _i64, _f32,
                                          _u64, _i32, _vp, _vp, _vp, _sz, _vp, _vp, _i32]),
    "sv_lmhead_workspace_bytes": (_i32, [_i64, _i64, _i64, _i64, _i64, _i32,
                                         ctypes.POINTER(_sz)]),
    "spec_verify_lmhead": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _f32,
                                  _u64, _i32, _vp, _vp, _vp, _sz, _vp]),
    "spec_verify_lmhead_debug": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                        _f32, _u64, _i32, _vp, _vp, _vp, _sz, _vp, _vp, _vp, _vp,
                                        _vp]),
    "spec_verify_lmhead_timed": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                        _f32, _u64, _i32, _vp, _vp, _vp, _sz, _vp, _vp, _i32]),
    "spec_verify_gated": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _f32, _i64, _f32, _u64,
                                 _i32, _vp, _vp, _vp, _sz, _vp, _vp, _i32, _vp]),
    "spec_verify_lmhead_gated": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                        _f32, _u64, _i32, _vp, _vp, _vp, _sz, _vp, _vp, _vp]),
    "sv_lmhead_logits": (_i32, [_vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "sv_philox": (_i32, [_u64, _vp, _vp, _i64, _vp]),
    "sv_error_string": (ctypes.c_char_p, [_i32]),
    "sv_version": (_i32, []),
    "sv_device_checks": (_i32, []),
}

_lock = threading.Lock()
_lib = None


class LibraryMissing(RuntimeError):
    pass


def load() -> ctypes.CDLL:
    """Load the in-tree CUDA library. There is no fallback: if the library has
    not been built (``python -c 'import __graft_entry__ as g; g.build()'``),
    this raises."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise LibraryMissing(
                    f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                    "(nvcc, sm_103a). The verification path has no CPU fallback.")
            import torch  # noqa: F401  -- share torch's CUDA runtime when both are loaded
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib
