"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
exactly what include/spec_verify.h declares, and rejects bad arguments on the
host before it makes any CUDA call."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")

SV_OK, SV_ERR_ARG, SV_ERR_DTYPE, SV_ERR_ALIGN, SV_ERR_WORKSPACE, SV_ERR_CUDA, SV_ERR_SIZE = \
    0, -1, -2, -3, -4, -5, -6


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from speculative_decoding_verification_66_gb300 import _build, _lib
    _build.build()
    return _lib.load()


def test_header_declares_the_api():
    assert declared_functions() == sorted([
        "sv_workspace_bytes", "spec_verify", "spec_verify_debug", "spec_verify_timed",
        "sv_host_staging_bytes", "spec_verify_host", "spec_verify_static", "spec_verify_gated",
        "sv_early_exit_workspace_bytes", "spec_verify_early_exit",
        "sv_sharded_workspace_bytes", "spec_verify_sharded", "sv_philox",
        "sv_filtered_workspace_bytes", "spec_verify_filtered", "spec_verify_filtered_timed",
        "spec_verify_filtered_debug",
        "sv_lmhead_workspace_bytes", "spec_verify_lmhead", "spec_verify_lmhead_debug",
        "spec_verify_lmhead_timed", "spec_verify_lmhead_gated", "sv_lmhead_logits",
        "sv_error_string",
        "sv_version", "sv_device_checks"])


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_nothing_else_is_exported(lib):
    from speculative_decoding_verification_66_gb300 import _lib
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines() if " T " in line)
    assert exported == declared_functions()


def test_python_binding_names_match_the_header():
    import speculative_decoding_verification_66_gb300 as sv
    from speculative_decoding_verification_66_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == declared_functions()
    for name in declared_functions():
        if name not in ("sv_error_string", "sv_version"):  # (sv_device_checks: api.py)
            assert callable(getattr(sv, name)), name


def test_error_strings_and_version(lib):
    for code in (SV_OK, SV_ERR_ARG, SV_ERR_DTYPE, SV_ERR_ALIGN, SV_ERR_WORKSPACE, SV_ERR_CUDA,
                 SV_ERR_SIZE, 12345):
        s = lib.sv_error_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.sv_version() == 105


FAKE = 0x10000  # never dereferenced: every case below fails before any device work


def call(lib, B=2, K=3, V=64, dtype=1, T=1.0, mode=0, target=FAKE, draft=FAKE, tokens=FAKE,
         out=FAKE, nacc=FAKE, ws=FAKE, ws_bytes=1 << 20):
    return lib.spec_verify(target, draft, tokens, B, K, V, dtype, T, 7, mode, out, nacc, ws,
                           ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), SV_OK),
    (dict(B=0, target=None, draft=None, tokens=None, out=None, nacc=None, ws=None), SV_OK),
    (dict(dtype=7), SV_ERR_DTYPE),
    (dict(mode=5), SV_ERR_ARG),
    (dict(T=0.0), SV_ERR_ARG),
    (dict(T=-1.0), SV_ERR_ARG),
    (dict(T=float("nan")), SV_ERR_ARG),
    (dict(T=float("inf")), SV_ERR_ARG),
    (dict(T=1e-45), SV_ERR_ARG),            # log2(e)/T overflows float
    (dict(B=-1), SV_ERR_ARG),
    (dict(K=-1), SV_ERR_ARG),
    (dict(V=0), SV_ERR_ARG),
    (dict(K=1025), SV_ERR_SIZE),
    (dict(V=1 << 31), SV_ERR_SIZE),
    (dict(B=1 << 31), SV_ERR_SIZE),
    (dict(B=1 << 30, K=1024, V=(1 << 31) - 1), SV_ERR_SIZE),
    (dict(target=None), SV_ERR_ARG),
    (dict(out=None), SV_ERR_ARG),
    (dict(nacc=None), SV_ERR_ARG),
    (dict(tokens=None), SV_ERR_ARG),
    (dict(draft=None), SV_ERR_ARG),
    (dict(target=FAKE + 2), SV_ERR_ALIGN),
    (dict(draft=FAKE + 8), SV_ERR_ALIGN),
    (dict(tokens=FAKE + 2), SV_ERR_ALIGN),
    (dict(out=FAKE + 1), SV_ERR_ALIGN),
    (dict(ws=None), SV_ERR_WORKSPACE),
    (dict(ws=FAKE + 16), SV_ERR_WORKSPACE),
])
def test_host_side_validation(lib, kw, code):
    assert call(lib, **kw) == code


def call_ee(lib, B=2, K=3, V=64, dtype=1, T=1.0, mode=0, target=FAKE, draft=FAKE, tokens=FAKE,
            out=FAKE, nacc=FAKE, ws=FAKE, ws_bytes=1 << 20):
    return lib.spec_verify_early_exit(target, draft, tokens, B, K, V, dtype, T, 7, mode, out, nacc,
                                      ws, ws_bytes, None)


def test_sharded_host_side_validation(lib):
    """spec_verify_sharded checks its shard arguments before any CUDA call."""
    import ctypes
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    bad = (ctypes.c_void_p * 2)(FAKE, FAKE + 2)
    nul = (ctypes.c_void_p * 2)(FAKE, None)

    def sh(G=2, t=arr, d=arr, B=2, K=3, Vs=32, dtype=1):
        return lib.spec_verify_sharded(ctypes.cast(t, ctypes.c_void_p) if t is not None else None,
                                       ctypes.cast(d, ctypes.c_void_p) if d is not None else None,
                                       G, FAKE, B, K, Vs, dtype, 1.0, 7, 0, FAKE, FAKE, FAKE,
                                       1 << 20, None)
    assert sh(B=0) == SV_OK
    assert sh(G=0) == SV_ERR_ARG
    assert sh(G=17) == SV_ERR_ARG
    assert sh(Vs=0) == SV_ERR_ARG
    assert sh(t=None) == SV_ERR_ARG
    assert sh(d=None) == SV_ERR_ARG
    assert sh(t=nul) == SV_ERR_ARG
    assert sh(t=bad) == SV_ERR_ALIGN
    assert sh(d=bad) == SV_ERR_ALIGN
    assert sh(dtype=9) == SV_ERR_DTYPE


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), SV_OK),
    (dict(dtype=7), SV_ERR_DTYPE),
    (dict(T=0.0), SV_ERR_ARG),
    (dict(K=1025), SV_ERR_SIZE),
    (dict(target=None), SV_ERR_ARG),
    (dict(draft=FAKE + 8), SV_ERR_ALIGN),
    (dict(ws=None), SV_ERR_WORKSPACE),
])
def test_early_exit_host_side_validation(lib, kw, code):
    """The early-exit entry shares spec_verify's checks, all before any CUDA call."""
    assert call_ee(lib, **kw) == code


def test_filtered_host_side_validation(lib):
    """spec_verify_filtered checks top_k / top_p with the other arguments,
    before any CUDA call."""
    def f(B=2, K=3, V=64, dtype=1, T=1.0, top_k=5, top_p=0.9, mode=0, target=FAKE, events=None,
          n_events=0):
        args = (target, FAKE, FAKE, B, K, V, dtype, T, top_k, top_p, 7, mode, FAKE, FAKE, FAKE,
                1 << 20, None)
        if events is None and n_events == 0:
            return lib.spec_verify_filtered(*args)
        return lib.spec_verify_filtered_timed(*args, events, n_events)
    assert f(B=0) == SV_OK
    assert f(B=0, top_k=0, top_p=1.0) == SV_OK
    assert f(top_k=-1) == SV_ERR_ARG
    assert f(top_p=0.0) == SV_ERR_ARG
    assert f(top_p=1.5) == SV_ERR_ARG
    assert f(top_p=float("nan")) == SV_ERR_ARG
    assert f(B=0, top_p=-0.5) == SV_ERR_ARG
    assert f(T=0.0) == SV_ERR_ARG
    assert f(target=FAKE + 2) == SV_ERR_ALIGN
    assert f(dtype=9) == SV_ERR_DTYPE
    assert f(K=2000) == SV_ERR_SIZE
    assert f(events=(ctypes.c_void_p * 2)(), n_events=2) == SV_ERR_ARG
    assert f(events=None, n_events=4) == SV_ERR_ARG
    dbg = lib.spec_verify_filtered_debug
    args = (FAKE, FAKE, FAKE, 2, 3, 64, 1, 1.0, 5, 0.9, 7, 0, FAKE, FAKE, FAKE, 1 << 20, None)
    assert dbg(*args, FAKE, FAKE, FAKE + 2, FAKE, FAKE) == SV_ERR_ALIGN
    assert dbg(*args, FAKE, FAKE, FAKE, FAKE + 1, FAKE) == SV_ERR_ALIGN
    assert dbg(*args, FAKE + 4, FAKE, FAKE, FAKE, FAKE) == SV_ERR_ALIGN


def test_lmhead_host_side_validation(lib):
    """spec_verify_lmhead and sv_lmhead_logits check sizes, pointers and
    alignment before any CUDA call."""
    def f(B=2, K=3, V=64, Dt=64, Dd=32, T=1.0, mode=0, ht=FAKE, wt=FAKE, hd=FAKE, wd=FAKE,
          tokens=FAKE, out=FAKE, ws=FAKE, events=None, n_events=0):
        args = (ht, wt, hd, wd, tokens, B, K, V, Dt, Dd, T, 7, mode, out, FAKE, ws, 1 << 20,
                None)
        if events is None and n_events == 0:
            return lib.spec_verify_lmhead(*args)
        return lib.spec_verify_lmhead_timed(*args, events, n_events)
    assert f(B=0) == SV_OK
    assert f(B=0, ht=None, wt=None, hd=None, wd=None, tokens=None, out=None, ws=None) == SV_OK
    assert f(Dt=12) == SV_ERR_ARG            # rows must be whole 16-byte vectors
    assert f(Dt=0) == SV_ERR_ARG
    assert f(Dd=4) == SV_ERR_ARG
    assert f(mode=1, Dd=4, hd=None, wd=None, ht=FAKE + 2) == SV_ERR_ALIGN  # Dd unused
    assert f(K=0, Dd=0, hd=None, wd=None, tokens=None, ws=None) == SV_ERR_WORKSPACE
    assert f(T=0.0) == SV_ERR_ARG
    assert f(T=float("nan")) == SV_ERR_ARG
    assert f(mode=3) == SV_ERR_ARG
    assert f(K=1025) == SV_ERR_SIZE
    assert f(V=0) == SV_ERR_ARG
    assert f(Dt=1 << 31) == SV_ERR_SIZE
    assert f(ht=None) == SV_ERR_ARG
    assert f(wt=None) == SV_ERR_ARG
    assert f(hd=None) == SV_ERR_ARG
    assert f(wd=None) == SV_ERR_ARG
    assert f(tokens=None) == SV_ERR_ARG
    assert f(out=None) == SV_ERR_ARG
    assert f(ws=None) == SV_ERR_WORKSPACE
    assert f(ws=FAKE + 64) == SV_ERR_WORKSPACE
    assert f(ht=FAKE + 2) == SV_ERR_ALIGN
    assert f(wt=FAKE + 8) == SV_ERR_ALIGN
    assert f(hd=FAKE + 4) == SV_ERR_ALIGN
    assert f(wd=FAKE + 12) == SV_ERR_ALIGN
    assert f(tokens=FAKE + 2) == SV_ERR_ALIGN
    assert f(out=FAKE + 1) == SV_ERR_ALIGN
    assert f(events=(ctypes.c_void_p * 4)(), n_events=4) == SV_ERR_ARG
    assert f(events=None, n_events=5) == SV_ERR_ARG
    # Greedy needs neither the draft head nor a temperature.
    assert f(mode=1, T=-1.0, hd=None, wd=None, Dd=0, ht=FAKE + 2) == SV_ERR_ALIGN
    dbg = lib.spec_verify_lmhead_debug
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, 2, 3, 64, 64, 32, 1.0, 7, 0, FAKE, FAKE, FAKE, 1 << 20,
            None)
    assert dbg(*args, FAKE + 4, FAKE, FAKE, FAKE) == SV_ERR_ALIGN
    assert dbg(*args, FAKE, FAKE, FAKE + 2, FAKE) == SV_ERR_ALIGN
    assert dbg(*args, FAKE, FAKE, FAKE, FAKE + 1) == SV_ERR_ALIGN
    sg = lib.spec_verify_gated
    sargs = (FAKE, FAKE, FAKE, 2, 3, 64, 1, 1.0, 5, 0.9, 7, 0, FAKE, FAKE, FAKE, 1 << 20, None,
             FAKE)
    assert sg(*sargs, 1, None) == SV_ERR_ARG
    assert sg(*sargs, 3, FAKE) == SV_ERR_ARG
    assert sg(*sargs, 0, FAKE) == SV_ERR_ARG
    assert sg(*sargs, 2, FAKE + 2) == SV_ERR_ALIGN
    gated = lib.spec_verify_lmhead_gated
    gargs = (FAKE, FAKE, FAKE, FAKE, FAKE, 2, 3, 64, 64, 32, 1.0, 7, 0, FAKE, FAKE, FAKE, 1 << 20,
             None, FAKE)
    assert gated(*gargs, None) == SV_ERR_ARG
    assert gated(*gargs, FAKE + 2) == SV_ERR_ALIGN
    g = lib.sv_lmhead_logits
    assert g(FAKE, FAKE, 0, 64, 100, FAKE, FAKE, None) == SV_OK
    assert g(FAKE, FAKE, 4, 60, 100, FAKE, FAKE, None) == SV_ERR_ARG
    assert g(FAKE, FAKE, 4, 64, 0, FAKE, FAKE, None) == SV_ERR_ARG
    assert g(FAKE, FAKE, -1, 64, 10, FAKE, FAKE, None) == SV_ERR_ARG
    assert g(FAKE, FAKE, 1 << 31, 64, 10, FAKE, FAKE, None) == SV_ERR_SIZE
    assert g(None, FAKE, 4, 64, 10, FAKE, FAKE, None) == SV_ERR_ARG
    assert g(FAKE, FAKE, 4, 64, 10, FAKE, None, None) == SV_ERR_ARG
    assert g(FAKE + 2, FAKE, 4, 64, 10, FAKE, FAKE, None) == SV_ERR_ALIGN
    assert g(FAKE, FAKE + 8, 4, 64, 10, FAKE, FAKE, None) == SV_ERR_ALIGN
    assert g(FAKE, FAKE, 4, 64, 10, FAKE + 2, FAKE, None) == SV_ERR_ALIGN


def test_greedy_ignores_temperature_and_draft(lib):
    # greedy: T and draft_logits are unused, so only later checks can fail
    assert call(lib, mode=1, T=-3.0, draft=None, target=FAKE + 2) == SV_ERR_ALIGN


def test_zero_drafts_need_no_tokens_or_draft(lib):
    assert call(lib, K=0, draft=None, tokens=None, target=FAKE + 4) == SV_ERR_ALIGN


def test_timed_needs_four_events(lib):
    ev = (ctypes.c_void_p * 2)()
    rc = lib.spec_verify_timed(FAKE, FAKE, FAKE, 2, 3, 64, 1, 1.0, 7, 0, FAKE, FAKE, FAKE,
                               1 << 20, None, ev, 2)
    assert rc == SV_ERR_ARG
    rc = lib.spec_verify_timed(FAKE, FAKE, FAKE, 2, 3, 64, 1, 1.0, 7, 0, FAKE, FAKE, FAKE,
                               1 << 20, None, None, 4)
    assert rc == SV_ERR_ARG


def test_debug_outputs_must_be_aligned(lib):
    rc = lib.spec_verify_debug(FAKE, FAKE, FAKE, 2, 3, 64, 1, 1.0, 7, 0, FAKE, FAKE, FAKE,
                               1 << 20, None, FAKE + 4, None, None, None)
    assert rc == SV_ERR_ALIGN


def test_host_entry_validates_before_copying(lib):
    n = ctypes.c_size_t(0)
    assert lib.sv_host_staging_bytes(2, 3, 64, 9, 0, ctypes.byref(n)) == SV_ERR_DTYPE
    assert lib.sv_host_staging_bytes(2, 3, 64, 1, 0, None) == SV_ERR_ARG
    assert lib.sv_workspace_bytes(2, 3, 0, 1, 0, ctypes.byref(n)) == SV_ERR_ARG
    assert lib.spec_verify_host(FAKE, FAKE, FAKE, 2, 2000, 64, 1, 1.0, 7, 0, FAKE, FAKE, FAKE,
                                1 << 20, None) == SV_ERR_SIZE


def test_philox_entry_validates_on_the_host(lib):
    """sv_philox checks its arguments before any CUDA call (no GPU needed)."""
    assert lib.sv_philox(0, None, None, 0, None) == 0      # nothing to do
    assert lib.sv_philox(0, None, None, -1, None) == -1    # SV_ERR_ARG
    assert lib.sv_philox(0, None, None, 4, None) == -1     # NULL pointers
    assert lib.sv_philox(0, 16, 32, 1 << 40, None) == -6   # SV_ERR_SIZE
    assert lib.sv_philox(0, 16 + 4, 32, 1, None) == -3     # SV_ERR_ALIGN


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No CPU fallback: a missing library is an error, not a silent detour."""
    from speculative_decoding_verification_66_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(_lib.LibraryMissing):
        _lib.load()


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_verification_66_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "sv_oracle" not in text and "svo_" not in text, f
