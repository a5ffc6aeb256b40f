"""spec_verify_static: verification for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc. One case is code inside a host framework
that owns all device memory through its own pool, where an extra allocation
fails or breaks the pool's accounting. Another is code on a latency-critical
path, where allocating or freeing would synchronise the device.
spec_verify_static serves them with a fixed scratch array inside the library
instead of a caller-provided workspace.

These tests call that entry point through the C ABI and check, on two calls in
a row, that it returns exactly what spec_verify returns with an ordinary
workspace (the outputs are integers: the comparison is exact). The file is
named to be collected last.
"""
import ctypes

import pytest
import torch

import speculative_decoding_verification_66_gb300 as sv
from speculative_decoding_verification_66_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

SV_ERR_SIZE = -6


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_static(lib, inp, wl, seed, out, nacc, stream):
    m = 0 if wl.mode == "sample" else 1
    return lib.spec_verify_static(
        _ptr(inp["target"]), _ptr(inp["draft"]), _ptr(inp["tokens"]), wl.B, wl.K, wl.V,
        1 if wl.dtype == "bf16" else 0, float(wl.temperature), seed, m, _ptr(out), _ptr(nacc),
        ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("name", ["llama3_bf16", "greedy_bf16", "small_f32"])
def test_static_scratch_matches_workspace_call(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    lib = sv.load()
    wl = WORKLOADS[name]
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((0x5EED0001, 0x5EED0002)):  # two calls in a row
        inp = make_inputs(wl, 40 + call, "cuda")
        out_s = torch.full((wl.B, wl.K + 1), -9, dtype=torch.int32, device="cuda")
        nacc_s = torch.full((wl.B,), -9, dtype=torch.int32, device="cuda")
        assert call_static(lib, inp, wl, seed, out_s, nacc_s, stream) == 0
        out_w, nacc_w = sv.spec_verify(inp["target"], inp["draft"], inp["tokens"],
                                       wl.temperature, seed, wl.mode)
        torch.cuda.synchronize()
        assert torch.equal(out_s, out_w), f"call {call}: out_tokens differ"
        assert torch.equal(nacc_s, nacc_w), f"call {call}: num_accepted differ"
        assert (nacc_s >= 0).all()


def test_static_scratch_rejects_problems_beyond_its_size():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    lib = sv.load()
    # 400k one-token sequences need more than the 8 MiB scratch (32 B of
    # per-sequence state each, plus the rest); the call must refuse before
    # touching any buffer, so no inputs are allocated here.
    need = sv.sv_workspace_bytes(400_000, 0, 1, torch.bfloat16, "sample")
    assert need > (8 << 20)
    rc = lib.spec_verify_static(None, None, None, 400_000, 0, 1, 1, 1.0, 1, 0, None, None, None)
    assert rc == SV_ERR_SIZE
