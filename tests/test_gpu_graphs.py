"""The verification entry points inside CUDA graphs.

A decode loop calls verification once per step with the same shapes, so a
caller can capture the launches once and replay them: no host work per step.
These tests capture each entry point with torch.cuda.graph, copy new inputs
into the captured buffers, replay, and compare with ordinary calls on the same
inputs, which must give identical tokens and counts.
"""
import pytest
import torch

import speculative_decoding_verification_66_gb300 as sv
from speculative_decoding_verification_66_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()
    torch.cuda.set_device(0)


def _call(entry, inp, wl, seed, **kw):
    if entry == "full":
        return sv.spec_verify(inp["target"], inp["draft"], inp["tokens"], wl.temperature, seed,
                              wl.mode, **kw)
    if entry == "early_exit":
        return sv.spec_verify_early_exit(inp["target"], inp["draft"], inp["tokens"],
                                         wl.temperature, seed, wl.mode, **kw)
    return sv.spec_verify_filtered(inp["target"], inp["draft"], inp["tokens"], wl.temperature,
                                   40, 0.9, seed, wl.mode, **kw)


def test_lmhead_capture_and_replay():
    """spec_verify_lmhead in a graph: tensor maps are kernel parameters, so the
    captured launches replay on whatever the captured buffers hold."""
    from speculative_decoding_verification_66_gb300.workloads import (LM_WORKLOADS,
                                                                       make_lmhead_inputs)
    lw = LM_WORKLOADS["lm_small"]
    static = make_lmhead_inputs(lw, 0, "cuda")
    out = torch.empty((lw.B, lw.K + 1), dtype=torch.int32, device="cuda")
    nacc = torch.empty((lw.B,), dtype=torch.int32, device="cuda")
    ws = torch.empty(sv.sv_lmhead_workspace_bytes(lw.B, lw.K, lw.V, lw.d_target, lw.d_draft,
                                                  lw.mode), dtype=torch.uint8, device="cuda")

    def call(inp, **kw):
        return sv.spec_verify_lmhead(inp["hidden_t"], inp["weight_t"], inp["hidden_d"],
                                     inp["weight_d"], inp["tokens"], lw.temperature, 21, lw.mode,
                                     **kw)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            call(static, out_tokens=out, num_accepted=nacc, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(static, out_tokens=out, num_accepted=nacc, workspace=ws)
    for seed in (1, 2):
        fresh = make_lmhead_inputs(lw, seed, "cuda")
        for k in static:
            static[k].copy_(fresh[k])
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_n = call(fresh)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), seed
        assert torch.equal(nacc, ref_n), seed


@pytest.mark.parametrize("entry", ["full", "early_exit", "filtered"])
@pytest.mark.parametrize("name", ["small_f32", "spiky_bf16", "greedy_bf16"])
def test_capture_and_replay(entry, name):
    wl = WORKLOADS[name]
    if entry == "filtered" and wl.mode == "greedy":
        pytest.skip("greedy ignores the cuts")
    static = make_inputs(wl, 0, "cuda")
    out = torch.empty((wl.B, wl.K + 1), dtype=torch.int32, device="cuda")
    nacc = torch.empty((wl.B,), dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm up outside the capture (workspace, attributes)
        for _ in range(2):
            _call(entry, static, wl, 11, out_tokens=out, num_accepted=nacc)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(entry, static, wl, 11, out_tokens=out, num_accepted=nacc)
    for seed in (1, 2, 3):
        fresh = make_inputs(wl, seed, "cuda")
        for k in static:
            if static[k] is not None:
                static[k].copy_(fresh[k])
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_n = _call(entry, fresh, wl, 11)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), (entry, name, seed)
        assert torch.equal(nacc, ref_n), (entry, name, seed)


def test_replay_latency_small_batch():
    """Replaying a captured call removes the per-call host work; report the
    device time per replayed call for the small configuration."""
    wl = WORKLOADS["small_f32"]
    static = make_inputs(wl, 0, "cuda")
    out = torch.empty((wl.B, wl.K + 1), dtype=torch.int32, device="cuda")
    nacc = torch.empty((wl.B,), dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _call("full", static, wl, 5, out_tokens=out, num_accepted=nacc)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(10):
            _call("full", static, wl, 5, out_tokens=out, num_accepted=nacc)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(20):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / 200
    print(f"small_f32: {us:.2f} us per call replayed from a graph")
    assert us > 0
