"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Discrete results (accepted counts, tokens, argmaxes, status) are compared
exactly, apart from the decisions the oracle flags as near-ties (see
parity_util). Normalisers and log-ratios are compared to 1e-5 relative.
Inputs come from the seeded workload generators, on the device; the oracle
reads host copies of the same tensors.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_66_gb300 as sv
from parity_util import compare, flag_count_plausible, oracle_flag_counts
from speculative_decoding_verification_66_gb300.workloads import (WORKLOADS, Workload,
                                                                   make_inputs, to_host_arrays)

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()
    torch.cuda.set_device(0)


def gpu_debug(inputs, wl, seed):
    r = sv.spec_verify_debug(inputs["target"], inputs["draft"], inputs["tokens"], wl.temperature,
                             seed, wl.mode)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


def oracle_run(host, wl, seed, ranges=None):
    t, d, x = host
    mode = oracle.SAMPLE if wl.mode == "sample" else oracle.GREEDY
    if ranges is None:
        return oracle.verify(t, d, x, wl.temperature, seed, mode, threads=THREADS)
    merged = None
    for lo, hi in ranges:
        r = oracle.verify(t, d, x, wl.temperature, seed, mode, threads=THREADS, seq_range=(lo, hi))
        if merged is None:
            merged = r
        else:
            for k in merged:
                merged[k][lo:hi] = r[k][lo:hi]
    return merged


def check(wl, seed, rows=None, device_inputs=None):
    inputs = device_inputs if device_inputs is not None else make_inputs(wl, seed, "cuda")
    host = to_host_arrays(inputs)
    gpu = gpu_debug(inputs, wl, 0x5EED0000 + seed)
    ranges = None
    if rows is not None:
        ranges = rows
        rows = [b for lo, hi in ranges for b in range(lo, hi)]
    orc = oracle_run(host, wl, 0x5EED0000 + seed, ranges)
    st = compare(gpu, orc, host[2], wl.K, wl.V, rows=rows, greedy=wl.mode == "greedy")
    if rows is None:
        st["oracle_decisions"], st["oracle_flagged"] = oracle_flag_counts(orc, wl.K)
    return st


# Sizes the oracle finishes in seconds; each still spans many pass-1 tiles.
TEST_SIZES = {
    "small_f32": {},
    "spiky_bf16": {},
    "llama3_bf16": {"B": 12},
    "qwen_long_bf16": {"B": 6},
    "greedy_bf16": {"B": 48},
}


@pytest.mark.parametrize("name", sorted(TEST_SIZES))
@pytest.mark.parametrize("seed", [0, 1])
def test_workload_parity(name, seed):
    wl = WORKLOADS[name].resized(**TEST_SIZES[name])
    st = check(wl, seed)
    assert flag_count_plausible(st["oracle_flagged"], st["oracle_decisions"]), st


# Ragged vocabularies: rows not 16-byte aligned, tails shorter than a vector,
# vocabularies smaller than one vector and one tile.
@pytest.mark.parametrize("V,dtype", [(1, "bf16"), (2, "f32"), (7, "bf16"), (33, "f32"),
                                     (50257, "bf16"), (8191, "f32"), (16391, "bf16"),
                                     (4100, "f32"), (151936, "bf16")])
@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_ragged_vocab(V, dtype, mode):
    base = WORKLOADS["small_f32"] if mode == "sample" else WORKLOADS["greedy_bf16"]
    wl = base.resized(B=5, K=3, V=V, dtype=dtype, mode=mode, temperature=0.9)
    check(wl, 3)


@pytest.mark.parametrize("K", [0, 1, 2, 16, 40, 1024])
@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_draft_counts(K, mode):
    base = WORKLOADS["small_f32"] if mode == "sample" else WORKLOADS["greedy_bf16"]
    wl = base.resized(B=3, K=K, V=3000, dtype="bf16", mode=mode)
    check(wl, 11)


def test_empty_batch():
    wl = WORKLOADS["spiky_bf16"].resized(B=0)
    inputs = make_inputs(wl, 0, "cuda")
    out, nacc = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"], 1.0, 1)
    torch.cuda.synchronize()
    assert out.shape == (0, wl.K + 1) and nacc.shape == (0,)


def test_p_equals_q_accepts_all_and_takes_bonus():
    wl = WORKLOADS["spiky_bf16"].resized(B=16, K=5, V=1000)
    inputs = make_inputs(wl, 5, "cuda")
    inputs["draft"] = inputs["target"][:, :wl.K].contiguous()
    st = check(wl, 5, device_inputs=inputs)
    r = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"], 1.0, 99)
    assert (r[1].cpu() == wl.K).all()
    assert st["decisions"] > 0


def test_masked_logits_and_invalid_rows():
    """-inf masking is valid; NaN / +inf / all -inf rows and out-of-range
    tokens invalidate exactly their sequence, as in the oracle."""
    wl = WORKLOADS["small_f32"].resized(B=8, K=3, V=700)
    inputs = make_inputs(wl, 21, "cuda")
    t, d, x = inputs["target"], inputs["draft"], inputs["tokens"]
    t[0, 1, ::3] = float("-inf")            # masking only: still valid
    d[1, 0, 5:] = float("-inf")
    x[1, 0] = 2
    t[2, 2, 17] = float("nan")
    t[3, :, :] = float("-inf")
    d[4, 2, 600] = float("inf")
    x[5, 1] = wl.V
    x[6, 0] = -4
    st = check(wl, 21, device_inputs=inputs)
    g = gpu_debug(inputs, wl, 0x5EED0000 + 21)
    assert list(g["seq_status"][:8]) == [0, 0, 2, 2, 2, 1, 1, 0]
    assert st["decisions"] > 0


def test_greedy_nan_and_ties():
    wl = WORKLOADS["greedy_bf16"].resized(B=6, K=4, V=5000)
    inputs = make_inputs(wl, 2, "cuda")
    t = inputs["target"]
    t[0] = torch.randint(-2, 2, t[0].shape, device="cuda").to(t.dtype)  # many exact ties
    t[1, 2, 4000] = float("nan")
    t[2] = float("-inf")
    inputs["tokens"][0] = t[0, :4].float().argmax(dim=-1).to(torch.int32)
    check(wl, 2, device_inputs=inputs)


def test_repeat_runs_are_identical():
    wl = WORKLOADS["spiky_bf16"]
    inputs = make_inputs(wl, 4, "cuda")
    a = gpu_debug(inputs, wl, 123)
    b = gpu_debug(inputs, wl, 123)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k
    c = gpu_debug(inputs, wl, 124)
    assert not np.array_equal(a["out_tokens"], c["out_tokens"])


def test_host_entry_matches_device_entry():
    wl = WORKLOADS["spiky_bf16"]
    inputs = make_inputs(wl, 8, "cuda")
    out_d, nacc_d = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"], 1.0, 42)
    torch.cuda.synchronize()
    ht = inputs["target"].cpu().pin_memory()
    hd = inputs["draft"].cpu().pin_memory()
    hx = inputs["tokens"].cpu().pin_memory()
    out_h, nacc_h = sv.spec_verify_host(ht, hd, hx, 1.0, 42)
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(nacc_h, nacc_d.cpu())


def test_timed_entry_matches_and_records_events():
    wl = WORKLOADS["small_f32"]
    inputs = make_inputs(wl, 9, "cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    out_t, nacc_t = sv.spec_verify_timed(inputs["target"], inputs["draft"], inputs["tokens"], ev,
                                         1.0, 5)
    out, nacc = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"], 1.0, 5)
    torch.cuda.synchronize()
    assert torch.equal(out_t, out) and torch.equal(nacc_t, nacc)
    assert ev[0].elapsed_time(ev[1]) > 0 and ev[0].elapsed_time(ev[3]) >= ev[0].elapsed_time(ev[1])


def test_stream_ordering_on_a_side_stream():
    wl = WORKLOADS["spiky_bf16"]
    inputs = make_inputs(wl, 10, "cuda")
    ref = gpu_debug(inputs, wl, 3)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, nacc = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"], 1.0, 3)
    s.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref["out_tokens"])


def test_binding_rejects_bad_tensors():
    wl = WORKLOADS["spiky_bf16"].resized(B=2, V=64)
    inputs = make_inputs(wl, 0, "cuda")
    with pytest.raises(ValueError):
        sv.spec_verify(inputs["target"].transpose(1, 2), inputs["draft"], inputs["tokens"])
    with pytest.raises(ValueError):
        sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"].long())
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"], temperature=0.0)
    bad = torch.empty(2 * 5 * 64 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(2, 5, 64)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify(bad, inputs["draft"], inputs["tokens"])


@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_timeout_path(mode):
    """Pass 1's timeout path, without a fault: its producers wait on a device
    flag that nothing sets. The wait runs out (about 2 s), the consumers mark
    their rows as timed out, and every sequence comes back as SV_SEQ_TIMEOUT.
    The context stays usable: an ordinary call afterwards still matches the
    oracle, and a gated call whose flag is already set matches spec_verify."""
    base = WORKLOADS["small_f32"] if mode == "sample" else WORKLOADS["greedy_bf16"]
    wl = base.resized(B=6, K=3, V=3000, dtype="bf16", mode=mode)
    inputs = make_inputs(wl, 4, "cuda")
    gate = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = sv.spec_verify_gated(inputs["target"], inputs["draft"], inputs["tokens"], gate,
                             wl.temperature, 9, mode)
    torch.cuda.synchronize()
    assert (r["seq_status"].cpu() == sv.SV_SEQ_TIMEOUT).all()
    assert (r["num_accepted"].cpu() == -1).all() and (r["out_tokens"].cpu() == -1).all()
    check(wl, 4, device_inputs=inputs)
    gate.fill_(1)
    r = sv.spec_verify_gated(inputs["target"], inputs["draft"], inputs["tokens"], gate,
                             wl.temperature, 9, mode)
    out, nacc = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"],
                               wl.temperature, 9, mode)
    torch.cuda.synchronize()
    assert (r["seq_status"].cpu() == 0).all()
    assert torch.equal(r["out_tokens"], out) and torch.equal(r["num_accepted"], nacc)


def test_sampler_timeout_path():
    """The sampler's timeout path, without a fault: its streaming warps wait on
    a device flag that nothing sets. They mark their slices with NaN block
    sums, and the race kernel reports every sequence as SV_SEQ_TIMEOUT; pass 1
    and the scan ran normally. An ordinary call afterwards still matches the
    oracle."""
    wl = WORKLOADS["small_f32"].resized(B=6, K=3, V=3000, dtype="bf16")
    inputs = make_inputs(wl, 6, "cuda")
    gate = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = sv.spec_verify_gated(inputs["target"], inputs["draft"], inputs["tokens"], gate,
                             wl.temperature, 9, "sample", stage=2)
    torch.cuda.synchronize()
    assert (r["seq_status"].cpu() == sv.SV_SEQ_TIMEOUT).all()
    assert (r["num_accepted"].cpu() == -1).all() and (r["out_tokens"].cpu() == -1).all()
    check(wl, 6, device_inputs=inputs)
