"""Parity of spec_verify_early_exit (phases that read a sequence's rows only up
to its first rejection) with the float64 oracle. The oracle is the same as
for spec_verify: reading fewer rows changes no result, except that values in
rows after the emitted position cannot invalidate a sequence.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_66_gb300 as sv
from parity_util import compare, flag_count_plausible
from speculative_decoding_verification_66_gb300.workloads import (WORKLOADS, make_inputs,
                                                                   to_host_arrays)

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()
    torch.cuda.set_device(0)


def ee_run(inputs, wl, seed):
    out, nacc = sv.spec_verify_early_exit(inputs["target"], inputs["draft"], inputs["tokens"],
                                          wl.temperature, seed, wl.mode)
    torch.cuda.synchronize()
    return {"out_tokens": out.cpu().numpy(), "num_accepted": nacc.cpu().numpy()}


def oracle_run(host, wl, seed, seq_range=None):
    t, d, x = host
    mode = oracle.SAMPLE if wl.mode == "sample" else oracle.GREEDY
    kw = {} if seq_range is None else {"seq_range": seq_range}
    return oracle.verify(t, d, x, wl.temperature, seed, mode, threads=THREADS, **kw)


def check(wl, seed, device_inputs=None, rows=None):
    inputs = device_inputs if device_inputs is not None else make_inputs(wl, seed, "cuda")
    host = to_host_arrays(inputs)
    g = ee_run(inputs, wl, 0x5EED0000 + seed)
    if rows is None:
        orc = oracle_run(host, wl, 0x5EED0000 + seed)
        idx = list(range(wl.B))
    else:
        orc = None
        for lo, hi in rows:
            r = oracle_run(host, wl, 0x5EED0000 + seed, (lo, hi))
            if orc is None:
                orc = r
            else:
                for k in orc:
                    orc[k][lo:hi] = r[k][lo:hi]
        idx = [b for lo, hi in rows for b in range(lo, hi)]
    bad_g = g["num_accepted"][idx] < 0
    bad_o = orc["seq_status"][idx] != 0
    assert np.array_equal(bad_g, bad_o), "invalid sequences differ"
    g["seq_status"] = np.where(g["num_accepted"] < 0, orc["seq_status"], 0)
    return compare(g, orc, host[2], wl.K, wl.V, rows=idx, greedy=wl.mode == "greedy",
                   check_stats=False)


SIZES = {
    "small_f32": {},
    "spiky_bf16": {},
    "llama3_bf16": {"B": 12},
    "qwen_long_bf16": {"B": 6},
    "greedy_bf16": {"B": 48},
}


@pytest.mark.parametrize("name", sorted(SIZES))
@pytest.mark.parametrize("seed", [0, 1])
def test_early_exit_parity(name, seed):
    wl = WORKLOADS[name].resized(**SIZES[name])
    st = check(wl, seed)
    assert flag_count_plausible(st["flagged_decisions"], st["decisions"]), st


@pytest.mark.parametrize("name", ["llama3_bf16", "qwen_long_bf16", "greedy_bf16"])
def test_early_exit_full_size_sampled_rows(name):
    wl = WORKLOADS[name]
    B = wl.B
    st = check(wl, 7, rows=[(0, 3), (B // 2 - 1, B // 2 + 1), (B - 3, B)])
    assert st["decisions"] > 0


@pytest.mark.parametrize("V,dtype", [(1, "bf16"), (7, "bf16"), (33, "f32"), (50257, "bf16"),
                                     (8191, "f32"), (151936, "bf16")])
@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_early_exit_ragged_vocab(V, dtype, mode):
    base = WORKLOADS["small_f32"] if mode == "sample" else WORKLOADS["greedy_bf16"]
    check(base.resized(B=5, K=3, V=V, dtype=dtype, mode=mode, temperature=0.9), 3)


@pytest.mark.parametrize("K", [0, 1, 2, 3, 7, 16, 40, 1024])
@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_early_exit_draft_counts(K, mode):
    """Phases of 1, 2, 4, ... positions: K = 0 (bonus only), phase ends that
    fall on K, and runs that need every phase."""
    base = WORKLOADS["small_f32"] if mode == "sample" else WORKLOADS["greedy_bf16"]
    check(base.resized(B=6, K=K, V=3000, dtype="bf16", mode=mode), 11)


def test_early_exit_every_phase_runs_when_all_accept():
    wl = WORKLOADS["spiky_bf16"].resized(B=16, K=9, V=1000)
    inputs = make_inputs(wl, 5, "cuda")
    inputs["draft"] = inputs["target"][:, :wl.K].contiguous()  # p = q: every draft accepted
    check(wl, 5, device_inputs=inputs)
    g = ee_run(inputs, wl, 99)
    assert (g["num_accepted"] == wl.K).all()


def test_early_exit_matches_full_pass():
    """Outside flagged near-ties the two entry points give the same tokens."""
    wl = WORKLOADS["llama3_bf16"].resized(B=32)
    inputs = make_inputs(wl, 9, "cuda")
    full_out, full_n = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"],
                                      wl.temperature, 4242, wl.mode)
    g = ee_run(inputs, wl, 4242)
    same = (full_n.cpu().numpy() == g["num_accepted"]) & \
        np.all(full_out.cpu().numpy() == g["out_tokens"], axis=1)
    assert same.mean() >= 0.9  # differences only where the oracle flags a near-tie
    check(wl, 9, device_inputs=inputs)


def test_early_exit_invalid_inputs():
    """Bad draft tokens anywhere invalidate the sequence; non-finite rows do
    when they lie at or before the emitted position."""
    wl = WORKLOADS["small_f32"].resized(B=8, K=3, V=700)
    inputs = make_inputs(wl, 21, "cuda")
    t, x = inputs["target"], inputs["tokens"]
    t[2, 0, 17] = float("nan")   # row 0 is always read
    t[3, :, :] = float("-inf")
    x[5, 2] = wl.V               # a bad token at the last position
    x[6, 0] = -4
    g = ee_run(inputs, wl, 0x5EED0000 + 21)
    assert list(g["num_accepted"][[2, 3, 5, 6]]) == [-1, -1, -1, -1]
    check(wl, 21, device_inputs=inputs)


def test_early_exit_ignores_rows_after_the_emitted_position():
    wl = WORKLOADS["spiky_bf16"].resized(B=32, K=4)
    inputs = make_inputs(wl, 13, "cuda")
    clean = {k: v.clone() for k, v in inputs.items()}
    g = ee_run(inputs, wl, 777)
    early = np.nonzero(g["num_accepted"] == 0)[0]
    assert early.size > 0
    b = int(early[0])
    inputs["target"][b, wl.K, 3] = float("nan")  # the bonus row: never read for b
    inputs["draft"][b, wl.K - 1, 5] = float("inf")
    g2 = ee_run(inputs, wl, 777)
    assert g2["num_accepted"][b] == 0
    assert np.array_equal(g2["out_tokens"], g["out_tokens"])
    host = to_host_arrays(clean)
    orc = oracle_run(host, wl, 777)
    assert orc["num_accepted"][b] == 0 or orc["accept_margin"][b][0] < 1e-5


def test_early_exit_empty_batch_and_repeats():
    wl = WORKLOADS["spiky_bf16"].resized(B=0)
    inputs = make_inputs(wl, 0, "cuda")
    out, nacc = sv.spec_verify_early_exit(inputs["target"], inputs["draft"], inputs["tokens"],
                                          1.0, 1)
    torch.cuda.synchronize()
    assert out.shape == (0, wl.K + 1) and nacc.shape == (0,)
    wl = WORKLOADS["qwen_long_bf16"].resized(B=8)
    inputs = make_inputs(wl, 4, "cuda")
    a = ee_run(inputs, wl, 5)
    b = ee_run(inputs, wl, 5)
    assert np.array_equal(a["out_tokens"], b["out_tokens"])
    assert np.array_equal(a["num_accepted"], b["num_accepted"])
