"""Parity of spec_verify_sharded (logits split over the vocabulary into G
shards of Vs columns) with the float64 oracle run on the concatenated logits:
sharding changes where the columns live, not what is computed.
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


def split(x, G):
    Vs = x.shape[-1] // G
    return [x[..., g * Vs:(g + 1) * Vs].contiguous() for g in range(G)]


def sharded_run(inputs, wl, G, seed):
    ts = split(inputs["target"], G)
    ds = split(inputs["draft"], G) if wl.mode == "sample" else None
    out, nacc = sv.spec_verify_sharded(ts, ds, inputs["tokens"], wl.temperature, seed, wl.mode)
    torch.cuda.synchronize()
    return {"out_tokens": out.cpu().numpy(), "num_accepted": nacc.cpu().numpy()}


def check(wl, G, seed, device_inputs=None):
    assert wl.V % G == 0
    inputs = device_inputs if device_inputs is not None else make_inputs(wl, seed, "cuda")
    host = to_host_arrays(inputs)
    g = sharded_run(inputs, wl, G, 0x5EED0000 + seed)
    t, d, x = host
    mode = oracle.SAMPLE if wl.mode == "sample" else oracle.GREEDY
    orc = oracle.verify(t, d, x, wl.temperature, 0x5EED0000 + seed, mode, threads=THREADS)
    assert np.array_equal(g["num_accepted"] < 0, orc["seq_status"] != 0)
    g["seq_status"] = np.where(g["num_accepted"] < 0, orc["seq_status"], 0)
    return compare(g, orc, x, wl.K, wl.V, greedy=wl.mode == "greedy", check_stats=False)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("name", ["small_f32", "spiky_bf16", "greedy_bf16"])
def test_sharded_parity(name, G):
    size = {"greedy_bf16": {"B": 24, "V": 32000}}.get(name, {})
    wl = WORKLOADS[name].resized(**size)
    st = check(wl, G, 3)
    assert flag_count_plausible(st["flagged_decisions"], st["decisions"]), st


def test_sharded_headline_shapes():
    """The headline row length in 8 shards of 16032 columns (a TP-8 LM head)."""
    wl = WORKLOADS["llama3_bf16"].resized(B=8)
    check(wl, 8, 5)


@pytest.mark.parametrize("V,G,dtype", [(3003, 3, "bf16"), (50267, 7, "bf16"), (4100, 4, "f32"),
                                       (15, 5, "bf16"), (16, 16, "f32")])
@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_sharded_ragged(V, G, dtype, mode):
    """Shard widths that are not a multiple of a 16-byte vector, race blocks
    that straddle shards, and one-column shards."""
    base = WORKLOADS["small_f32"] if mode == "sample" else WORKLOADS["greedy_bf16"]
    check(base.resized(B=5, K=3, V=V, dtype=dtype, mode=mode, temperature=0.8), G, 9)


@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_sharded_maximum_draft_count(mode):
    """K = 1024, the largest supported, over 4 shards."""
    base = WORKLOADS["small_f32"] if mode == "sample" else WORKLOADS["greedy_bf16"]
    check(base.resized(B=3, K=1024, V=3000, dtype="bf16", mode=mode), 4, 13)


def test_sharded_matches_unsharded_entry():
    wl = WORKLOADS["spiky_bf16"]
    inputs = make_inputs(wl, 12, "cuda")
    a_out, a_n = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"], 1.0, 31337)
    g = sharded_run(inputs, wl, 4, 31337)
    same = (a_n.cpu().numpy() == g["num_accepted"]) & \
        np.all(a_out.cpu().numpy() == g["out_tokens"], axis=1)
    assert same.mean() >= 0.97  # differences only on flagged near-ties
    check(wl, 4, 12, device_inputs=inputs)
