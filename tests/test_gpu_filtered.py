"""Parity of spec_verify_filtered (top-k / top-p applied to the target and the
draft row of every position) with the float64 oracle's filtered verification.

Thresholds are integer work on the logits' order, so they must match exactly;
a top-p boundary that the oracle puts within 1e-5 (relative) of top_p flags
the decisions that use its row, like a near-tie of the acceptance draw.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_66_gb300 as sv
from parity_util import compare
from speculative_decoding_verification_66_gb300.workloads import (WORKLOADS, draw_from_logits,
                                                                   make_inputs, to_host_arrays)

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()
    torch.cuda.set_device(0)


def f_run(inputs, wl, seed, top_k, top_p):
    out, nacc = sv.spec_verify_filtered(inputs["target"], inputs["draft"], inputs["tokens"],
                                        wl.temperature, top_k, top_p, seed, wl.mode)
    torch.cuda.synchronize()
    return {"out_tokens": out.cpu().numpy(), "num_accepted": nacc.cpu().numpy()}


def f_debug(inputs, wl, seed, top_k, top_p):
    r = sv.spec_verify_filtered_debug(inputs["target"], inputs["draft"], inputs["tokens"],
                                      wl.temperature, top_k, top_p, seed, wl.mode)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


def check_rows(g, orc, idx, K):
    """Per-row thresholds: equal to the oracle's, or the oracle's top-p
    boundary lies within the near-tie band. Where they are equal the kept
    normalisers agree to 1e-5 and the row needs no flag; the returned oracle
    dict keeps the filter flags of the other rows only."""
    orc = dict(orc)
    fm_t = orc["filter_margin_t"].copy()
    fm_d = orc["filter_margin_d"].copy()
    n_rows = n_diff = 0
    for b in idx:
        if orc["seq_status"][b] != 0:
            continue
        for i in range(2 * K + 1):
            tgt = i <= K
            gi = i if tgt else i - K - 1
            gthr = float((g["thr_t"] if tgt else g["thr_d"])[b, gi])
            othr = float(orc["filter_thr"][b, i])
            margin = (fm_t if tgt else fm_d)[b, gi]
            n_rows += 1
            if gthr == othr:
                glse = (g["lse_t"] if tgt else g["lse_d"])[b, gi]
                olse = (orc["lse_t"] if tgt else orc["lse_d"])[b, gi] + orc["filter_log_mass"][b, i]
                assert abs(glse - olse) <= 1e-5 * max(1.0, abs(olse)), (b, i, glse, olse)
                (fm_t if tgt else fm_d)[b, gi] = np.inf
            else:
                n_diff += 1
                assert margin < 1e-5, (b, i, gthr, othr, margin)
    orc["filter_margin_t"], orc["filter_margin_d"] = fm_t, fm_d
    return orc, n_rows, n_diff


def oracle_run(host, wl, seed, top_k, top_p, seq_range=None):
    t, d, x = host
    mode = oracle.SAMPLE if wl.mode == "sample" else oracle.GREEDY
    kw = {} if seq_range is None else {"seq_range": seq_range}
    return oracle.verify(t, d, x, wl.temperature, seed, mode, threads=THREADS, top_k=top_k,
                         top_p=top_p, **kw)


def check(wl, seed, top_k, top_p, device_inputs=None, rows=None):
    inputs = device_inputs if device_inputs is not None else \
        make_inputs(wl, seed, "cuda", top_k=top_k, top_p=top_p)
    host = to_host_arrays(inputs)
    s = 0xF117E000 + seed
    g = f_debug(inputs, wl, s, top_k, top_p) if wl.mode == "sample" else \
        f_run(inputs, wl, s, top_k, top_p)
    if rows is None:
        orc = oracle_run(host, wl, s, top_k, top_p)
        idx = list(range(wl.B))
    else:
        orc = None
        for lo, hi in rows:
            r = oracle_run(host, wl, s, top_k, top_p, (lo, hi))
            if orc is None:
                orc = r
            else:
                for k in orc:
                    orc[k][lo:hi] = r[k][lo:hi]
        idx = [b for lo, hi in rows for b in range(lo, hi)]
    bad_g = g["num_accepted"][idx] < 0
    bad_o = orc["seq_status"][idx] != 0
    assert np.array_equal(bad_g, bad_o), "invalid sequences differ"
    if wl.mode == "sample":
        assert np.array_equal(g["seq_status"][idx], orc["seq_status"][idx])
        orc, n_rows, n_diff = check_rows(g, orc, idx, wl.K)
        assert n_diff <= max(2, 0.05 * n_rows), (n_diff, n_rows)
    else:
        g["seq_status"] = np.where(g["num_accepted"] < 0, orc["seq_status"], 0)
    return compare(g, orc, host[2], wl.K, wl.V, rows=idx, greedy=wl.mode == "greedy",
                   check_stats=False), g, orc


CASES = [
    ("small_f32", {}, 50, 1.0),        # fp32: three-level top-k descent
    ("small_f32", {}, 0, 0.9),         # fp32 top-p alone
    ("small_f32", {}, 300, 0.7),       # top-p inside a top-k set
    ("spiky_bf16", {}, 20, 1.0),
    ("spiky_bf16", {}, 0, 0.95),
    ("spiky_bf16", {}, 1, 1.0),        # top-1: p' one-hot at the maximum
    ("spiky_bf16", {}, 64, 0.5),
    ("llama3_bf16", {"B": 12}, 50, 0.9),
    ("llama3_bf16", {"B": 12}, 0, 0.8),
    ("qwen_long_bf16", {"B": 4}, 100, 0.95),
    ("qwen_long_bf16", {"B": 4}, 0, 0.9),    # flat rows: top-p bins refined twice
    ("spiky_bf16", {"B": 16}, 200, 1.0),     # lists of 129..512 keys: block-wide select
    ("spiky_bf16", {"B": 16}, 500, 0.8),
    ("llama3_bf16", {"B": 8}, 1000, 0.9),    # longer lists: radix select on the list
    ("small_f32", {"B": 4}, 1000, 1.0),
    ("spiky_bf16", {"B": 16}, 3000, 1.0),    # k beyond the candidate list: whole-row select
    ("small_f32", {"B": 4}, 4000, 0.8),
]


@pytest.mark.parametrize("name,size,top_k,top_p", CASES)
@pytest.mark.parametrize("seed", [0, 1])
def test_filtered_parity(name, size, top_k, top_p, seed):
    wl = WORKLOADS[name].resized(**size)
    st, _, _ = check(wl, seed, top_k, top_p)
    assert st["flagged_decisions"] <= max(2, 1e-2 * st["decisions"]), st


def test_filtered_full_size_sampled_rows():
    wl = WORKLOADS["llama3_bf16"]
    B = wl.B
    st, _, _ = check(wl, 7, 50, 0.9, rows=[(0, 3), (B // 2 - 1, B // 2 + 1), (B - 3, B)])
    assert st["decisions"] > 0


@pytest.mark.parametrize("V,dtype", [(1, "bf16"), (7, "bf16"), (33, "f32"), (50257, "bf16"),
                                     (8191, "f32"), (151936, "bf16")])
@pytest.mark.parametrize("top_k,top_p", [(5, 1.0), (0, 0.6), (3, 0.9)])
def test_filtered_ragged_vocab(V, dtype, top_k, top_p):
    """Rows that do not start on 16-byte boundaries (head and tail elements),
    vocabularies shorter than k, and single-token rows."""
    wl = WORKLOADS["small_f32"].resized(B=5, K=3, V=V, dtype=dtype, temperature=0.9)
    check(wl, 3, top_k, top_p)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("top_k,top_p", [(7, 1.0), (0, 0.75), (12, 0.6), (2, 1.0)])
def test_filtered_ties_at_the_boundary(dtype, top_k, top_p):
    """Logits on a coarse grid: most boundaries fall inside a run of equal
    values, all of which stay, including -0 next to +0."""
    wl = WORKLOADS["small_f32"].resized(B=24, K=4, V=2000, dtype=dtype)
    inputs = make_inputs(wl, 17, "cuda", top_k=top_k, top_p=top_p)
    for key in ("target", "draft"):
        t = inputs[key].float()
        t = torch.round(t * 2) / 2
        t[t == 0] = torch.where(torch.rand_like(t[t == 0]) < 0.5, -0.0, 0.0)
        inputs[key] = t.to(inputs[key].dtype)
    check(wl, 17, top_k, top_p, device_inputs=inputs)


def test_filtered_masked_vocabulary():
    """-inf logits (a masked vocabulary): top-k larger than the number of
    finite logits keeps them all, and masked tokens never come out."""
    wl = WORKLOADS["spiky_bf16"].resized(B=16, K=3, V=3000)
    inputs = make_inputs(wl, 5, "cuda", top_k=40)
    for key in ("target", "draft"):
        inputs[key][:, :, 100:] = float("-inf")
    inputs["tokens"] = torch.randint(0, 100, inputs["tokens"].shape, device="cuda",
                                     dtype=torch.int32)
    for top_k, top_p in [(40, 1.0), (150, 1.0), (0, 0.9)]:
        _, g, _ = check(wl, 5, top_k, top_p, device_inputs=inputs)
        assert (g["out_tokens"][g["out_tokens"] >= 0] < 100).all()


@pytest.mark.parametrize("top_k,top_p", [(5, 1.0), (5, 0.5), (0, 0.9)])
def test_filtered_many_ties_at_the_top(top_k, top_p):
    """10000 tokens share the maximum: the top-k candidate list overflows and
    the whole-row select takes over; top-p keeps the whole tied group."""
    wl = WORKLOADS["spiky_bf16"].resized(B=6, K=3, V=32000)
    inputs = make_inputs(wl, 23, "cuda", top_k=top_k, top_p=top_p)
    for key in ("target", "draft"):
        inputs[key][:, :, 1000:11000] = inputs[key].float().amax(dim=-1, keepdim=True).to(
            inputs[key].dtype)
    st, g, orc = check(wl, 23, top_k, top_p, device_inputs=inputs)
    assert (g["num_accepted"] >= 0).all()


def _top_block(wl, seed, top_k, top_p, values, step):
    """Inputs whose every row has len(values) logits set to `values`, `step`
    tokens apart, above all the other logits (clamped to 3); tokens drawn
    from the filtered draft rows. A thread share of the group-maxima kernel
    is every 256th 16-byte vector of the row (8 bf16 or 4 float32 logits)."""
    inputs = make_inputs(wl, seed, "cuda", top_k=top_k, top_p=top_p)
    n = len(values)
    for j, key in enumerate(("target", "draft")):
        x = inputs[key].float().clamp(max=3.0)
        pos = torch.arange(n, device="cuda") * step + 3 * j + 1
        x[..., pos] = torch.tensor(values, device="cuda", dtype=torch.float32)
        inputs[key] = x.to(inputs[key].dtype)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    inputs["tokens"] = draw_from_logits(inputs["draft"], wl.temperature, gen, top_k, top_p)
    return inputs


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("top_p", [1.0, 0.9])
@pytest.mark.parametrize("top_k", [1, 31, 32, 33, 63, 64])
def test_filtered_list_of_k_distinct_keys(dtype, top_k, top_p):
    """80 distinct values above the rest of the row, 392 tokens apart (49
    bf16 or 98 float32 vectors: 80 different thread shares either way): the
    k-th largest thread maximum is the k-th of them, so the candidate list
    holds exactly k keys -- across the one-warp select's 32 / 64-key network
    sizes."""
    wl = WORKLOADS["small_f32"].resized(B=4, K=2, V=32000, dtype=dtype)
    values = [8.0 + 0.0625 * i for i in range(80)]
    inputs = _top_block(wl, 41, top_k, top_p, values, 392)
    st, g, orc = check(wl, 41, top_k, top_p, device_inputs=inputs)
    assert (g["num_accepted"] >= 0).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("top_k,top_p", [(5, 1.0), (64, 0.5)])
@pytest.mark.parametrize("m", [32, 33, 64, 65, 128, 129])
def test_filtered_list_of_m_tied_maxima(dtype, m, top_k, top_p):
    """m logits tied at the row maximum, spread over the row: with k <= m the
    bound is the maximum itself and the candidate list is the m ties (two in
    one thread share are read again, not lost) -- across the one-warp
    select's 32 / 64 / 128-key sizes and the hand-over to the CTA select
    above 128; with k = 64 > m = 32 or 33 the list also takes the largest of
    the other logits."""
    wl = WORKLOADS["small_f32"].resized(B=4, K=2, V=32000, dtype=dtype)
    inputs = _top_block(wl, 43, top_k, top_p, [9.0] * m, wl.V // m)
    st, g, orc = check(wl, 43, top_k, top_p, device_inputs=inputs)
    assert (g["num_accepted"] >= 0).all()


@pytest.mark.parametrize("fill", ["max", "-inf", "-5"])
@pytest.mark.parametrize("top_k,top_p", [(0, 0.9), (100, 1.0), (150000, 0.95), (2000, 0.8)])
def test_filtered_value_shared_by_2_16_tokens(fill, top_k, top_p):
    """bfloat16 rows where 70000 tokens share one value (the row maximum, -inf
    or -5): a 16-bit count of that value wraps, the wrap shows in the sum of
    all counts, and the row is counted again with 32-bit counts; top-k up to
    almost V reaches into the shared value from above and below."""
    wl = WORKLOADS["qwen_long_bf16"].resized(B=2, K=2)
    inputs = make_inputs(wl, 29, "cuda", top_k=top_k, top_p=top_p)
    for key in ("target", "draft"):
        x = inputs[key]
        if fill == "max":
            v = x.float().amax(dim=-1, keepdim=True).to(x.dtype)
        else:
            v = torch.full_like(x[..., :1], float(fill))
        x[..., 50000:120000] = v
    gen = torch.Generator(device="cuda")
    gen.manual_seed(29)
    inputs["tokens"] = draw_from_logits(inputs["draft"], wl.temperature, gen, top_k, top_p)
    st, g, orc = check(wl, 29, top_k, top_p, device_inputs=inputs)
    assert (g["num_accepted"] >= 0).all()


@pytest.mark.parametrize("case", ["zeros", "tiny", "huge"])
@pytest.mark.parametrize("top_k,top_p", [(0, 0.99), (2500, 1.0), (3000, 0.9)])
def test_filtered_values_outside_the_count_window(case, top_k, top_p):
    """bfloat16 rows whose crossing falls among values the value-count kernel
    keeps only in its outer words (|x| < 2^-64: exact zeros of both signs, or
    tiny magnitudes) or whose maximum is 2^64 or more; the row is then counted
    again with 32-bit counts over the whole range of magnitudes."""
    wl = WORKLOADS["spiky_bf16"].resized(B=4, K=3, V=4000)
    inputs = make_inputs(wl, 37, "cuda", top_k=top_k, top_p=top_p)
    g = torch.Generator(device="cuda")
    g.manual_seed(37)
    for key in ("target", "draft"):
        x = inputs[key].float()
        if case == "zeros":
            # 2000 logits near 0.5, the rest +0 and -0: the crossings of
            # top-p 0.99 and of k = 2500 / 3000 lie among the zeros.
            x = torch.where(torch.rand(x.shape, generator=g, device="cuda") < 0.5,
                            0.5 + 0.01 * x, torch.zeros_like(x))
            x = torch.where((x == 0) & (torch.rand(x.shape, generator=g, device="cuda") < 0.5),
                            -x, x)
        elif case == "tiny":
            # Half the logits are of magnitude 2^-80 .. 2^-70, both signs.
            tiny = torch.sign(x) * 2.0 ** (-80 + 10 * torch.rand(x.shape, generator=g,
                                                                  device="cuda"))
            x = torch.where(torch.rand(x.shape, generator=g, device="cuda") < 0.5, 0.3 * x, tiny)
        else:
            # The maximum of every row at 2^70 (the other logits ordinary).
            x[..., 17] = 2.0 ** 70
        inputs[key] = x.to(inputs[key].dtype)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(37)
    inputs["tokens"] = draw_from_logits(inputs["draft"], wl.temperature, gen, top_k, top_p)
    st, g_out, orc = check(wl, 37, top_k, top_p, device_inputs=inputs)
    assert (g_out["num_accepted"] >= 0).all()


def test_filtered_off_is_spec_verify():
    wl = WORKLOADS["spiky_bf16"].resized(B=32)
    inputs = make_inputs(wl, 2, "cuda")
    a = sv.spec_verify(inputs["target"], inputs["draft"], inputs["tokens"], wl.temperature, 99)
    for top_k, top_p in [(0, 1.0), (wl.V, 1.0), (wl.V + 10, 1.0)]:
        b = sv.spec_verify_filtered(inputs["target"], inputs["draft"], inputs["tokens"],
                                    wl.temperature, top_k, top_p, 99)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_filtered_greedy_ignores_the_cuts():
    wl = WORKLOADS["greedy_bf16"].resized(B=16)
    inputs = make_inputs(wl, 3, "cuda")
    a = sv.spec_verify(inputs["target"], None, inputs["tokens"], 1.0, 5, "greedy")
    b = sv.spec_verify_filtered(inputs["target"], None, inputs["tokens"], 1.0, 3, 0.5, 5,
                                "greedy")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_filtered_p_equals_q_accepts_everything():
    wl = WORKLOADS["llama3_bf16"].resized(B=16, K=5)
    inputs = make_inputs(wl, 8, "cuda", top_k=30, top_p=0.9)
    inputs["draft"] = inputs["target"][:, :wl.K].contiguous()
    # redraw the drafts from the (now identical) filtered target rows
    from speculative_decoding_verification_66_gb300.workloads import draw_from_logits
    gen = torch.Generator(device="cuda")
    gen.manual_seed(8)
    inputs["tokens"] = draw_from_logits(inputs["draft"], wl.temperature, gen, 30, 0.9)
    st, g, _ = check(wl, 8, 30, 0.9, device_inputs=inputs)
    # tokens are drawn by the input generator's own cut; only where it agrees
    # with the verifier's do all drafts pass
    assert (g["num_accepted"] == wl.K).mean() > 0.9


def test_filtered_invalid_rows():
    wl = WORKLOADS["small_f32"].resized(B=8, K=3, V=700)
    inputs = make_inputs(wl, 21, "cuda", top_k=10)
    t, d, x = inputs["target"], inputs["draft"], inputs["tokens"]
    t[2, 1, 17] = float("nan")
    d[3, 0, 5] = float("inf")
    t[4, :, :] = float("-inf")
    x[5, 2] = wl.V
    _, g, _ = check(wl, 21, 10, 0.9, device_inputs=inputs)
    assert list(g["num_accepted"][[2, 3, 4, 5]]) == [-1, -1, -1, -1]


def test_filtered_repeatable_and_empty():
    wl = WORKLOADS["llama3_bf16"].resized(B=8)
    inputs = make_inputs(wl, 4, "cuda", top_k=50, top_p=0.9)
    a = f_run(inputs, wl, 5, 50, 0.9)
    b = f_run(inputs, wl, 5, 50, 0.9)
    assert np.array_equal(a["out_tokens"], b["out_tokens"])
    assert np.array_equal(a["num_accepted"], b["num_accepted"])
    wl0 = wl.resized(B=0)
    i0 = make_inputs(wl0, 0, "cuda")
    out, nacc = sv.spec_verify_filtered(i0["target"], i0["draft"], i0["tokens"], 1.0, 5, 0.9, 1)
    torch.cuda.synchronize()
    assert out.shape == (0, wl.K + 1) and nacc.shape == (0,)


def test_filtered_timed_events():
    wl = WORKLOADS["spiky_bf16"].resized(B=16)
    inputs = make_inputs(wl, 6, "cuda", top_k=20, top_p=0.9)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    a = sv.spec_verify_filtered_timed(inputs["target"], inputs["draft"], inputs["tokens"], ev,
                                      wl.temperature, 20, 0.9, 3)
    torch.cuda.synchronize()
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0 for i in range(3))
    b = sv.spec_verify_filtered(inputs["target"], inputs["draft"], inputs["tokens"],
                                wl.temperature, 20, 0.9, 3)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("K", [0, 1, 16, 1024])
@pytest.mark.parametrize("top_k,top_p", [(20, 1.0), (0, 0.8), (50, 0.9)])
def test_filtered_draft_counts(K, top_k, top_p):
    """K = 0 (only the bonus row, drawn from the filtered p'_0), one draft, and
    long runs."""
    wl = WORKLOADS["spiky_bf16"].resized(B=6, K=K, V=3000)
    check(wl, 31, top_k, top_p)


def test_filtered_single_sequence_full_vocab():
    wl = WORKLOADS["llama3_bf16"].resized(B=1)
    st, _, _ = check(wl, 41, 50, 0.9)
    assert st["decisions"] > 0


@pytest.mark.parametrize("top_k,top_p", [(40, 0.9), (0, 0.9)])
def test_thresholds_kernel_timeout_path(top_k, top_p):
    """The thresholds kernels' timeout path, without a fault: their reads are
    held behind a device flag that nothing sets; every CTA marks its rows as
    timed out, and every sequence is reported as SV_SEQ_TIMEOUT. A gated call
    whose flag is already set matches spec_verify_filtered. Top-k 40 runs the
    group-maxima kernel, top-p alone (bf16) the value-count kernel."""
    wl = WORKLOADS["spiky_bf16"].resized(B=6, K=3, V=3000)
    inputs = make_inputs(wl, 2, "cuda", top_k=top_k, top_p=top_p)
    gate = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = sv.spec_verify_gated(inputs["target"], inputs["draft"], inputs["tokens"], gate,
                             wl.temperature, 9, "sample", stage=1, top_k=top_k, top_p=top_p)
    torch.cuda.synchronize()
    assert (r["seq_status"].cpu() == sv.SV_SEQ_TIMEOUT).all()
    assert (r["num_accepted"].cpu() == -1).all()
    gate.fill_(1)
    r = sv.spec_verify_gated(inputs["target"], inputs["draft"], inputs["tokens"], gate,
                             wl.temperature, 9, "sample", stage=1, top_k=top_k, top_p=top_p)
    out, nacc = sv.spec_verify_filtered(inputs["target"], inputs["draft"], inputs["tokens"],
                                        wl.temperature, top_k, top_p, 9, "sample")
    torch.cuda.synchronize()
    assert (r["seq_status"].cpu() == 0).all()
    assert torch.equal(r["out_tokens"], out) and torch.equal(r["num_accepted"], nacc)
