"""The LM head on the tensor cores, and verification from hidden states.

Two levels, each against the float64 oracle:

* ``sv_lmhead_logits`` (the GEMM alone) against the exact products h W^T of
  the same bfloat16 values: every element within the float32 accumulation
  bound D 2^-21 sum_d |h_d W_vd| (recursive summation in float32 is within
  (D - 1) 2^-24 of that sum; the factor 8 leaves room for the tensor core's
  own order of additions). A wrong operand layout, swizzle, descriptor or
  tile index gives errors of the size of the logits themselves.
* ``spec_verify_lmhead`` against ``oracle.verify_lmhead`` (the oracle's
  verification run on the exact float64 logits). The GPU's logits carry
  float32 accumulation error, about 1e-5 on a logit at D = 4096, which moves
  an acceptance ratio by a few 1e-5: the near-tie band is therefore 1e-3
  here (instead of 1e-5) and the normaliser tolerance 1e-4 relative.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_66_gb300 as sv
from speculative_decoding_verification_66_gb300.workloads import (LM_WORKLOADS, lm_host_arrays,
                                                                   make_lmhead_inputs)
from parity_util import compare, valid_output

pytestmark = pytest.mark.gpu

FLAG_LM = 1e-3
RTOL_LM = 1e-4
# Greedy decides on an argmax: the GPU takes it on float32-accumulated logits,
# the oracle on exact ones, so a row whose two largest exact logits lie within
# the accumulation error may go either way. 1e-3 is about 100x that error at
# D = 4096 for these weight scales.
GREEDY_GAP = 1e-3


def _greedy_compare(gpu, host, lw, rows):
    """Greedy LM-head results against the oracle, with near-ties flagged: up to
    the first position whose row has a top-2 gap below GREEDY_GAP the tokens
    must be identical; past it the output only has to be a valid result."""
    ht, wt, _, _, tok = host
    K, V = lw.K, lw.V
    rows = list(rows)
    b0, b1 = min(rows), max(rows) + 1
    orc = oracle.verify_lmhead(ht, wt, None, None, tok, 1.0, 0, oracle.GREEDY,
                               seq_range=(b0, b1))
    logits = oracle.lm_head_logits(ht[b0:b1], wt)  # [n, K+1, V], exact
    top2 = np.sort(logits, axis=-1)[..., -2:]
    gap = top2[..., 1] - top2[..., 0]
    flagged = 0
    for b in rows:
        assert int(gpu["seq_status"][b]) == int(orc["seq_status"][b]), b
        og, oo = gpu["out_tokens"][b], orc["out_tokens"][b]
        ng, no = int(gpu["num_accepted"][b]), int(orc["num_accepted"][b])
        if int(orc["seq_status"][b]) != 0:
            assert ng == -1 and np.all(og == -1), b
            continue
        near = [i for i in range(min(no, K) + 1) if gap[b - b0, i] < GREEDY_GAP]
        if not near:
            assert ng == no and np.array_equal(og, oo), (b, og, oo)
            continue
        flagged += 1
        f = near[0]
        assert ng >= min(f, no) and np.array_equal(og[:f], oo[:f]), (b, og, oo)
        assert valid_output(og, ng, tok[b], K, V), (b, og)
    return {"flagged_sequences": flagged, "sequences": len(rows)}


def _greedy_flag_cap(n):
    """Most greedy near-ties a check of n sequences may flag. A row's top-2
    gap falls below GREEDY_GAP with probability of a few 1e-3 for these
    logit scales (spacing of the top order statistics about sigma / sqrt(2 ln V)),
    so 2 + 2% of the sequences leaves room for the spread and still catches a
    systematic greedy error near ties."""
    return 2 + n // 50


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()
    torch.cuda.set_device(0)


def _bf16(shape, g, scale=1.0):
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


@pytest.mark.parametrize("R,D,V", [(128, 64, 256), (1, 8, 1), (300, 200, 1000), (129, 520, 513),
                                   (77, 136, 131), (256, 4096, 768), (640, 64, 2000)])
def test_lmhead_logits_match_exact_products(R, D, V):
    g = torch.Generator(device="cuda")
    g.manual_seed(R * 1000003 + D * 1009 + V)
    h = _bf16((R, D), g)
    w = _bf16((V, D), g, 1.0 / D ** 0.5)
    out = sv.sv_lmhead_logits(h, w)
    torch.cuda.synchronize()
    hb, wb = oracle.bf16_bits_to_f64(sv.workloads.bf16_bits(h)), \
        oracle.bf16_bits_to_f64(sv.workloads.bf16_bits(w))
    exact = oracle.lm_head_logits(sv.workloads.bf16_bits(h), sv.workloads.bf16_bits(w))
    bound = D * 2.0 ** -21 * (np.abs(hb) @ np.abs(wb).T) + 1e-30
    err = np.abs(out.cpu().numpy().astype(np.float64) - exact)
    worst = float((err / bound).max())
    assert worst <= 1.0, f"R={R} D={D} V={V}: error {err.max():.3g}, {worst:.3g} x the bound"


def test_lmhead_logits_one_hot_rows_pick_columns():
    """h = e_d selects column d of W exactly (no rounding at all)."""
    R, D, V = 200, 192, 700
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    w = _bf16((V, D), g)
    h = torch.zeros((R, D), dtype=torch.bfloat16, device="cuda")
    cols = torch.arange(R, device="cuda") % D
    h[torch.arange(R, device="cuda"), cols] = 1.0
    out = sv.sv_lmhead_logits(h, w)
    assert torch.equal(out, w.float()[:, cols].T.contiguous())


def _lm_call(inp, lw, seed, **kw):
    return sv.spec_verify_lmhead(inp["hidden_t"], inp["weight_t"], inp["hidden_d"],
                                 inp["weight_d"], inp["tokens"], lw.temperature, seed, lw.mode,
                                 **kw)


def _check(lw, seed, seq_ranges=None, inp=None):
    if inp is None:
        inp = make_lmhead_inputs(lw, seed, "cuda")
    s = 0x1A4EAD00 + seed
    greedy = lw.mode == "greedy"
    gpu = _lm_call(inp, lw, s, diagnostics=True)
    torch.cuda.synchronize()
    gpu = {k: v.cpu().numpy() for k, v in gpu.items()}
    host = lm_host_arrays(inp)
    st = None
    g_flagged = g_seqs = 0
    for rng in (seq_ranges or [None]):
        rows = range(lw.B) if rng is None else range(*rng)
        if greedy:
            if lw.B > 0:
                st = _greedy_compare(gpu, host, lw, rows)
                g_flagged += st["flagged_sequences"]
                g_seqs += st["sequences"]
            continue
        orc = oracle.verify_lmhead(*host[:4], host[4], lw.temperature, s, oracle.SAMPLE,
                                   seq_range=rng, threads=8)
        st = compare(gpu, orc, host[4], lw.K, lw.V, rows=rows, greedy=False, flag=FLAG_LM,
                     rtol=RTOL_LM)
    if greedy and g_seqs > 0:
        print(f"greedy near-ties: {g_flagged} of {g_seqs} sequences flagged")
        assert g_flagged <= _greedy_flag_cap(g_seqs), (g_flagged, g_seqs)
    # The plain call gives the same tokens as the diagnostic one.
    out, nacc = _lm_call(inp, lw, s)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), gpu["out_tokens"])
    assert np.array_equal(nacc.cpu().numpy(), gpu["num_accepted"])
    return st


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lmhead_verify_small(seed):
    st = _check(LM_WORKLOADS["lm_small"], seed)
    assert st["flagged_sequences"] <= 3


@pytest.mark.parametrize("kw", [dict(K=0), dict(K=1), dict(B=1, K=7), dict(V=7, d_target=8,
                                                                         d_draft=8),
                                dict(V=257, d_target=64, d_draft=1024),
                                dict(mode="greedy"), dict(mode="greedy", K=0),
                                dict(temperature=0.3), dict(B=130, K=2, V=3000),
                                dict(B=2, K=1024, V=1000)])
def test_lmhead_verify_edges(kw):
    _check(LM_WORKLOADS["lm_small"].resized(**kw), 5)


def test_lmhead_verify_empty_batch():
    lw = LM_WORKLOADS["lm_small"].resized(B=0)
    inp = make_lmhead_inputs(lw, 0, "cuda")
    out, nacc = _lm_call(inp, lw, 1)
    assert out.shape == (0, lw.K + 1) and nacc.shape == (0,)


def test_lmhead_nonfinite_hidden_state_flags_sequence():
    lw = LM_WORKLOADS["lm_small"]
    inp = make_lmhead_inputs(lw, 3, "cuda")
    inp["hidden_t"][5, 2, 17] = float("nan")
    inp["hidden_d"][9, 1, 3] = float("inf")
    gpu = _lm_call(inp, lw, 9, diagnostics=True)
    torch.cuda.synchronize()
    st = gpu["seq_status"].cpu().numpy()
    assert st[5] == sv.SV_SEQ_NONFINITE and st[9] == sv.SV_SEQ_NONFINITE
    assert (np.delete(st, [5, 9]) == 0).all()
    assert (gpu["out_tokens"][5].cpu() == -1).all() and int(gpu["num_accepted"][9]) == -1


@pytest.mark.parametrize("name", ["lm_llama3_bf16", "lm_greedy_bf16"])
def test_lmhead_verify_full_size_sampled(name):
    """The full-size configuration the benchmark times; the oracle checks
    every output of 6 sequences spread over the batch (their logits in
    float64: 17 rows x 128256 x 4096 products each)."""
    lw = LM_WORKLOADS[name]
    _check(lw, 11, seq_ranges=[(0, 2), (127, 129), (254, 256)])


@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_lmhead_timeout_path(mode):
    """The bounded waits' timeout path, without a fault: the statistics GEMM's
    producer waits on a device flag that nothing sets. The wait runs out
    (about 2 s), the kernel drains and releases its tensor memory, and every
    sequence comes back as SV_SEQ_TIMEOUT. The context stays usable: an
    ordinary call afterwards still matches the oracle, and a gated call whose
    flag is already set matches the ordinary call."""
    lw = LM_WORKLOADS["lm_small"].resized(B=8, mode=mode)
    inp = make_lmhead_inputs(lw, 2, "cuda")
    gate = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = sv.spec_verify_lmhead_gated(inp["hidden_t"], inp["weight_t"], inp["hidden_d"],
                                    inp["weight_d"], inp["tokens"], gate, lw.temperature, 3, mode)
    torch.cuda.synchronize()
    assert (r["seq_status"].cpu() == sv.SV_SEQ_TIMEOUT).all()
    assert (r["num_accepted"].cpu() == -1).all() and (r["out_tokens"].cpu() == -1).all()
    _check(lw, 2, inp=inp)
    gate.fill_(1)
    r = sv.spec_verify_lmhead_gated(inp["hidden_t"], inp["weight_t"], inp["hidden_d"],
                                    inp["weight_d"], inp["tokens"], gate, lw.temperature, 3, mode)
    out, nacc = _lm_call(inp, lw, 3)
    torch.cuda.synchronize()
    assert (r["seq_status"].cpu() == 0).all()
    assert torch.equal(r["out_tokens"], out) and torch.equal(r["num_accepted"], nacc)


@pytest.mark.parametrize("v1,v2", [(100, 300), (10, 20), (255, 256), (0, 999)])
def test_lmhead_greedy_ties_take_the_lowest_index(v1, v2):
    """Greedy ties across and within 256-column tiles: one-hot hidden states
    make every logit an exact copy of one weight, and two vocabulary entries
    share the largest weight of every column, so each row's maximum is tied
    between v1 and v2 exactly. The lowest index must win, as the oracle's."""
    B, K, V, D = 6, 3, 1000, 64
    g = torch.Generator(device="cuda")
    g.manual_seed(v1 * 7 + v2)
    w = (torch.rand((V, D), generator=g, device="cuda") * 2 - 1).to(torch.bfloat16)
    w[v1] = 4.0
    w[v2] = 4.0
    cols = torch.randint(0, D, (B, K + 1), generator=g, device="cuda")
    h = torch.zeros((B, K + 1, D), dtype=torch.bfloat16, device="cuda")
    h.scatter_(2, cols.unsqueeze(-1), 1.0)
    # Drafts: the tie winner for the first b mod K positions of sequence b,
    # then the loser, so sequences stop at different positions (b mod K).
    tok = torch.full((B, K), v1, dtype=torch.int32, device="cuda")
    for b in range(B):
        tok[b, b % K:] = v2
    r = sv.spec_verify_lmhead(h, w, None, None, tok, 1.0, 5, "greedy", diagnostics=True)
    torch.cuda.synchronize()
    host = (sv.workloads.bf16_bits(h), sv.workloads.bf16_bits(w), None, None,
            tok.cpu().numpy())
    orc = oracle.verify_lmhead(*host[:4], host[4], 1.0, 5, oracle.GREEDY)
    assert np.array_equal(r["num_accepted"].cpu().numpy(), orc["num_accepted"])
    assert np.array_equal(r["out_tokens"].cpu().numpy(), orc["out_tokens"])
    assert (r["out_tokens"].cpu().numpy() != v2).all()


def test_lmhead_emitted_tokens_follow_target_law():
    """The pages' invariant (the output follows the target distribution) through
    the whole LM-head path: statistics GEMM, scan, emitted-pair GEMM and
    sampler. 2^19 sequences share one set of hidden states; drafts x_i ~ q_i
    from numpy's generator. Among sequences that reach position i, the token
    at i must follow p_i = softmax(h_t,i W_t^T) (exact float64 logits from the
    oracle), by chi-square with a Bonferroni-corrected threshold; the first
    acceptance rate must match sum_x min(p_0(x), q_0(x)) to five standard
    deviations."""
    from scipy import stats
    K, B, V, Dt, Dd = 2, 1 << 19, 8, 64, 32
    rng = np.random.default_rng(77)

    def bf16_bits(a):
        u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    ht = bf16_bits(rng.normal(size=(K + 1, Dt)))
    wt = bf16_bits(rng.normal(size=(V, Dt)) * 1.2 / Dt ** 0.5)
    hd = bf16_bits(rng.normal(size=(K, Dd)))
    wd = bf16_bits(rng.normal(size=(V, Dd)) * 1.2 / Dd ** 0.5)
    lt = oracle.lm_head_logits(ht, wt)
    ld = oracle.lm_head_logits(hd, wd)
    p = np.exp(lt - lt.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    q = np.exp(ld - ld.max(1, keepdims=True))
    q /= q.sum(1, keepdims=True)
    x = np.stack([rng.choice(V, size=B, p=q[i]) for i in range(K)], 1).astype(np.int32)

    def dev(bits, shape):
        t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()
        return t.unsqueeze(0).expand(*shape).contiguous() if len(shape) == 3 else t

    h_t = dev(ht, (B, K + 1, Dt))
    h_d = dev(hd, (B, K, Dd))
    out, nacc = sv.spec_verify_lmhead(h_t, dev(wt, ()), h_d, dev(wd, ()),
                                      torch.from_numpy(x).cuda(), 1.0, 0x5EED, "sample")
    torch.cuda.synchronize()
    out, nacc = out.cpu().numpy(), nacc.cpu().numpy()
    assert np.all((nacc >= 0) & (nacc <= K))
    pvals = []
    for i in range(K + 1):
        toks = out[nacc >= i, i]
        assert np.all((toks >= 0) & (toks < V))
        counts = np.bincount(toks, minlength=V)
        pvals.append(stats.chisquare(counts, p[i] * counts.sum()).pvalue)
    assert min(pvals) > 1e-3 / (K + 1), pvals
    beta0 = np.minimum(p[0], q[0]).sum()
    rate = np.mean(nacc >= 1)
    assert abs(rate - beta0) < 5 * np.sqrt(beta0 * (1 - beta0) / B)
