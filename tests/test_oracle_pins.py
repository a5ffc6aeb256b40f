"""Pins of the float64 oracle to facts fixed outside the oracle itself.

Every check here compares the oracle with something it does not compute:
numbers printed on the pages (tests/golden/worked_examples.json), closed forms
of rejection sampling, exact path sums on tiny vocabularies, library routines
(torch float64 logsumexp / argmax), and an independently written Philox.
All run on the CPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def softmax64(logits, T=1.0):
    """Reference softmax in float64 numpy (not the oracle's code)."""
    s = np.asarray(logits, dtype=np.float64) / T
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def draw_tokens(rng, q):
    """x ~ q independently per row of q [B, K, V] (inverse CDF with numpy's RNG)."""
    c = np.cumsum(q, axis=-1)
    u = rng.random(q.shape[:-1] + (1,))
    return np.minimum((u > c).sum(axis=-1), q.shape[-1] - 1).astype(np.int32)


# --------------------------------------------------------------------------
# The pages' worked examples.
# --------------------------------------------------------------------------
GOLDEN = json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))["examples"]


@pytest.mark.parametrize("ex", GOLDEN, ids=[e["name"] for e in GOLDEN])
def test_worked_example_values(oracle_mod, ex):
    o = oracle_mod
    p, q = np.array(ex["p"]), np.array(ex["q"])
    t_row = np.log(p).astype(np.float32)
    d_row = np.log(q).astype(np.float32)
    st_t, lse_t = o.row_lse(t_row, 1.0)
    st_d, lse_d = o.row_lse(d_row, 1.0)
    assert st_t == 0 and st_d == 0
    p_or = np.array([math.exp(o.log_prob(t_row, k, 1.0, lse_t)) for k in range(2)])
    q_or = np.array([math.exp(o.log_prob(d_row, k, 1.0, lse_d)) for k in range(2)])
    np.testing.assert_allclose(p_or, p, atol=1e-7)
    np.testing.assert_allclose(q_or, q, atol=1e-7)
    r = np.array([o.accept_prob(o.log_prob(t_row, k, 1.0, lse_t), o.log_prob(d_row, k, 1.0, lse_d))
                  for k in range(2)])
    np.testing.assert_allclose(r, ex["accept"], atol=1e-6)
    assert r[1] == 1.0  # B is accepted whenever it is proposed
    w = o.sample_weights(t_row, d_row, 1.0, lse_t, lse_d)
    assert w[0] == 0.0
    np.testing.assert_allclose(w / w.sum(), ex["residual"], atol=1e-12)
    # Path sum: P(final = v) = q_v r_v + (rejected mass) * residual_v.
    rejected = float(np.sum(q_or * (1.0 - r)))
    final = q_or * r + rejected * (w / w.sum())
    np.testing.assert_allclose(final, ex["final"], atol=1e-6)
    if "final_B_parts" in ex:
        np.testing.assert_allclose([q_or[1] * r[1], rejected * (w / w.sum())[1]],
                                   ex["final_B_parts"], atol=1e-6)


@pytest.mark.parametrize("ex", GOLDEN, ids=[e["name"] for e in GOLDEN])
def test_worked_example_sampled(oracle_mod, ex):
    """The full verify step, run 400k times with x ~ q, emits A at rate p_A."""
    o = oracle_mod
    n = 400_000
    p, q = np.array(ex["p"]), np.array(ex["q"])
    target = np.broadcast_to(np.log(p).astype(np.float32), (n, 2, 2)).copy()
    draft = np.broadcast_to(np.log(q).astype(np.float32), (n, 1, 2)).copy()
    tokens = draw_tokens(np.random.default_rng(11), softmax64(draft))
    res = o.verify(target, draft, tokens, 1.0, seed=0xABCDEF, threads=4)
    first = res["out_tokens"][:, 0]
    freq_A = np.mean(first == 0)
    sd = math.sqrt(p[0] * (1 - p[0]) / n)
    assert abs(freq_A - p[0]) < 5 * sd
    # Acceptance rate = sum_x min(p, q) (closed form of min(1, p/q) under x ~ q).
    beta = float(np.minimum(p, q).sum())
    acc = np.mean(res["num_accepted"] == 1)
    assert abs(acc - beta) < 5 * math.sqrt(beta * (1 - beta) / n)
    # A rejection always emits B: the residual sits entirely on B.
    rej = res["num_accepted"] == 0
    assert np.all(first[rej] == 1)


# --------------------------------------------------------------------------
# Softmax normaliser and argmax against library routines.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 2, 7, 1000, 32000])
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_lse_against_torch(oracle_mod, V, T, dtype):
    g = torch.Generator().manual_seed(V * 31 + int(T * 10))
    row = torch.randn(V, generator=g) * 3.0
    if dtype == "bf16":
        row = row.to(torch.bfloat16)
        arr = row.view(torch.int16).numpy().view(np.uint16)
    else:
        arr = row.numpy().astype(np.float32)
    T32 = float(np.float32(T))
    ref = torch.logsumexp(row.to(torch.float64) / T32, dim=0).item()
    st, lse = oracle_mod.row_lse(arr, T32)
    assert st == 0
    assert abs(lse - ref) <= 1e-12 * max(1.0, abs(ref))
    k = V // 2
    lp_ref = torch.log_softmax(row.to(torch.float64) / T32, dim=0)[k].item()
    assert abs(oracle_mod.log_prob(arr, k, T32, lse) - lp_ref) <= 1e-12 * max(1.0, abs(lp_ref))


def test_lse_closed_form_constant_row(oracle_mod):
    for V in (1, 3, 128256):
        for c in (-5.0, 0.0, 2.25):
            row = np.full(V, c, dtype=np.float32)
            st, lse = oracle_mod.row_lse(row, 0.5)
            assert st == 0
            assert abs(lse - (c / 0.5 + math.log(V))) < 1e-12 * max(1, abs(c / 0.5 + math.log(V)))


def test_bf16_widening_against_torch(oracle_mod):
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.elem(bits, k) for k in range(0, 65536, 97)])
    exp = ref[::97]
    same = (got == exp) | (np.isnan(got) & np.isnan(exp))
    assert same.all()


def test_argmax_against_torch_first_occurrence(oracle_mod):
    g = torch.Generator().manual_seed(5)
    for V in (1, 2, 9, 4096, 50257):
        for _ in range(5):
            # small integers => many exact ties; torch.argmax returns the first maximal index
            row = torch.randint(-4, 5, (V,), generator=g).to(torch.bfloat16)
            k, nan = oracle_mod.row_argmax(row.view(torch.int16).numpy().view(np.uint16))
            assert not nan
            assert k == int(torch.argmax(row.float()).item())
            rowf = torch.randint(-3, 3, (V,), generator=g).float()
            k, nan = oracle_mod.row_argmax(rowf.numpy())
            assert k == int(torch.argmax(rowf).item())


def test_argmax_nan_and_neg_inf(oracle_mod):
    row = np.array([1.0, np.nan, 3.0], dtype=np.float32)
    _, nan = oracle_mod.row_argmax(row)
    assert nan
    row = np.full(5, -np.inf, dtype=np.float32)
    k, nan = oracle_mod.row_argmax(row)
    assert k == 0 and not nan


# --------------------------------------------------------------------------
# Philox4x32-10 against an independent implementation.
# --------------------------------------------------------------------------
_TRITON_SCRIPT = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def _k(out_ptr, c0_ptr, c1_ptr, c2_ptr, c3_ptr, seed, N: tl.constexpr):
    o = tl.arange(0, N)
    c0 = tl.load(c0_ptr + o); c1 = tl.load(c1_ptr + o)
    c2 = tl.load(c2_ptr + o); c3 = tl.load(c3_ptr + o)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3, 10)
    tl.store(out_ptr + o * 4 + 0, a.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + o * 4 + 1, b.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + o * 4 + 2, c.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + o * 4 + 3, d.to(tl.int64) & 0xFFFFFFFF)

cases = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cases:
    ctrs = np.array(ctrs, dtype=np.int64)
    N = ctrs.shape[0]
    cols = [torch.from_numpy(ctrs[:, i].astype(np.uint32).view(np.int32).copy()) for i in range(4)]
    out = torch.zeros(N * 4, dtype=torch.int64)
    _k[(1,)](out, *cols, seed, N)
    res.append(out.view(N, 4).tolist())
print(json.dumps(res))
"""


def test_philox_against_triton_interpreter(oracle_mod):
    """triton ships its own Philox4x32-10 (key = (lo, hi) of the seed); its CPU
    interpreter runs it without a GPU."""
    pytest.importorskip("triton")
    import subprocess
    import sys
    rng = np.random.default_rng(2024)
    cases = []
    for seed in (0, 1, 0x5EED0003, 0xDEADBEEFCAFEF00D, 2**63 + 12345):
        ctrs = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64)
        ctrs[:8, 2:] = 0  # the counters the verifier uses: (pos, seq, 0, 0)
        ctrs[0] = 0
        cases.append([int(seed), ctrs.astype(np.int64).tolist()])
    p = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(cases),
                       capture_output=True, text=True, timeout=600)
    if p.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + p.stderr.strip().splitlines()[-1])
    ref = json.loads(p.stdout.strip().splitlines()[-1])
    for (seed, ctrs), want in zip(cases, ref):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for c, w in zip(ctrs, want):
            got = oracle_mod.philox(c, key)
            assert [int(x) for x in got] == [int(x) for x in w], (seed, c)


def test_uniform_is_24bit_and_uniform(oracle_mod):
    from scipy import stats
    n = 200_000
    u = np.array([oracle_mod.uniform(77, b, i, 0) for b in range(n // 4) for i in range(4)])
    assert u.min() >= 0.0 and u.max() <= 1.0 - 2.0 ** -24
    assert np.all(u * 2**24 == np.floor(u * 2**24))  # exact multiples of 2^-24
    counts = np.histogram(u, bins=256, range=(0.0, 1.0))[0]
    assert stats.chisquare(counts).pvalue > 1e-4


def test_race_uniform_open_interval_and_uniform(oracle_mod):
    from scipy import stats
    v = np.array([oracle_mod.race_uniform(5, b, j, k)
                  for b in range(50) for j in range(4) for k in range(1000)])
    assert v.min() > 0.0 and v.max() < 1.0
    m = v * 2**24
    assert np.all(m == np.floor(m)) and np.all(m % 2 == 1)  # odd multiples of 2^-24
    counts = np.histogram(v, bins=200, range=(0.0, 1.0))[0]
    assert stats.chisquare(counts).pvalue > 1e-4
    # the race stream does not reuse the acceptance uniforms of the same position
    a = np.array([oracle_mod.uniform(5, b, 0, 0) for b in range(3000)])
    r = np.array([oracle_mod.race_uniform(5, b, 0, 0) for b in range(3000)])
    assert abs(np.corrcoef(a, r)[0, 1]) < 0.1


@pytest.mark.parametrize("V", [2, 7, 300])
def test_race_draws_proportional_to_weight(oracle_mod, V):
    """The exponential race picks token k with probability w_k / sum(w);
    zero-weight tokens are never picked."""
    from scipy import stats
    rng = np.random.default_rng(V)
    w = rng.gamma(0.7, size=V)
    if V > 2:
        w[rng.integers(V)] = 0.0
    n = 60_000 if V > 10 else 40_000
    toks = np.array([oracle_mod.race_sample(w, 31, b, 2)[0] for b in range(n)])
    counts = np.bincount(toks, minlength=V)
    assert counts[w == 0].sum() == 0
    keep = w > 0
    exp = w[keep] / w.sum() * n
    if V > 10:  # pool sparse cells
        order = np.argsort(exp)
        grp = np.cumsum(exp[order]) // 50
        c2 = np.bincount(grp.astype(int), weights=counts[keep][order])
        e2 = np.bincount(grp.astype(int), weights=exp[order])
        nz = e2 > 0
        assert stats.chisquare(c2[nz], e2[nz]).pvalue > 1e-3
    else:
        assert stats.chisquare(counts[keep], exp).pvalue > 1e-3


def test_two_level_race_law(oracle_mod):
    """Four blocks of the two-level race (V > 3 blocks): the winning block
    follows W_c / Z and the token within it w_k / W_c, so every token follows
    w_k / Z. Weights sit on a few tokens per block (including the first token
    of block 0 and the last token of the row) so that each race is cheap."""
    from scipy import stats
    L = oracle_mod.RACE_BLOCK
    V = 3 * L + 100
    w = np.zeros(V)
    rng = np.random.default_rng(12)
    block_mass = [0.1, 0.4, 0.2, 0.3]
    picks = []
    for c, mass in enumerate(block_mass):
        lo, hi = c * L, min((c + 1) * L, V)
        idx = rng.choice(np.arange(lo + 1, hi - 1), size=3, replace=False).tolist()
        idx += [lo] if c == 0 else []
        idx += [V - 1] if c == 3 else []
        share = rng.dirichlet(np.ones(len(idx)))
        w[idx] = mass * share
        picks += idx
    n = 20_000
    toks = np.array([oracle_mod.race_sample(w, 99, b, 3)[0] for b in range(n)])
    blocks = np.bincount(toks // L, minlength=4)
    assert stats.chisquare(blocks, np.array(block_mass) * n).pvalue > 1e-3
    picks = np.array(sorted(picks))
    counts = np.array([(toks == k).sum() for k in picks])
    assert counts.sum() == n
    assert stats.chisquare(counts, w[picks] / w.sum() * n).pvalue > 1e-3


def _plain_race(o, w, seed, seq, pos):
    """A one-level exponential race written out here, independently of the
    oracle's race: token = argmax over w_k > 0 of w_k / E_k, E_k = -ln v_k, v_k
    from lane k mod 4 of Philox4x32-10 at counter (pos, seq, 1 + k div 4, 0)
    mapped to (2 (word >> 9) + 1) 2^-24; the lowest index wins an exact tie.
    Only the Philox words come from the oracle (``philox_many``, itself pinned
    against triton's generator). Returns (token, relative top-2 gap)."""
    V = len(w)
    n = (V + 3) // 4
    ctr = np.zeros((n, 4), dtype=np.uint32)
    ctr[:, 0] = pos
    ctr[:, 1] = seq
    ctr[:, 2] = 1 + np.arange(n)
    words = o.philox_many(ctr, [seed & 0xFFFFFFFF, seed >> 32]).reshape(-1)[:V]
    best, second, tok = -math.inf, 0.0, -1
    for k in range(V):
        if w[k] > 0.0:
            v = (2.0 * float(int(words[k]) >> 9) + 1.0) * 2.0 ** -24
            score = w[k] / -math.log(v)
            if score > best:
                if tok >= 0:
                    second = best
                best, tok = score, k
            elif score > second:
                second = score
    return tok, ((best - second) / best if tok >= 0 else 0.0)


@pytest.mark.parametrize("V", [1, 5, 300, 2000])
def test_race_one_block_is_the_plain_race(oracle_mod, V):
    """With one block (block length >= V) the two-level race is the plain
    one-level race argmax_k w_k / E_k: same token, same margin, seed by seed."""
    rng = np.random.default_rng(V + 5)
    w = rng.gamma(0.6, size=V)
    if V > 2:
        w[rng.choice(V, size=V // 4, replace=False)] = 0.0
    for block in (V, V + 3, 4096):
        for seq in range(150):
            want, gap = _plain_race(oracle_mod, w, 4242 + seq, seq, 3)
            got, margin = oracle_mod.race_sample(w, 4242 + seq, seq, 3, block=block)
            assert got == want, (block, seq)
            # level 1 has a single candidate (margin 1), so the margin is level 2's gap
            assert margin == pytest.approx(gap, rel=1e-12, abs=1e-300), (block, seq)


@pytest.mark.parametrize("block", [1, 7, 512, 1100])
def test_two_level_race_law_any_block(oracle_mod, block):
    """The draw follows w / Z whatever the block length: 1 (level 1 alone),
    7 (many blocks, a ragged last block of one token), 512 (the library's
    length, a ragged last block) and V (one block). Chi-square of the tokens,
    pooled into cells of >= 50 expected draws, and of the blocks."""
    from scipy import stats
    V = 1100
    rng = np.random.default_rng(block)
    w = rng.gamma(0.5, size=V)
    w[rng.choice(V, size=200, replace=False)] = 0.0
    w[V - 1] = 3.0 * w.max()  # the last token alone in a ragged block for block 7
    n = 30_000
    toks = np.array([oracle_mod.race_sample(w, 555, b, 1, block=block)[0] for b in range(n)])
    assert toks.min() >= 0 and np.all(w[toks] > 0)
    counts = np.bincount(toks, minlength=V)
    exp = w / w.sum() * n
    keep = w > 0
    order = np.argsort(exp[keep])
    grp = (np.cumsum(exp[keep][order]) // 50).astype(int)
    c2 = np.bincount(grp, weights=counts[keep][order])
    e2 = np.bincount(grp, weights=exp[keep][order])
    nz = e2 > 0
    assert stats.chisquare(c2[nz], e2[nz] * c2[nz].sum() / e2[nz].sum()).pvalue > 1e-3
    nb = (V + block - 1) // block
    if 1 < nb <= 200:
        W = np.add.reduceat(w, np.arange(0, V, block))
        cb = np.bincount(toks // block, minlength=nb)
        eb = W / W.sum() * n
        ok = eb > 0
        assert cb[~ok].sum() == 0
        assert stats.chisquare(cb[ok], eb[ok] * cb[ok].sum() / eb[ok].sum()).pvalue > 1e-3


def test_verify_one_block_draws_the_plain_race(oracle_mod):
    """The verifier with race_block >= V emits, at position j, the token of the
    plain one-level race over its own weights (max(0, p - q) after a rejection,
    p of the bonus row otherwise), clocks keyed by (j, b)."""
    o = oracle_mod
    rng = np.random.default_rng(8)
    B, K, V, T, seed = 60, 3, 600, 0.8, 0xABCDEF12345
    t = (rng.normal(size=(B, K + 1, V)) * 1.5).astype(np.float32)
    d = (t[:, :K] + rng.normal(size=(B, K, V)).astype(np.float32)).astype(np.float32)
    tok = draw_tokens(rng, softmax64(d, T))
    res = o.verify(t, d, tok, T, seed, race_block=V)
    res512 = o.verify(t, d, tok, T, seed)
    np.testing.assert_array_equal(res["num_accepted"], res512["num_accepted"])
    Tf = float(np.float32(T))
    for b in range(B):
        j = int(res["num_accepted"][b])
        lse_t = res["lse_t"][b, j]
        if j < K:
            w = o.sample_weights(t[b, j], d[b, j], Tf, lse_t, res["lse_d"][b, j])
        else:
            w = o.sample_weights(t[b, K], None, Tf, lse_t, 0.0)
        want, gap = _plain_race(o, w, seed, b, j)
        assert res["out_tokens"][b, j] == want, b
        assert res["sample_margin"][b] == pytest.approx(gap, rel=1e-12, abs=1e-300)


def test_block_uniforms_are_their_own_stream(oracle_mod):
    b = np.array([oracle_mod.block_uniform(3, s, 1, c) for s in range(500) for c in range(8)])
    t = np.array([oracle_mod.race_uniform(3, s, 1, c) for s in range(500) for c in range(8)])
    assert b.min() > 0 and b.max() < 1
    assert np.all((b * 2**24) % 2 == 1)
    assert abs(np.corrcoef(b, t)[0, 1]) < 0.1


@pytest.mark.parametrize("V, levels", [(500, 1), (2000, 2)])
def test_race_near_tie_law(oracle_mod, V, levels):
    """Closed form: the relative gap between a race's two best scores is below
    tau with probability at most tau (memorylessness of the exponential clocks),
    whatever the number of tokens. A row of one block has one such gap (level 1
    has a single candidate, margin 1); a row of several blocks has two, so at
    most 2 tau. This is what keeps near-ties rare at V = 128k."""
    assert (V <= oracle_mod.RACE_BLOCK) == (levels == 1)
    rng = np.random.default_rng(1)
    w = rng.lognormal(sigma=2.0, size=V)
    n = 20_000
    margins = np.array([oracle_mod.race_sample(w, 77, b, 0)[1] for b in range(n)])
    tau = 0.02
    frac = np.mean(margins < tau)
    bound = levels * tau
    sd = math.sqrt(bound * (1 - bound) / n)
    assert frac < bound + 5 * sd
    assert frac > 0.3 * tau  # and it is not degenerate
    assert np.all((margins >= 0) & (margins <= 1))


# --------------------------------------------------------------------------
# Exact path sums on tiny vocabularies: the output law is the target law.
# --------------------------------------------------------------------------
def _random_rows(rng, K, V, scale=1.5):
    t = (rng.normal(size=(K + 1, V)) * scale).astype(np.float32)
    d = (rng.normal(size=(K, V)) * scale).astype(np.float32)
    return t, d


@pytest.mark.parametrize("V,K", [(2, 1), (2, 3), (3, 2), (4, 3)])
def test_exact_path_sum(oracle_mod, V, K):
    """Enumerate every draft sequence and every accept/reject branch with the
    oracle's acceptance probabilities and sampling weights; the probability of
    each output, grouped by prefix, must factor as P(prefix) * p_i(y_i)."""
    o = oracle_mod
    rng = np.random.default_rng(100 * V + K)
    t, d = _random_rows(rng, K, V)
    T = 0.8
    p = softmax64(t, T)
    q = softmax64(d, T)
    lse_t = [o.row_lse(t[i], T)[1] for i in range(K + 1)]
    lse_d = [o.row_lse(d[i], T)[1] for i in range(K)]
    r = np.array([[o.accept_prob(o.log_prob(t[i], x, T, lse_t[i]), o.log_prob(d[i], x, T, lse_d[i]))
                   for x in range(V)] for i in range(K)])
    res = []
    for i in range(K):
        w = o.sample_weights(t[i], d[i], T, lse_t[i], lse_d[i])
        res.append(w / w.sum())
    wb = o.sample_weights(t[K], None, T, lse_t[K], 0.0)
    bonus = wb / wb.sum()

    out = {}  # output tuple -> probability

    def walk(i, prefix, prob):
        if i == K:
            for v in range(V):
                out[prefix + (v,)] = out.get(prefix + (v,), 0.0) + prob * bonus[v]
            return
        for x in range(V):
            px = prob * q[i, x]
            walk(i + 1, prefix + (x,), px * r[i, x])
            for v in range(V):
                key = prefix + (v,)
                out[key] = out.get(key, 0.0) + px * (1.0 - r[i, x]) * res[i][v]

    walk(0, (), 1.0)
    assert abs(sum(out.values()) - 1.0) < 1e-12
    # P(position i emitted with prefix y_<i and value v) = P(reach i with prefix) * p_i(v)
    reach = {(): 1.0}
    for i in range(K + 1):
        emitted = {}
        for seq, pr in out.items():
            if len(seq) > i:
                emitted[seq[:i + 1]] = emitted.get(seq[:i + 1], 0.0) + pr
        for pre, pr_pre in reach.items():
            for v in range(V):
                got = emitted.get(pre + (v,), 0.0)
                assert abs(got - pr_pre * p[i, v]) < 1e-12, (i, pre, v)
        # reaching i+1 with prefix y_<=i means y_i was an accepted draft
        nxt = {}
        if i < K:
            for pre, pr_pre in reach.items():
                for v in range(V):
                    nxt[pre + (v,)] = pr_pre * q[i, v] * r[i, v]
        reach = nxt
    # acceptance at each position is sum_x min(p, q)
    for i in range(K):
        assert abs(np.sum(q[i] * r[i]) - np.minimum(p[i], q[i]).sum()) < 1e-12


# --------------------------------------------------------------------------
# Monte Carlo over the full verify step.
# --------------------------------------------------------------------------
def _mc(oracle_mod, V, K, n, T, seed, same=False):
    rng = np.random.default_rng(seed)
    t, d = _random_rows(rng, K, V)
    if same:
        d = t[:K].copy()
    target = np.broadcast_to(t, (n, K + 1, V)).copy()
    draft = np.broadcast_to(d, (n, K, V)).copy()
    tokens = draw_tokens(rng, np.broadcast_to(softmax64(d, T), (n, K, V)))
    res = oracle_mod.verify(target, draft, tokens, T, seed=seed * 7 + 3, threads=8)
    return t, d, tokens, res


@pytest.mark.parametrize("V,K,n", [(2, 1, 200_000), (5, 3, 1_000_000), (8, 4, 300_000)])
def test_output_marginal_chisquare(oracle_mod, V, K, n):
    """Among trials that reach position i, the emitted token follows p_i."""
    from scipy import stats
    T = 0.9
    t, d, tokens, res = _mc(oracle_mod, V, K, n, float(np.float32(T)), seed=V * 10 + K)
    p = softmax64(t, float(np.float32(T)))
    na = res["num_accepted"]
    assert (res["seq_status"] == 0).all()
    n_tests = K + 1
    for i in range(K + 1):
        sel = na >= i
        y = res["out_tokens"][sel, i]
        counts = np.bincount(y, minlength=V)
        exp = p[i] * sel.sum()
        keep = exp > 0
        pv = stats.chisquare(counts[keep], exp[keep] * counts.sum() / exp[keep].sum()).pvalue
        assert pv > 1e-3 / n_tests, (i, counts, exp)


@pytest.mark.parametrize("V,K", [(6, 4)])
def test_acceptance_closed_form(oracle_mod, V, K):
    """P(accept at i | reached i) = sum_x min(p_i, q_i); P(num_accepted >= j) = prod beta."""
    n = 500_000
    T = 1.0
    t, d, tokens, res = _mc(oracle_mod, V, K, n, T, seed=4242)
    p, q = softmax64(t, T), softmax64(d, T)
    beta = np.minimum(p[:K], q).sum(axis=1)
    na = res["num_accepted"]
    for i in range(K):
        reached = (na >= i).sum()
        acc = (na >= i + 1).sum()
        sd = math.sqrt(beta[i] * (1 - beta[i]) / reached)
        assert abs(acc / reached - beta[i]) < 5 * sd
    for j in range(K + 1):
        pj = float(np.prod(beta[:j]))
        f = np.mean(na >= j)
        assert abs(f - pj) < 5 * math.sqrt(pj * (1 - pj) / n) + 1e-12


def test_p_equals_q_accepts_everything(oracle_mod):
    """Identical target and draft rows: every ratio is 1, all K drafts pass and
    the last token is a bonus draw from p_K."""
    from scipy import stats
    V, K, n = 7, 3, 300_000
    t, d, tokens, res = _mc(oracle_mod, V, K, n, 1.0, seed=99, same=True)
    assert (res["num_accepted"] == K).all()
    np.testing.assert_array_equal(res["out_tokens"][:, :K], tokens)
    assert np.nanmax(np.abs(res["log_ratio"])) == 0.0
    counts = np.bincount(res["out_tokens"][:, K], minlength=V)
    p = softmax64(t[K])
    assert stats.chisquare(counts, p * n).pvalue > 1e-3


def test_temperature_scales_both_rows(oracle_mod):
    """With T = 0.5 and logits that are multiples of 1/4, l / T is exact, so the
    oracle at (l, T) must equal the oracle at (2 l, 1) bit for bit -- which
    holds only if T divides the draft rows as well as the target rows."""
    rng = np.random.default_rng(3)
    B, K, V = 64, 3, 17
    t = (rng.integers(-16, 16, size=(B, K + 1, V)) / 4).astype(np.float32)
    d = (rng.integers(-16, 16, size=(B, K, V)) / 4).astype(np.float32)
    tokens = draw_tokens(rng, softmax64(d, 0.5))
    a = oracle_mod.verify(t, d, tokens, 0.5, seed=5)
    b = oracle_mod.verify(2 * t, 2 * d, tokens, 1.0, seed=5)
    for k in ("out_tokens", "num_accepted"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(a["lse_t"], b["lse_t"])
    c = oracle_mod.verify(t, 2 * d, tokens, 0.5, seed=5)  # T on the target only would look like this
    assert not np.array_equal(c["lse_d"], a["lse_d"])


def test_truncation_and_padding(oracle_mod):
    """Position 0 certain to pass (p = q), position 1 certain to fail (p(x_1) = 0):
    exactly one draft is kept, position 1 holds a residual token != x_1, the
    rest is -1."""
    V, K = 6, 4
    rng = np.random.default_rng(8)
    t = rng.normal(size=(K + 1, V)).astype(np.float32)
    d = rng.normal(size=(K, V)).astype(np.float32)
    d[0] = t[0]
    x = np.array([2, 3, 1, 0], dtype=np.int32)
    t[1, 3] = -np.inf
    res = oracle_mod.verify(t[None], d[None], x[None], 1.0, seed=1)
    assert res["num_accepted"][0] == 1
    out = res["out_tokens"][0]
    assert out[0] == 2 and out[1] != 3 and out[1] >= 0
    assert (out[2:] == -1).all()


def test_greedy_semantics(oracle_mod):
    """Greedy: accept while the target argmax equals the draft; emit the target
    argmax at the first mismatch, or the bonus row's argmax; ties go to the
    lowest index; temperature plays no part."""
    t = np.array([[[0, 5, 1, 5], [9, 0, 0, 0], [0, 0, 2, 2], [1, 1, 1, 1]]], dtype=np.float32)
    # row argmaxes: 1, 0, 2, 0
    for T in (1.0, 0.3):
        r = oracle_mod.verify(t, None, np.array([[1, 0, 3]], dtype=np.int32), T, 0, mode=1)
        assert r["num_accepted"][0] == 2
        assert list(r["out_tokens"][0]) == [1, 0, 2, -1]
    r = oracle_mod.verify(t, None, np.array([[1, 0, 2]], dtype=np.int32), 1.0, 0, mode=1)
    assert r["num_accepted"][0] == 3 and list(r["out_tokens"][0]) == [1, 0, 2, 0]
    r = oracle_mod.verify(t, None, np.array([[3, 0, 2]], dtype=np.int32), 1.0, 0, mode=1)
    assert r["num_accepted"][0] == 0 and list(r["out_tokens"][0]) == [1, -1, -1, -1]


def test_invalid_inputs_are_reported(oracle_mod):
    o = oracle_mod
    V, K = 5, 2
    base_t = np.zeros((3, K + 1, V), dtype=np.float32)
    base_d = np.zeros((3, K, V), dtype=np.float32)
    tok = np.zeros((3, K), dtype=np.int32)
    t = base_t.copy()
    t[0, 1, 2] = np.nan
    t[1, 2, :] = -np.inf
    d = base_d.copy()
    d[2, 0, 4] = np.inf
    r = o.verify(t, d, tok, 1.0, 0)
    assert list(r["seq_status"]) == [o.NONFINITE] * 3
    assert (r["num_accepted"] == -1).all() and (r["out_tokens"] == -1).all()
    tok2 = tok.copy()
    tok2[1, 1] = V
    tok2[2, 0] = -1
    r = o.verify(base_t, base_d, tok2, 1.0, 0)
    assert list(r["seq_status"]) == [0, o.BAD_TOKEN, o.BAD_TOKEN]
    assert r["num_accepted"][0] == K  # uniform rows, p = q
    tg = base_t.copy()
    tg[0, 0, 0] = np.nan
    tg[1, :, :] = -np.inf  # all -inf is a valid greedy row (argmax 0)
    r = o.verify(tg, None, tok, 1.0, 0, mode=1)
    assert list(r["seq_status"]) == [o.NONFINITE, 0, 0]
    assert r["num_accepted"][1] == K and r["num_accepted"][2] == K


def test_zero_drafts_is_plain_sampling(oracle_mod):
    """K = 0: no draft to check, the single token is a draw from the target row."""
    from scipy import stats
    V, n = 4, 200_000
    row = np.array([0.5, -1.0, 2.0, 0.0], dtype=np.float32)
    t = np.broadcast_to(row, (n, 1, V)).copy()
    r = oracle_mod.verify(t, None, np.zeros((n, 0), dtype=np.int32), 1.0, seed=12)
    assert (r["num_accepted"] == 0).all()
    counts = np.bincount(r["out_tokens"][:, 0], minlength=V)
    assert stats.chisquare(counts, softmax64(row) * n).pvalue > 1e-3


def test_threads_do_not_change_results(oracle_mod):
    rng = np.random.default_rng(1)
    B, K, V = 37, 3, 50
    t = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    d = rng.normal(size=(B, K, V)).astype(np.float32)
    tok = draw_tokens(rng, softmax64(d))
    a = oracle_mod.verify(t, d, tok, 1.0, seed=4, threads=1)
    b = oracle_mod.verify(t, d, tok, 1.0, seed=4, threads=5)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_philox_many_is_philox_per_counter(oracle_mod):
    rng = np.random.default_rng(5)
    ctr = rng.integers(0, 2**32, size=(257, 4), dtype=np.uint64).astype(np.uint32)
    key = np.array([0x89ABCDEF, 0x01234567], dtype=np.uint32)
    many = oracle_mod.philox_many(ctr, key)
    for r in range(ctr.shape[0]):
        assert np.array_equal(many[r], oracle_mod.philox(ctr[r], key))


# --------------------------------------------------------------------------
# Top-k / top-p applied to both rows ([VN], paragraph on temperature, top-k
# and top-p). The filtered rows are p' and q'; every law above must hold with
# p' in place of p.
# --------------------------------------------------------------------------
def brute_filter(row, T, top_k, top_p):
    """The cut straight from its definition, by trying every value of the row
    as a threshold: top-k keeps the largest value v with #{x >= v} >= k;
    top-p, inside that set, the largest v whose upper set holds >= top_p of
    the set's mass. Returns (threshold, kept mask, p' over the row, margin)."""
    x = np.asarray(row, dtype=np.float64)
    V = x.size
    p = softmax64(x, T)
    cands = sorted(set(x.tolist()))
    tk = -math.inf
    if 0 < top_k < V:
        tk = max(v for v in cands if (x >= v).sum() >= top_k)
    mass_k = p[x >= tk].sum()
    thr, margin = tk, math.inf
    if top_p < 1.0:
        target = top_p * mass_k
        thr = max(v for v in cands if v >= tk and p[x >= v].sum() >= target)
        after, before = p[x >= thr].sum(), p[x > thr].sum()
        margin = min(after - target, target - before) / mass_k
    kept = x >= thr
    pf = np.where(kept, p, 0.0)
    return thr, kept, pf / pf.sum(), margin


def _tied_row(rng, V, T):
    """Logits on a coarse grid, so that ties are common."""
    return (rng.integers(-8, 8, size=V) / 2).astype(np.float32)


@pytest.mark.parametrize("top_k,top_p", [(0, 1.0), (1, 1.0), (3, 1.0), (5, 1.0), (0, 0.3),
                                         (0, 0.9), (4, 0.5), (6, 0.95), (2, 0.01), (11, 0.7)])
@pytest.mark.parametrize("T", [1.0, 0.6])
def test_filter_row_against_brute_force(oracle_mod, top_k, top_p, T):
    rng = np.random.default_rng(17 + top_k)
    for trial in range(40):
        V = int(rng.integers(1, 14))
        row = _tied_row(rng, V, T) if trial % 2 else rng.normal(size=V).astype(np.float32)
        lse = np.log(np.exp(row.astype(np.float64) / T).sum())
        thr, log_mass, margin = oracle_mod.filter_row(row, T, lse, top_k, top_p)
        bthr, kept, pf, bmargin = brute_filter(row, T, top_k, top_p)
        assert thr == bthr, (row, top_k, top_p)
        p = softmax64(row, T)
        assert math.isclose(log_mass, math.log(p[kept].sum()), rel_tol=1e-12, abs_tol=1e-12)
        if math.isinf(bmargin):
            assert math.isinf(margin)
        else:
            assert math.isclose(margin, bmargin, rel_tol=1e-9, abs_tol=1e-12)


def test_filter_row_closed_forms(oracle_mod):
    """p proportional to [4, 2, 1, 1]: top-p walks the groups 1/2, 3/4, 1 (the
    two 1s are one group, kept or dropped together)."""
    row = np.log(np.array([4.0, 2.0, 1.0, 1.0])).astype(np.float32)
    lse = float(np.log(np.exp(row.astype(np.float64)).sum()))
    r = {}
    for top_k, top_p in [(0, 0.45), (0, 0.6), (0, 0.85), (1, 1.0), (3, 1.0), (3, 0.4), (0, 1.0)]:
        r[(top_k, top_p)] = oracle_mod.filter_row(row, 1.0, lse, top_k, top_p)
    p = softmax64(row)
    assert r[(0, 0.45)][0] == row[0] and math.isclose(r[(0, 0.45)][2], 0.05 / 1.0, rel_tol=1e-6)
    assert r[(0, 0.6)][0] == row[1] and math.isclose(r[(0, 0.6)][2], 0.1, rel_tol=1e-6)
    # the boundary group holds both 1s: margin = min(1 - 0.85, 0.85 - 0.75)
    assert r[(0, 0.85)][0] == row[2] and math.isclose(r[(0, 0.85)][2], 0.1, rel_tol=1e-6)
    assert r[(1, 1.0)][0] == row[0] and math.isclose(r[(1, 1.0)][1], math.log(p[0]))
    # third-largest value is a tie: top-3 keeps all four tokens
    assert r[(3, 1.0)][0] == row[2] and abs(r[(3, 1.0)][1]) < 1e-12
    # top-p inside the top-3 set (all of it here): 0.4 of it is reached by {4}
    assert r[(3, 0.4)][0] == row[0]
    assert r[(0, 1.0)][0] == -math.inf and math.isinf(r[(0, 1.0)][2])


def test_filters_off_change_nothing(oracle_mod):
    rng = np.random.default_rng(8)
    B, K, V = 40, 3, 30
    t = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    d = rng.normal(size=(B, K, V)).astype(np.float32)
    tok = draw_tokens(rng, softmax64(d))
    a = oracle_mod.verify(t, d, tok, 1.0, seed=6)
    for top_k, top_p in [(0, 1.0), (V, 1.0), (V + 5, 1.0), (-1, 1.0)]:
        b = oracle_mod.verify(t, d, tok, 1.0, seed=6, top_k=top_k, top_p=top_p)
        for k in a:
            np.testing.assert_array_equal(a[k], b[k])


def _draw_filtered(rng, rows, T, top_k, top_p, n):
    """n draws per position from the brute-force filtered rows [K, V]."""
    q = np.stack([brute_filter(r, T, top_k, top_p)[2] for r in rows])
    return draw_tokens(rng, np.broadcast_to(q, (n,) + q.shape))


@pytest.mark.parametrize("V,K,top_k,top_p", [(8, 2, 4, 1.0), (8, 3, 0, 0.8), (10, 2, 6, 0.75),
                                             (6, 2, 2, 1.0)])
def test_filtered_output_marginal_chisquare(oracle_mod, V, K, top_k, top_p):
    """With both rows filtered and drafts drawn from q', the token emitted at
    every reached position follows the filtered target p'."""
    from scipy import stats
    n, T = 300_000, 0.8
    Tw = float(np.float32(T))
    rng = np.random.default_rng(V * 1000 + K * 10 + top_k)
    t, d = _random_rows(rng, K, V)
    d = (0.7 * t[:K] + 0.5 * d).astype(np.float32)  # a draft that overlaps the target
    tokens = _draw_filtered(rng, d, Tw, top_k, top_p, n)
    res = oracle_mod.verify(np.broadcast_to(t, (n, K + 1, V)).copy(),
                            np.broadcast_to(d, (n, K, V)).copy(), tokens, T, seed=77,
                            threads=8, top_k=top_k, top_p=top_p)
    assert (res["seq_status"] == 0).all()
    na = res["num_accepted"]
    for i in range(K + 1):
        pf = brute_filter(t[i], Tw, top_k, top_p)[2]
        sel = na >= i
        assert sel.sum() > n // 50, (i, sel.sum())
        counts = np.bincount(res["out_tokens"][sel, i], minlength=V)
        assert counts[pf == 0].sum() == 0, (i, counts, pf)
        keep = pf > 0
        if keep.sum() > 1:
            pv = stats.chisquare(counts[keep], pf[keep] * sel.sum()).pvalue
            assert pv > 1e-3 / (K + 1), (i, counts, pf)


def test_filtered_acceptance_rate(oracle_mod):
    """P(accept at 0) = sum_x min(p'(x), q'(x)) with x ~ q'."""
    n, V, K, T, top_k, top_p = 400_000, 9, 1, 1.0, 5, 0.85
    rng = np.random.default_rng(31)
    t, d = _random_rows(rng, K, V)
    tokens = _draw_filtered(rng, d, T, top_k, top_p, n)
    res = oracle_mod.verify(np.broadcast_to(t, (n, K + 1, V)).copy(),
                            np.broadcast_to(d, (n, K, V)).copy(), tokens, T, seed=5, threads=8,
                            top_k=top_k, top_p=top_p)
    beta = np.minimum(brute_filter(t[0], T, top_k, top_p)[2],
                      brute_filter(d[0], T, top_k, top_p)[2]).sum()
    f = np.mean(res["num_accepted"] >= 1)
    assert abs(f - beta) < 5 * math.sqrt(beta * (1 - beta) / n)


def test_token_outside_filtered_rows_is_rejected(oracle_mod):
    """top-k = 1 on rows that share their maximum: p' = q' = one-hot at it. A
    draft token anywhere else has p'(x) = q'(x) = 0 and is rejected; the
    residual is empty, so the emitted token is the draw from p': the maximum."""
    V, K, B = 12, 3, 64
    rng = np.random.default_rng(2)
    t = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    d = rng.normal(size=(B, K, V)).astype(np.float32)
    t[:, :, 5] = 10.0
    d[:, :, 5] = 9.0
    tok = np.full((B, K), 5, dtype=np.int32)
    pos = rng.integers(0, K, size=B)
    other = rng.integers(0, V - 1, size=B)
    other = other + (other >= 5)
    tok[np.arange(B), pos] = other
    r = oracle_mod.verify(t, d, tok, 1.0, seed=3, top_k=1)
    np.testing.assert_array_equal(r["num_accepted"], pos)
    np.testing.assert_array_equal(r["out_tokens"][np.arange(B), pos], 5)
    # unfiltered, the same tokens have p, q > 0 and some survive
    u = oracle_mod.verify(t, d, tok, 1.0, seed=3)
    assert (u["num_accepted"] > pos).any()


def test_filtered_p_equals_q_accepts_everything(oracle_mod):
    from scipy import stats
    V, K, n, top_k, top_p = 9, 2, 200_000, 6, 0.9
    rng = np.random.default_rng(12)
    t, _ = _random_rows(rng, K, V)
    tokens = _draw_filtered(rng, t[:K], 1.0, top_k, top_p, n)
    res = oracle_mod.verify(np.broadcast_to(t, (n, K + 1, V)).copy(),
                            np.broadcast_to(t[:K], (n, K, V)).copy(), tokens, 1.0, seed=9,
                            threads=8, top_k=top_k, top_p=top_p)
    assert (res["num_accepted"] == K).all()
    pf = brute_filter(t[K], 1.0, top_k, top_p)[2]
    counts = np.bincount(res["out_tokens"][:, K], minlength=V)
    keep = pf > 0
    assert counts[~keep].sum() == 0
    assert stats.chisquare(counts[keep], pf[keep] * n).pvalue > 1e-3


def test_filter_margins_reported(oracle_mod):
    rng = np.random.default_rng(4)
    B, K, V, top_p = 20, 2, 15, 0.7
    t = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    d = rng.normal(size=(B, K, V)).astype(np.float32)
    tok = draw_tokens(rng, softmax64(d))
    r = oracle_mod.verify(t, d, tok, 1.0, seed=1, top_k=8, top_p=top_p)
    for b in range(B):
        for i in range(K + 1):
            assert math.isclose(r["filter_margin_t"][b, i],
                                brute_filter(t[b, i], 1.0, 8, float(np.float32(top_p)))[3],
                                rel_tol=1e-9, abs_tol=1e-12)
        for i in range(K):
            assert math.isclose(r["filter_margin_d"][b, i],
                                brute_filter(d[b, i], 1.0, 8, float(np.float32(top_p)))[3],
                                rel_tol=1e-9, abs_tol=1e-12)
        # per-row thresholds and log kept masses, target rows then draft rows
        rows = list(t[b]) + list(d[b])
        for i, row in enumerate(rows):
            thr, kept, _, _ = brute_filter(row, 1.0, 8, float(np.float32(top_p)))
            assert r["filter_thr"][b, i] == thr
            assert math.isclose(r["filter_log_mass"][b, i],
                                math.log(softmax64(row)[kept].sum()), rel_tol=1e-9, abs_tol=1e-12)
    u = oracle_mod.verify(t, d, tok, 1.0, seed=1)
    assert np.all(u["filter_thr"] == -np.inf) and np.all(u["filter_log_mass"] == 0.0)
