"""Pins of the CUDA path that hold whatever the oracle says about single
inputs: the device Philox4x32-10 generator word for word against the oracle's
independent implementation, and the law of the emitted tokens over many
sequences (the target distribution, by the rejection-sampling argument of
"Speculative decoding" (aihero.vn), section on accepting by ratio, and
Hung-yi Lee's lecture 16 notes, §4 item 4 for the bonus row).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_66_gb300 as sv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()
    torch.cuda.set_device(0)


def _counters(n, rng):
    """Random counters plus the structured ones the verification kernels use:
    acceptance (i, b, 0, 0), race (k div 4 + 1 with the level in word 3), and
    the extremes of each word."""
    c = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    i, b = np.meshgrid(np.arange(64, dtype=np.uint32), np.arange(64, dtype=np.uint32))
    acc = np.stack([i.ravel(), b.ravel(), 0 * i.ravel(), 0 * i.ravel()], 1)
    race = np.stack([i.ravel(), b.ravel(), 1 + i.ravel(), (b.ravel() & 1)], 1)
    ext = np.array([[0, 0, 0, 0], [0xFFFFFFFF] * 4, [0xFFFFFFFF, 0, 0xFFFFFFFF, 0],
                    [1, 2, 3, 4]], dtype=np.uint32)
    return np.concatenate([c, acc.astype(np.uint32), race.astype(np.uint32), ext])


@pytest.mark.parametrize("seed", [0, 0x5EED0002, 0xFFFFFFFFFFFFFFFF, 0x0123456789ABCDEF])
def test_device_philox_matches_oracle(seed):
    rng = np.random.default_rng(seed & 0xFFFF)
    ctr = _counters(1 << 20, rng)
    dev = torch.from_numpy(ctr.view(np.int32)).cuda()
    got = sv.sv_philox(seed, dev)
    torch.cuda.synchronize()
    got = got.cpu().numpy().view(np.uint32)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
    want = oracle.philox_many(ctr, key)
    bad = np.nonzero(np.any(got != want, axis=1))[0]
    assert bad.size == 0, f"{bad.size} counters differ, first {ctr[bad[0]]}"


def test_device_philox_binding_checks_shape():
    c = torch.zeros((4, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        sv.sv_philox(0, c.view(-1))
    with pytest.raises(ValueError):
        sv.sv_philox(0, c.to(torch.int64))


def _law_case(V, K, B, seed):
    """One set of K + 1 target rows and K draft rows, shared by all B
    sequences; draft tokens x_i ~ q_i from numpy's generator (independent of
    the library's Philox streams)."""
    rng = np.random.default_rng(seed)
    t = (rng.normal(size=(K + 1, V)) * 1.2).astype(np.float32)
    d = (t[:K] + rng.normal(size=(K, V)) * 1.0).astype(np.float32)
    p = np.empty((K + 1, V))
    q = np.empty((K, V))
    for i in range(K + 1):
        _, lse = oracle.row_lse(t[i], 1.0)
        p[i] = [np.exp(oracle.log_prob(t[i], k, 1.0, lse)) for k in range(V)]
    for i in range(K):
        _, lse = oracle.row_lse(d[i], 1.0)
        q[i] = [np.exp(oracle.log_prob(d[i], k, 1.0, lse)) for k in range(V)]
    x = np.stack([rng.choice(V, size=B, p=q[i] / q[i].sum()) for i in range(K)], 1).astype(np.int32)
    return t, d, x, p, q


@pytest.mark.parametrize("V", [5, 8])  # 20-byte rows (staged sampler), 32-byte rows (streamed)
def test_emitted_tokens_follow_target_law(V):
    """Among sequences that reach position i, the token at i follows p_i; the
    bonus token (all K kept) follows p_K. Chi-square over 2^19 sequences with
    a Bonferroni-corrected threshold; the first acceptance rate also matches
    its closed form sum_x min(p_0(x), q_0(x)) to five standard deviations."""
    from scipy import stats
    K, B = 2, 1 << 19
    t, d, x, p, q = _law_case(V, K, B, 40 + V)
    tt = torch.from_numpy(t).cuda().unsqueeze(0).expand(B, K + 1, V).contiguous()
    dd = torch.from_numpy(d).cuda().unsqueeze(0).expand(B, K, V).contiguous()
    xx = torch.from_numpy(x).cuda()
    out, nacc = sv.spec_verify(tt, dd, xx, 1.0, 0xABCDEF + V, "sample")
    torch.cuda.synchronize()
    out, nacc = out.cpu().numpy(), nacc.cpu().numpy()
    assert np.all((nacc >= 0) & (nacc <= K))
    tests = 0
    pvals = []
    for i in range(K + 1):
        reached = nacc >= i
        toks = out[reached, i]
        assert np.all((toks >= 0) & (toks < V))
        counts = np.bincount(toks, minlength=V)
        pvals.append(stats.chisquare(counts, p[i] / p[i].sum() * counts.sum()).pvalue)
        tests += 1
    assert min(pvals) > 1e-3 / tests, pvals
    beta0 = np.minimum(p[0], q[0]).sum()
    rate = np.mean(nacc >= 1)
    assert abs(rate - beta0) < 5 * np.sqrt(beta0 * (1 - beta0) / B)
    # Tokens after the emitted position are -1, tokens before it the drafts.
    cols = np.arange(K + 1)[None, :]
    assert np.all(out[cols > nacc[:, None]] == -1)
    kept = cols < nacc[:, None]
    assert np.all(out[:, :K][kept[:, :K]] == x[kept[:, :K]])
