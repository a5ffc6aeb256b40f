"""Pins for the oracle's LM head (logits = h W^T from bfloat16 operands) and
for its float64 logits input, all on the CPU.

The pages take each model's logits as given ("Как работает speculative
decoding на уровне логитов..." (aivaro.ru) §4 and §5 step 1: a vector of V
logits per position); the output layer that makes them is the product h W^T.
The pins fix that product independently of numpy's matmul: brute-force sums
in exact rational arithmetic, one-hot hidden states selecting columns, exact
scaling; and they fix the float64 reader of the verification oracle against
its float32 reader on values both represent exactly.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def bf16(x):
    """Round-to-nearest-even float32 -> bfloat16 bit patterns (input generation)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_bf16_bits_to_f64_known_values():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F80, 0xFF80, 0x3F00],
                    dtype=np.uint16)
    v = oracle.bf16_bits_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -1.0 and v[2] == 3.140625 and v[3] == 0.0
    assert np.signbit(v[4]) and v[5] == np.inf and v[6] == -np.inf and v[7] == 0.5
    assert np.isnan(oracle.bf16_bits_to_f64(np.array([0x7FC0], dtype=np.uint16)))[0]


@pytest.mark.parametrize("R,D,V", [(1, 1, 1), (3, 5, 4), (2, 17, 9), (4, 64, 3)])
def test_lm_head_matches_exact_rational_sums(R, D, V):
    rng = np.random.default_rng(R * 100 + D * 10 + V)
    h = bf16(rng.standard_normal((R, D)) * 3)
    w = bf16(rng.standard_normal((V, D)))
    got = oracle.lm_head_logits(h, w)
    hv, wv = oracle.bf16_bits_to_f64(h), oracle.bf16_bits_to_f64(w)
    for r in range(R):
        for v in range(V):
            exact = sum(Fraction(float(hv[r, d])) * Fraction(float(wv[v, d])) for d in range(D))
            # float64 sum of D exact products: within D 2^-53 of the sum of |terms|.
            bound = D * 2.0 ** -53 * float(sum(abs(hv[r, d] * wv[v, d]) for d in range(D)))
            assert abs(got[r, v] - float(exact)) <= bound


def test_one_hot_hidden_states_select_columns_of_w():
    rng = np.random.default_rng(1)
    D, V = 24, 11
    w = bf16(rng.standard_normal((V, D)))
    h = np.zeros((D, D), dtype=np.uint16)
    h[np.arange(D), np.arange(D)] = 0x3F80  # 1.0
    got = oracle.lm_head_logits(h, w)
    assert np.array_equal(got, oracle.bf16_bits_to_f64(w).T)  # row d = column d of W


def test_logits_scale_exactly_with_a_power_of_two_hidden_state():
    rng = np.random.default_rng(2)
    h = bf16(rng.standard_normal((3, 40)))
    w = bf16(rng.standard_normal((7, 40)))
    h2 = bf16(oracle.bf16_bits_to_f64(h) * 4.0)  # exact in bfloat16
    assert np.array_equal(oracle.lm_head_logits(h2, w), 4.0 * oracle.lm_head_logits(h, w))


def test_leading_batch_dimensions_and_transpose():
    rng = np.random.default_rng(3)
    h = bf16(rng.standard_normal((2, 3, 8)))
    w = bf16(rng.standard_normal((5, 8)))
    got = oracle.lm_head_logits(h, w)
    assert got.shape == (2, 3, 5)
    # Logit (b, i, v) pairs row (b, i) of h with row v of W, not column v.
    hv, wv = oracle.bf16_bits_to_f64(h), oracle.bf16_bits_to_f64(w)
    assert got[1, 2, 4] == pytest.approx(float(np.dot(hv[1, 2], wv[4])), abs=1e-12)
    with pytest.raises(ValueError):
        oracle.lm_head_logits(h, bf16(rng.standard_normal((5, 9))))


@pytest.mark.parametrize("mode", [oracle.SAMPLE, oracle.GREEDY])
def test_float64_logits_read_like_float32_on_shared_values(mode):
    """Logits that float32 represents exactly give identical results through
    the float64 reader and the float32 reader (strides, rows, every output)."""
    rng = np.random.default_rng(4)
    B, K, V = 5, 3, 301
    t32 = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    d32 = (t32[:, :K] + 0.5 * rng.standard_normal((B, K, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    draft32 = d32 if mode == oracle.SAMPLE else None
    draft64 = None if draft32 is None else draft32.astype(np.float64)
    a = oracle.verify(t32, draft32, tok, 0.9, 77, mode)
    b = oracle.verify(t32.astype(np.float64), draft64, tok, 0.9, 77, mode)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_verify_lmhead_is_verify_on_the_products_and_ranges_agree():
    rng = np.random.default_rng(5)
    B, K, V, Dt, Dd = 6, 3, 97, 24, 16
    ht = bf16(rng.standard_normal((B, K + 1, Dt)))
    wt = bf16(rng.standard_normal((V, Dt)) * 0.4)
    hd = bf16(rng.standard_normal((B, K, Dd)))
    wd = bf16(rng.standard_normal((V, Dd)) * 0.5)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    full = oracle.verify_lmhead(ht, wt, hd, wd, tok, 0.8, 9)
    ref = oracle.verify(oracle.lm_head_logits(ht, wt), oracle.lm_head_logits(hd, wd), tok, 0.8, 9)
    for k in ref:
        assert np.array_equal(full[k], ref[k], equal_nan=True), k
    part = oracle.verify_lmhead(ht, wt, hd, wd, tok, 0.8, 9, seq_range=(2, 5))
    for k in ref:
        assert np.array_equal(part[k][2:5], ref[k][2:5], equal_nan=True), k
    assert (part["num_accepted"][:2] == -7).all() and (part["num_accepted"][5:] == -7).all()
    g = oracle.verify_lmhead(ht, wt, None, None, tok, 1.0, 9, mode=oracle.GREEDY)
    gref = oracle.verify(oracle.lm_head_logits(ht, wt), None, tok, 1.0, 9, oracle.GREEDY)
    assert np.array_equal(g["out_tokens"], gref["out_tokens"])
