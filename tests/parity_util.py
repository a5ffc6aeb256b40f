"""Comparison of the CUDA path with the float64 oracle (test infrastructure).

Bit-exact where the method is discrete (accepted counts, tokens, argmaxes,
status), except for decisions the oracle flags as near-ties: an acceptance
draw with |u - r| < 1e-5, or a sampling draw whose two-level exponential race
(blocks of 512 tokens) has, at either level, a relative gap
(best - second) / best below 1e-5 between its two largest scores w / E. A
flagged sequence is compared exactly up to its
first flagged decision; past it, either branch is correct, so the GPU output
is only checked to be a valid verification result. Normalisers and
log-ratios must agree to 1e-5 relative (absolute below magnitude 1).
"""
from __future__ import annotations

import numpy as np

FLAG = 1e-5
RTOL = 1e-5


def close(a, b, tol=RTOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.abs(a - b) <= tol * np.maximum(1.0, np.abs(b))


def valid_output(out, nacc, x, K, V):
    if not (0 <= nacc <= K):
        return False
    if nacc > 0 and not np.array_equal(out[:nacc], x[:nacc]):
        return False
    if not (0 <= out[nacc] < V):
        return False
    return bool(np.all(out[nacc + 1:] == -1))


def compare(gpu: dict, orc: dict, tokens: np.ndarray, K: int, V: int, rows=None, greedy=False,
            check_stats=True, flag=FLAG, rtol=RTOL) -> dict:
    """Compare GPU outputs with oracle outputs on sequences ``rows`` (all by default).

    ``gpu`` holds numpy arrays for the whole batch; ``orc`` holds the oracle's
    arrays for the whole batch (only ``rows`` need to be filled). ``flag`` and
    ``rtol`` widen the near-tie band and the normaliser tolerance where the
    GPU's inputs themselves carry rounding (logits it computed). Raises
    AssertionError on a mismatch; returns counts of decisions and flags.
    """
    B = gpu["num_accepted"].shape[0]
    rows = range(B) if rows is None else rows
    n_dec = n_flag_dec = n_flag_seq = n_flag_diff = 0
    for b in rows:
        sg, so = int(gpu["seq_status"][b]), int(orc["seq_status"][b])
        assert sg == so, f"seq {b}: status gpu {sg} oracle {so}"
        og, oo = gpu["out_tokens"][b], orc["out_tokens"][b]
        ng, no = int(gpu["num_accepted"][b]), int(orc["num_accepted"][b])
        if so != 0:
            assert ng == -1 and np.all(og == -1), f"seq {b}: invalid sequence not reported"
            continue
        x = tokens[b]
        if check_stats and not greedy:
            lt_ok = close(gpu["lse_t"][b], orc["lse_t"][b], rtol)
            assert lt_ok.all(), f"seq {b}: lse_t {gpu['lse_t'][b]} vs {orc['lse_t'][b]}"
            if K > 0:
                assert close(gpu["lse_d"][b], orc["lse_d"][b], rtol).all(), f"seq {b}: lse_d"
                assert close(gpu["log_ratio"][b], orc["log_ratio"][b], rtol).all(), \
                    f"seq {b}: log_ratio {gpu['log_ratio'][b]} vs {orc['log_ratio'][b]}"
        if greedy:
            n_dec += min(no + 1, K) + 1
            assert ng == no and np.array_equal(og, oo), f"seq {b}: greedy gpu {og} oracle {oo}"
            continue
        am = orc["accept_margin"][b].copy()
        s_flag = orc["sample_margin"][b] < flag
        if "filter_margin_t" in orc:
            # Top-p boundaries: a row whose boundary lies within FLAG of top_p
            # may keep one more or one fewer group of tokens on either side;
            # that flags every decision that uses the row.
            fm_t, fm_d = orc["filter_margin_t"][b], orc["filter_margin_d"][b]
            if K > 0:
                am = np.minimum(am, np.minimum(fm_t[:K], fm_d))
            s_flag = s_flag or fm_t[no] < flag or (no < K and fm_d[no] < flag)
        decisions = list(range(min(no + 1, K)))
        n_dec += len(decisions) + 1
        first_flag = next((i for i in decisions if am[i] < flag), None)
        if first_flag is not None:
            n_flag_seq += 1
            n_flag_dec += 1
            assert ng >= first_flag, f"seq {b}: diverged before flagged position {first_flag}"
            assert np.array_equal(og[:first_flag], oo[:first_flag])
            assert valid_output(og, ng, x, K, V), f"seq {b}: invalid GPU output {og}"
            n_flag_diff += int(ng != no or not np.array_equal(og, oo))
        elif s_flag:
            n_flag_seq += 1
            n_flag_dec += 1
            assert ng == no, f"seq {b}: num_accepted gpu {ng} oracle {no}"
            assert np.array_equal(og[:no], oo[:no])
            assert valid_output(og, ng, x, K, V), f"seq {b}: invalid GPU output {og}"
            n_flag_diff += int(og[no] != oo[no])
        else:
            assert ng == no, f"seq {b}: num_accepted gpu {ng} oracle {no} (out {og} vs {oo})"
            assert np.array_equal(og, oo), f"seq {b}: tokens gpu {og} oracle {oo}"
    return {"decisions": n_dec, "flagged_decisions": n_flag_dec, "flagged_sequences": n_flag_seq,
            "flagged_differing": n_flag_diff}


# The parity rule's budget for near-ties: under 0.01% of decisions.
FLAG_BUDGET = 1e-4


def oracle_flag_counts(orc: dict, K: int, flag=FLAG) -> tuple:
    """(decisions, flagged) over every decision the oracle took, counting each
    flagged decision (not only a sequence's first): the acceptance draws at
    positions 0 .. min(j, K - 1) and the one draw of the emitted token.
    Invalid sequences take no decision."""
    ok = orc["seq_status"] == 0
    j = orc["num_accepted"][ok].astype(np.int64)
    am = orc["accept_margin"][ok]
    taken = np.arange(K)[None, :] <= np.minimum(j, K - 1)[:, None] if K > 0 else \
        np.zeros((len(j), 0), dtype=bool)
    n_acc = int(taken.sum())
    f_acc = int((taken & (am < flag)).sum())
    f_smp = int((orc["sample_margin"][ok] < flag).sum())
    return n_acc + len(j), f_acc + f_smp


def flag_count_plausible(flagged: int, decisions: int, budget=FLAG_BUDGET, alpha=1e-6) -> bool:
    """True unless ``flagged`` near-ties in ``decisions`` would be implausible
    (one-sided binomial tail below ``alpha``) at a flag rate of ``budget``."""
    from scipy import stats
    if flagged == 0:
        return True
    return bool(stats.binom.sf(flagged - 1, decisions, budget) >= alpha)


def flag_rate_upper_bound(flagged: int, decisions: int, conf=0.99) -> float:
    """One-sided Clopper-Pearson upper confidence bound of a binomial rate."""
    from scipy import stats
    if flagged >= decisions:
        return 1.0
    return float(stats.beta.ppf(conf, flagged + 1, decisions - flagged))
