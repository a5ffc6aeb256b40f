"""Float64 CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE ONLY. This package wraps ``sv_oracle.c`` (plain C99,
double precision, single-threaded) with ctypes. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it; the CUDA library and its Python binding never do, and the two share no
code.

Parity status of each function (how it is pinned, see ``tests/test_oracle_*.py``):

* ``philox`` / ``uniform`` -- pinned against triton's independently written
  Philox4x32-10 run in its CPU interpreter, plus a uniformity chi-square.
* ``row_lse`` / ``log_prob`` -- pinned against ``torch.logsumexp`` /
  ``torch.log_softmax`` in float64 and closed forms on constant rows.
* ``accept_prob`` / ``sample_weights`` / ``race_sample`` / ``verify`` --
  pinned by the pages' two worked two-token examples, the p == q special case,
  exact path sums on tiny vocabularies (output law == target law), Monte-Carlo
  chi-square of the output marginal and of the race alone (for race block
  lengths 1, 7, 512 and V), the race's near-tie law, closed-form acceptance
  rates, and, at one block (block length >= V), token-for-token equality with
  a plain one-level race written out in the test.
* ``row_argmax`` -- pinned against ``torch.argmax`` (first occurrence).

* ``lm_head_logits`` / ``verify_lmhead`` -- the LM head h W^T (the pages take
  each model's logits as given; this is the product a language model's output
  layer computes), pinned by brute-force sums on tiny inputs, one-hot hidden
  states that pick out one column of W, and linearity; then ``verify`` on the
  float64 logits.

Arrays: float32 logits are passed as ``np.float32``; bfloat16 logits as their
raw 16-bit patterns in ``np.uint16``; float64 logits (the LM head's exact
products) as ``np.float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_HDR = os.path.join(_HERE, "sv_oracle.h")
_LIB = os.path.join(_HERE, "libsvoracle.so")

F32, BF16, F64 = 0, 1, 2
SAMPLE, GREEDY = 0, 1
BAD_TOKEN, NONFINITE = 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libsvoracle.so`` with gcc (no fast-math: IEEE double throughout)."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest_src:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    """The oracle's shared library. ``SVO_LIB_PATH`` names a different build of
    the same source (the mutation tests load deliberately broken copies)."""
    global _lib
    with _lock:
        if _lib is None:
            override = os.environ.get("SVO_LIB_PATH")
            L = ctypes.CDLL(override if override else build())
            vp, i64, i32, dbl, u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_uint64)
            L.svo_philox4x32_10.argtypes = [vp, vp, vp]
            L.svo_philox_many.argtypes = [vp, i64, vp, vp]
            L.svo_philox4x32_10.restype = None
            L.svo_philox_many.restype = None
            L.svo_uniform.argtypes = [u64, ctypes.c_uint32, ctypes.c_uint32, i32]
            L.svo_uniform.restype = dbl
            L.svo_elem.argtypes = [vp, i64, i32]
            L.svo_elem.restype = dbl
            L.svo_row_lse.argtypes = [vp, i64, i32, dbl, vp]
            L.svo_row_lse.restype = i32
            L.svo_log_prob.argtypes = [vp, i64, i32, dbl, dbl]
            L.svo_log_prob.restype = dbl
            L.svo_accept_prob.argtypes = [dbl, dbl]
            L.svo_accept_prob.restype = dbl
            L.svo_sample_weights.argtypes = [vp, vp, i64, i32, dbl, dbl, dbl, vp]
            L.svo_sample_weights.restype = None
            L.svo_race_uniform.argtypes = [u64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
            L.svo_race_uniform.restype = dbl
            L.svo_block_uniform.argtypes = [u64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
            L.svo_block_uniform.restype = dbl
            L.svo_race_sample.argtypes = [vp, i64, i64, u64, ctypes.c_uint32, ctypes.c_uint32,
                                          vp]
            L.svo_race_sample.restype = i64
            L.svo_row_argmax.argtypes = [vp, i64, i32, vp]
            L.svo_row_argmax.restype = i64
            L.svo_verify.argtypes = [vp, vp, vp, i64, i64, i64, i32, dbl, u64, i32, i64, i64,
                                     i64, vp, vp, vp, vp, vp, vp, vp, vp]
            L.svo_verify.restype = i32
            L.svo_verify_filtered.argtypes = [vp, vp, vp, i64, i64, i64, i32, dbl, u64, i32, i64,
                                              i64, dbl, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp, vp, vp, vp]
            L.svo_verify_filtered.restype = i32
            L.svo_filter_row.argtypes = [vp, i64, i32, dbl, dbl, i64, dbl, vp, vp, vp]
            L.svo_filter_row.restype = i32
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"logits must be float32, uint16 (bfloat16 bits) or float64, got {a.dtype}")


def philox(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().svo_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def philox_many(ctr, key) -> np.ndarray:
    """Philox4x32-10 of each row of an [n, 4] counter array."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(-1, 4)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros_like(c)
    lib().svo_philox_many(_ptr(c), c.shape[0], _ptr(k), _ptr(out))
    return out


def uniform(seed: int, seq: int, pos: int, lane: int) -> float:
    return lib().svo_uniform(seed, seq, pos, lane)


def elem(row: np.ndarray, k: int) -> float:
    row = np.ascontiguousarray(row)
    return lib().svo_elem(_ptr(row), k, _dtype_code(row))


def row_lse(row: np.ndarray, T: float):
    """Returns (status, lse)."""
    row = np.ascontiguousarray(row)
    out = np.zeros(1, dtype=np.float64)
    st = lib().svo_row_lse(_ptr(row), row.shape[-1], _dtype_code(row), T, _ptr(out))
    return st, float(out[0])


def log_prob(row: np.ndarray, k: int, T: float, lse: float) -> float:
    row = np.ascontiguousarray(row)
    return lib().svo_log_prob(_ptr(row), k, _dtype_code(row), T, lse)


def accept_prob(log_p: float, log_q: float) -> float:
    return lib().svo_accept_prob(log_p, log_q)


def sample_weights(target_row, draft_row, T: float, lse_t: float, lse_d: float) -> np.ndarray:
    t = np.ascontiguousarray(target_row)
    d = None if draft_row is None else np.ascontiguousarray(draft_row)
    if d is not None and d.dtype != t.dtype:
        raise TypeError("target and draft rows must share a dtype")
    w = np.zeros(t.shape[-1], dtype=np.float64)
    lib().svo_sample_weights(_ptr(t), _ptr(d), t.shape[-1], _dtype_code(t), T, lse_t, lse_d,
                             _ptr(w))
    return w


def race_uniform(seed: int, seq: int, pos: int, k: int) -> float:
    return lib().svo_race_uniform(seed, seq, pos, k)


# Block length of the corrected / bonus token's two-level race in ``verify``.
# The pages fix only the law of that draw, which the race meets for every block
# length; the length decides which random numbers are used. 512 is the length
# the CUDA library streams its block sums at, so it is the verifier's default.
RACE_BLOCK = 512


def block_uniform(seed: int, seq: int, pos: int, c: int) -> float:
    return lib().svo_block_uniform(seed, seq, pos, c)


def race_sample(w: np.ndarray, seed: int, seq: int, pos: int, block: int = RACE_BLOCK):
    """Two-level race over blocks of ``block`` tokens; returns (token, margin)."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    tok = lib().svo_race_sample(_ptr(w), w.shape[0], int(block), seed, seq, pos, _ptr(m))
    return int(tok), float(m[0])


def row_argmax(row: np.ndarray):
    """Returns (index, has_nan)."""
    row = np.ascontiguousarray(row)
    flag = np.zeros(1, dtype=np.int32)
    k = lib().svo_row_argmax(_ptr(row), row.shape[-1], _dtype_code(row), _ptr(flag))
    return int(k), bool(flag[0])


def filter_row(row: np.ndarray, T: float, lse: float, top_k: int, top_p: float):
    """Top-k / top-p cut of one row: (threshold logit, log kept mass, top-p margin)."""
    row = np.ascontiguousarray(row)
    out = np.zeros(3)
    lib().svo_filter_row(_ptr(row), row.shape[-1], _dtype_code(row), T, lse, int(top_k),
                         float(top_p), _ptr(out[0:1]), _ptr(out[1:2]), _ptr(out[2:3]))
    return float(out[0]), float(out[1]), float(out[2])


def verify(target: np.ndarray, draft, tokens, temperature: float, seed: int, mode: int = SAMPLE,
           threads: int = 1, seq_range=None, top_k: int = 0, top_p: float = 1.0,
           race_block: int = RACE_BLOCK) -> dict:
    """Run the oracle over a batch.

    target: [B, K+1, V] float32 or uint16 (bf16 bits); draft: [B, K, V] or None
    (greedy); tokens: [B, K] int32. ``temperature`` is widened from the float32
    value the CUDA path receives. ``threads`` > 1 splits the sequences into
    contiguous ranges run on a thread pool (the C code is unchanged and holds no
    shared state). ``seq_range=(b0, b1)`` restricts the work; outputs outside it
    are left at their fill values. ``top_k`` / ``top_p`` filter both rows of
    every position (0 and 1.0: off); ``top_p`` is widened from float32 like T.
    ``race_block`` is the block length of the corrected / bonus token's race.
    """
    target = np.ascontiguousarray(target)
    if target.ndim != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    dt = _dtype_code(target)
    if draft is not None:
        draft = np.ascontiguousarray(draft)
        if draft.dtype != target.dtype or draft.shape != (B, K, V):
            raise ValueError("draft must match target's dtype and be [B, K, V]")
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(B, K))
    T = float(np.float32(temperature))
    out = {
        "out_tokens": np.full((B, K + 1), -7, dtype=np.int32),
        "num_accepted": np.full(B, -7, dtype=np.int32),
        "lse_t": np.full((B, K + 1), np.nan),
        "lse_d": np.full((B, K), np.nan),
        "log_ratio": np.full((B, K), np.nan),
        "accept_margin": np.full((B, K), np.nan),
        "sample_margin": np.full(B, np.nan),
        "filter_margin_t": np.full((B, K + 1), np.inf),
        "filter_margin_d": np.full((B, K), np.inf),
        "filter_thr": np.full((B, 2 * K + 1), np.nan),
        "filter_log_mass": np.full((B, 2 * K + 1), np.nan),
        "seq_status": np.full(B, -7, dtype=np.int32),
    }
    P = float(np.float32(top_p))
    b0, b1 = (0, B) if seq_range is None else seq_range
    L = lib()

    def run(lo, hi):
        rc = L.svo_verify_filtered(_ptr(target), _ptr(draft), _ptr(tokens), B, K, V, dt, T,
                                   seed, mode, int(race_block), int(top_k), P, lo, hi,
                                   _ptr(out["out_tokens"]), _ptr(out["num_accepted"]),
                                   _ptr(out["lse_t"]), _ptr(out["lse_d"]), _ptr(out["log_ratio"]),
                                   _ptr(out["accept_margin"]), _ptr(out["sample_margin"]),
                                   _ptr(out["filter_margin_t"]), _ptr(out["filter_margin_d"]),
                                   _ptr(out["filter_thr"]), _ptr(out["filter_log_mass"]),
                                   _ptr(out["seq_status"]))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")

    n = b1 - b0
    threads = max(1, min(int(threads), n if n > 0 else 1))
    if threads == 1:
        run(b0, b1)
    else:
        bounds = [b0 + (n * t) // threads for t in range(threads + 1)]
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda t: run(bounds[t], bounds[t + 1]), range(threads)))
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to float64, exactly: the 16 bits are the
    high half of a binary32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def lm_head_logits(hidden_bits: np.ndarray, weight_bits: np.ndarray) -> np.ndarray:
    """logits[..., v] = sum_d h[..., d] W[v, d] in float64.

    hidden_bits [..., D] and weight_bits [V, D] are bfloat16 bit patterns.
    Every product of two bfloat16 values is exact in float64 (8 + 8
    significant bits), and the float64 sum over D terms is within D 2^-53 of
    the exact dot product, far below the float32 accumulation the GPU does.
    The matrix product is the library's; no blocking or reordering here.
    """
    h = bf16_bits_to_f64(hidden_bits)
    w = bf16_bits_to_f64(weight_bits)
    if h.shape[-1] != w.shape[1]:
        raise ValueError("hidden [..., D] and weight [V, D] disagree on D")
    return h @ w.T


def verify_lmhead(hidden_t, weight_t, hidden_d, weight_d, tokens, temperature: float, seed: int,
                  mode: int = SAMPLE, seq_range=None, threads: int = 1) -> dict:
    """``verify`` on the logits the two LM heads produce: target logits
    hidden_t [B, K+1, Dt] x weight_t [V, Dt]^T, draft logits hidden_d [B, K, Dd]
    x weight_d [V, Dd]^T (None in greedy mode), all bfloat16 bit patterns.
    ``seq_range=(b0, b1)`` computes the logits of those sequences only (the
    other rows stay zero pages that are never touched) and verifies them; the
    other sequences' outputs keep their fill values."""
    hidden_t = np.ascontiguousarray(hidden_t, dtype=np.uint16)
    B, K1, _ = hidden_t.shape
    K = K1 - 1
    V = weight_t.shape[0]
    b0, b1 = (0, B) if seq_range is None else seq_range
    lt = np.zeros((B, K1, V), dtype=np.float64)
    lt[b0:b1] = lm_head_logits(hidden_t[b0:b1], weight_t)
    ld = None
    if mode == SAMPLE and hidden_d is not None:
        hidden_d = np.ascontiguousarray(hidden_d, dtype=np.uint16)
        ld = np.zeros((B, K, V), dtype=np.float64)
        ld[b0:b1] = lm_head_logits(hidden_d[b0:b1], weight_d)
    return verify(lt, ld, tokens, temperature, seed, mode, threads=threads, seq_range=(b0, b1))
