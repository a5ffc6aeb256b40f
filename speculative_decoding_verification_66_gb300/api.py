"""Python binding of the spec_verify C ABI: the same names, torch tensors in.

Argument marshalling only. Every step of the verification runs in the CUDA
kernels of libspecverify.so; this module turns tensors into pointers and
sizes, picks the current CUDA stream, and keeps a workspace buffer per device
and stream so that repeated calls do not allocate.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _lib

SV_F32, SV_BF16 = 0, 1
SV_SAMPLE, SV_GREEDY = 0, 1
SV_SEQ_BAD_TOKEN, SV_SEQ_NONFINITE, SV_SEQ_TIMEOUT, SV_SEQ_INDEX = 1, 2, 4, 8


def sv_device_checks() -> bool:
    """True when the loaded library is the variant built with device-side
    index checks (see _build.build(debug=True) and the SV_LIBRARY variable)."""
    return bool(_lib.load().sv_device_checks())

def launches(mode, V: int, dtype) -> int:
    """Kernel launches one spec_verify call makes: row statistics and the scan,
    and in sampling mode the sampler. V and dtype do not change the count."""
    return 2 if mode_code(mode) == SV_GREEDY else 4


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = _lib.load().sv_error_string(code).decode()
        super().__init__(f"{where}: {msg} (code {code})")
        self.code = code


def _check(code: int, where: str):
    if code != 0:
        raise SpecVerifyError(code, where)


def dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SV_F32
    if t == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t}")


def mode_code(mode) -> int:
    if isinstance(mode, str):
        return {"sample": SV_SAMPLE, "greedy": SV_GREEDY}[mode]
    return int(mode)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def sv_workspace_bytes(B: int, K: int, V: int, dtype, mode) -> int:
    n = ctypes.c_size_t(0)
    d = dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    _check(_lib.load().sv_workspace_bytes(B, K, V, d, mode_code(mode), ctypes.byref(n)),
           "sv_workspace_bytes")
    return int(n.value)


def sv_host_staging_bytes(B: int, K: int, V: int, dtype, mode) -> int:
    n = ctypes.c_size_t(0)
    d = dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    _check(_lib.load().sv_host_staging_bytes(B, K, V, d, mode_code(mode), ctypes.byref(n)),
           "sv_host_staging_bytes")
    return int(n.value)


_ws_lock = threading.Lock()
_ws_cache: dict = {}


def workspace_for(device: torch.device, stream: torch.cuda.Stream, nbytes: int) -> torch.Tensor:
    """A reusable workspace of at least nbytes for (device, stream)."""
    key = (device.index, stream.cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
    return ws


def _shapes(target_logits, draft_logits, draft_tokens, mode):
    if target_logits.dim() != 3 or not target_logits.is_cuda:
        raise ValueError("target_logits must be a CUDA tensor [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    if K < 0:
        raise ValueError("target_logits needs K+1 >= 1 rows per sequence")
    if not target_logits.is_contiguous():
        raise ValueError("target_logits must be contiguous")
    if mode == SV_SAMPLE and K > 0:
        if draft_logits is None or tuple(draft_logits.shape) != (B, K, V):
            raise ValueError("draft_logits must be [B, K, V] in sampling mode")
        if draft_logits.dtype != target_logits.dtype or not draft_logits.is_contiguous():
            raise ValueError("draft_logits must be contiguous with target_logits' dtype")
        if draft_logits.device != target_logits.device:
            raise ValueError("draft_logits must be on target_logits' device")
    if K > 0:
        if draft_tokens is None or tuple(draft_tokens.shape) != (B, K):
            raise ValueError("draft_tokens must be [B, K]")
        if draft_tokens.dtype != torch.int32 or not draft_tokens.is_contiguous():
            raise ValueError("draft_tokens must be contiguous int32")
        if draft_tokens.device != target_logits.device:
            raise ValueError("draft_tokens must be on target_logits' device")
    return B, K, V


def _prepare(target_logits, draft_logits, draft_tokens, mode, out_tokens, num_accepted,
             workspace, stream):
    m = mode_code(mode)
    B, K, V = _shapes(target_logits, draft_logits, draft_tokens, m)
    dev = target_logits.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    d = dtype_code(target_logits.dtype)
    need = sv_workspace_bytes(B, K, V, d, m)
    if workspace is None:
        workspace = workspace_for(dev, stream, need)
    return m, B, K, V, d, stream, out_tokens, num_accepted, workspace


def spec_verify(target_logits, draft_logits, draft_tokens, temperature: float = 1.0,
                seed: int = 0, mode="sample", *, out_tokens=None, num_accepted=None,
                workspace=None, stream=None):
    """Verify B sequences of K drafts. Returns (out_tokens [B, K+1], num_accepted [B]).

    Asynchronous on ``stream`` (default: the current stream of the logits' device).
    """
    m, B, K, V, d, stream, out_tokens, num_accepted, workspace = _prepare(
        target_logits, draft_logits, draft_tokens, mode, out_tokens, num_accepted, workspace,
        stream)
    with torch.cuda.device(target_logits.device):
        _check(_lib.load().spec_verify(
            _ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, d, float(temperature),
            int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream)), "spec_verify")
    return out_tokens, num_accepted


def sv_early_exit_workspace_bytes(B: int, K: int, V: int, dtype, mode) -> int:
    n = ctypes.c_size_t(0)
    d = dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    _check(_lib.load().sv_early_exit_workspace_bytes(B, K, V, d, mode_code(mode), ctypes.byref(n)),
           "sv_early_exit_workspace_bytes")
    return int(n.value)


def spec_verify_early_exit(target_logits, draft_logits, draft_tokens, temperature: float = 1.0,
                           seed: int = 0, mode="sample", *, out_tokens=None, num_accepted=None,
                           workspace=None, stream=None):
    """spec_verify that reads a sequence's rows only up to its first rejection
    (phases of 1, 2, 4, ... positions). Same results as spec_verify except
    that non-finite values in rows after the emitted position go unnoticed."""
    m = mode_code(mode)
    B, K, V = _shapes(target_logits, draft_logits, draft_tokens, m)
    dev = target_logits.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    d = dtype_code(target_logits.dtype)
    if workspace is None:
        workspace = workspace_for(dev, stream, sv_early_exit_workspace_bytes(B, K, V, d, m))
    with torch.cuda.device(dev):
        _check(_lib.load().spec_verify_early_exit(
            _ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, d, float(temperature),
            int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream)),
            "spec_verify_early_exit")
    return out_tokens, num_accepted


def sv_sharded_workspace_bytes(B: int, K: int, Vs: int, G: int, dtype, mode) -> int:
    n = ctypes.c_size_t(0)
    d = dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    _check(_lib.load().sv_sharded_workspace_bytes(B, K, Vs, G, d, mode_code(mode),
                                                  ctypes.byref(n)), "sv_sharded_workspace_bytes")
    return int(n.value)


def spec_verify_sharded(target_shards, draft_shards, draft_tokens, temperature: float = 1.0,
                        seed: int = 0, mode="sample", *, out_tokens=None, num_accepted=None,
                        workspace=None, stream=None):
    """spec_verify on logits split over the vocabulary: target_shards is a list
    of G contiguous [B, K+1, Vs] tensors (shard g = columns [g Vs, (g+1) Vs)),
    draft_shards G [B, K, Vs] tensors (None in greedy mode). Token ids are
    global (0 .. G Vs - 1)."""
    m = mode_code(mode)
    G = len(target_shards)
    if G < 1:
        raise ValueError("need at least one shard")
    t0 = target_shards[0]
    if t0.dim() != 3 or not t0.is_cuda:
        raise ValueError("target shards must be CUDA tensors [B, K+1, Vs]")
    B, K1, Vs = t0.shape
    K = K1 - 1
    for t in target_shards:
        if tuple(t.shape) != (B, K1, Vs) or t.dtype != t0.dtype or not t.is_contiguous() \
                or t.device != t0.device:
            raise ValueError("target shards must share shape, dtype and device, contiguous")
    sampling = m == SV_SAMPLE and K > 0
    if sampling:
        if draft_shards is None or len(draft_shards) != G:
            raise ValueError("draft_shards must hold G tensors in sampling mode")
        for d in draft_shards:
            if tuple(d.shape) != (B, K, Vs) or d.dtype != t0.dtype or not d.is_contiguous() \
                    or d.device != t0.device:
                raise ValueError("draft shards must be contiguous [B, K, Vs] like the targets")
    if K > 0:
        if draft_tokens is None or tuple(draft_tokens.shape) != (B, K) \
                or draft_tokens.dtype != torch.int32 or not draft_tokens.is_contiguous():
            raise ValueError("draft_tokens must be contiguous int32 [B, K]")
    dev = t0.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    d = dtype_code(t0.dtype)
    if workspace is None:
        workspace = workspace_for(dev, stream, sv_sharded_workspace_bytes(B, K, Vs, G, d, m))
    tp = (ctypes.c_void_p * G)(*[t.data_ptr() for t in target_shards])
    dp = (ctypes.c_void_p * G)(*[x.data_ptr() for x in draft_shards]) if sampling else None
    with torch.cuda.device(dev):
        _check(_lib.load().spec_verify_sharded(
            ctypes.cast(tp, ctypes.c_void_p), ctypes.cast(dp, ctypes.c_void_p) if dp else None, G,
            _ptr(draft_tokens if K > 0 else None), B, K, Vs, d, float(temperature),
            int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream)),
            "spec_verify_sharded")
    return out_tokens, num_accepted


def sv_filtered_workspace_bytes(B: int, K: int, V: int, dtype, mode) -> int:
    n = ctypes.c_size_t(0)
    d = dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype)
    _check(_lib.load().sv_filtered_workspace_bytes(B, K, V, d, mode_code(mode), ctypes.byref(n)),
           "sv_filtered_workspace_bytes")
    return int(n.value)


def spec_verify_filtered(target_logits, draft_logits, draft_tokens, temperature: float = 1.0,
                         top_k: int = 0, top_p: float = 1.0, seed: int = 0, mode="sample", *,
                         out_tokens=None, num_accepted=None, workspace=None, stream=None,
                         events=None):
    """spec_verify with top-k / top-p applied to both rows of every position
    (top_k = 0 and top_p = 1.0: off). ``events``: 4 torch.cuda.Event(enable_timing=True)
    recorded before the thresholds launch, after it, after the scan and after the
    sampler."""
    m = mode_code(mode)
    B, K, V = _shapes(target_logits, draft_logits, draft_tokens, m)
    dev = target_logits.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    d = dtype_code(target_logits.dtype)
    if workspace is None:
        workspace = workspace_for(dev, stream, sv_filtered_workspace_bytes(B, K, V, d, m))
    args = [_ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, d, float(temperature), int(top_k),
            float(top_p), int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream)]
    with torch.cuda.device(dev):
        if events is None:
            _check(_lib.load().spec_verify_filtered(*args), "spec_verify_filtered")
        else:
            for e in events:
                if not e.cuda_event:  # created lazily by torch on the first record
                    e.record(stream)
            handles = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
            _check(_lib.load().spec_verify_filtered_timed(*args, handles, len(events)),
                   "spec_verify_filtered_timed")
    return out_tokens, num_accepted


def spec_verify_filtered_debug(target_logits, draft_logits, draft_tokens,
                               temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                               seed: int = 0, mode="sample", *, workspace=None,
                               stream=None) -> dict:
    """spec_verify_filtered plus each row's kept-token normaliser and threshold."""
    m = mode_code(mode)
    B, K, V = _shapes(target_logits, draft_logits, draft_tokens, m)
    dev = target_logits.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    d = dtype_code(target_logits.dtype)
    if workspace is None:
        workspace = workspace_for(dev, stream, sv_filtered_workspace_bytes(B, K, V, d, m))
    out = {"out_tokens": torch.empty((B, K + 1), dtype=torch.int32, device=dev),
           "num_accepted": torch.empty((B,), dtype=torch.int32, device=dev),
           "lse_t": torch.full((B, K + 1), float("nan"), dtype=torch.float64, device=dev),
           "lse_d": torch.full((B, K), float("nan"), dtype=torch.float64, device=dev),
           "thr_t": torch.full((B, K + 1), float("nan"), dtype=torch.float32, device=dev),
           "thr_d": torch.full((B, K), float("nan"), dtype=torch.float32, device=dev),
           "seq_status": torch.full((B,), -7, dtype=torch.int32, device=dev)}
    with torch.cuda.device(dev):
        _check(_lib.load().spec_verify_filtered_debug(
            _ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, d, float(temperature), int(top_k),
            float(top_p), int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out["out_tokens"]),
            _ptr(out["num_accepted"]), _ptr(workspace), workspace.numel(),
            ctypes.c_void_p(stream.cuda_stream), _ptr(out["lse_t"]), _ptr(out["lse_d"]),
            _ptr(out["thr_t"]), _ptr(out["thr_d"]), _ptr(out["seq_status"])),
            "spec_verify_filtered_debug")
    return out


def spec_verify_filtered_timed(target_logits, draft_logits, draft_tokens, events,
                               temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                               seed: int = 0, mode="sample", **kw):
    """spec_verify_filtered with its 4 timing events (see there)."""
    return spec_verify_filtered(target_logits, draft_logits, draft_tokens, temperature, top_k,
                                top_p, seed, mode, events=events, **kw)


def spec_verify_debug(target_logits, draft_logits, draft_tokens, temperature: float = 1.0,
                      seed: int = 0, mode="sample", *, workspace=None, stream=None) -> dict:
    """spec_verify plus the normalisers, log-ratios and per-sequence status."""
    m, B, K, V, d, stream, out_tokens, num_accepted, workspace = _prepare(
        target_logits, draft_logits, draft_tokens, mode, None, None, workspace, stream)
    dev = target_logits.device
    lse_t = torch.full((B, K + 1), float("nan"), dtype=torch.float64, device=dev)
    lse_d = torch.full((B, K), float("nan"), dtype=torch.float64, device=dev)
    log_ratio = torch.full((B, K), float("nan"), dtype=torch.float64, device=dev)
    seq_status = torch.full((B,), -7, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.load().spec_verify_debug(
            _ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, d, float(temperature),
            int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream),
            _ptr(lse_t), _ptr(lse_d), _ptr(log_ratio), _ptr(seq_status)), "spec_verify_debug")
    return {"out_tokens": out_tokens, "num_accepted": num_accepted, "lse_t": lse_t,
            "lse_d": lse_d, "log_ratio": log_ratio, "seq_status": seq_status}


def spec_verify_timed(target_logits, draft_logits, draft_tokens, events, temperature: float = 1.0,
                      seed: int = 0, mode="sample", *, out_tokens=None, num_accepted=None,
                      workspace=None, stream=None):
    """spec_verify with ``events`` (4 torch.cuda.Event(enable_timing=True)) recorded
    on the launch stream before pass 1, after pass 1, after the scan and after the
    sampler."""
    m, B, K, V, d, stream, out_tokens, num_accepted, workspace = _prepare(
        target_logits, draft_logits, draft_tokens, mode, out_tokens, num_accepted, workspace,
        stream)
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event lazily, on its first record
            e.record(stream)
    handles = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    with torch.cuda.device(target_logits.device):
        _check(_lib.load().spec_verify_timed(
            _ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, d, float(temperature),
            int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream),
            handles, len(events)), "spec_verify_timed")
    return out_tokens, num_accepted


def spec_verify_host(target_logits, draft_logits, draft_tokens, temperature: float = 1.0,
                     seed: int = 0, mode="sample", *, out_tokens=None, num_accepted=None,
                     staging=None, device=None, stream=None, synchronize: bool = True):
    """End to end from host memory: CPU tensors in (pinned for asynchronous copies),
    CPU tensors out. The library copies inputs to ``staging`` on the device, verifies,
    and copies the results back, all on one stream."""
    m = mode_code(mode)
    if target_logits.dim() != 3 or target_logits.is_cuda:
        raise ValueError("target_logits must be a CPU tensor [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    d = dtype_code(target_logits.dtype)
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32).pin_memory()
    need = sv_host_staging_bytes(B, K, V, d, m)
    if staging is None:
        staging = workspace_for(dev, stream, need)
    for t in (target_logits, draft_logits, draft_tokens):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("host inputs must be contiguous CPU tensors")
    with torch.cuda.device(dev):
        _check(_lib.load().spec_verify_host(
            _ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, d, float(temperature),
            int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(staging), staging.numel(), ctypes.c_void_p(stream.cuda_stream)),
            "spec_verify_host")
    if synchronize:
        stream.synchronize()
    return out_tokens, num_accepted


def spec_verify_static(target_logits, draft_logits, draft_tokens, temperature: float = 1.0,
                       seed: int = 0, mode="sample", *, out_tokens=None, num_accepted=None,
                       stream=None):
    """spec_verify without a workspace, for callers that cannot allocate device
    memory: the library's fixed 8 MiB device scratch array is used instead. The
    output tensors are the caller's (allocated here only when not given). Calls
    that overlap on the GPU share that one array and race on it."""
    m = mode_code(mode)
    B, K, V = _shapes(target_logits, draft_logits, draft_tokens, m)
    dev = target_logits.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.load().spec_verify_static(
            _ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, dtype_code(target_logits.dtype),
            float(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens),
            _ptr(num_accepted), ctypes.c_void_p(stream.cuda_stream)), "spec_verify_static")
    return out_tokens, num_accepted


def sv_lmhead_workspace_bytes(B: int, K: int, V: int, d_target: int, d_draft: int,
                              mode) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.load().sv_lmhead_workspace_bytes(B, K, V, d_target, d_draft, mode_code(mode),
                                                 ctypes.byref(n)), "sv_lmhead_workspace_bytes")
    return n.value


def _lm_shapes(hidden_target, weight_target, hidden_draft, weight_draft, draft_tokens, m):
    for name, t in (("hidden_target", hidden_target), ("weight_target", weight_target)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    if hidden_target.dim() != 3 or weight_target.dim() != 2:
        raise ValueError("hidden_target must be [B, K+1, D] and weight_target [V, D]")
    B, K1, Dt = hidden_target.shape
    K = K1 - 1
    V = weight_target.shape[0]
    if weight_target.shape[1] != Dt:
        raise ValueError("weight_target must be [V, d_target]")
    Dd = Dt
    if m == SV_SAMPLE and K > 0:
        for name, t in (("hidden_draft", hidden_draft), ("weight_draft", weight_draft)):
            if t is None or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
        Dd = hidden_draft.shape[-1]
        if tuple(hidden_draft.shape) != (B, K, Dd) or tuple(weight_draft.shape) != (V, Dd):
            raise ValueError("hidden_draft must be [B, K, d_draft] and weight_draft [V, d_draft]")
    if K > 0 and (draft_tokens is None or tuple(draft_tokens.shape) != (B, K)
                  or draft_tokens.dtype != torch.int32 or not draft_tokens.is_contiguous()):
        raise ValueError("draft_tokens must be a contiguous [B, K] int32 tensor")
    return B, K, V, Dt, Dd


def spec_verify_lmhead(hidden_target, weight_target, hidden_draft, weight_draft, draft_tokens,
                       temperature: float = 1.0, seed: int = 0, mode="sample", *,
                       out_tokens=None, num_accepted=None, workspace=None, stream=None,
                       events=None, diagnostics=False):
    """Verification from the models' last hidden states: the LM head (h W^T)
    runs on the tensor cores with the row statistics folded in, so the logits
    are never written. ``events``: 5 torch.cuda.Event(enable_timing=True)
    (before the statistics GEMM, after it, after the scan, after the emitted
    pairs' GEMM, at the end). ``diagnostics=True`` returns a dict with the
    per-row normalisers, log-ratios and per-sequence status as well."""
    m = mode_code(mode)
    B, K, V, Dt, Dd = _lm_shapes(hidden_target, weight_target, hidden_draft, weight_draft,
                                 draft_tokens, m)
    dev = hidden_target.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = workspace_for(dev, stream, sv_lmhead_workspace_bytes(B, K, V, Dt, Dd, m))
    with_draft = m == SV_SAMPLE and K > 0
    args = [_ptr(hidden_target), _ptr(weight_target),
            _ptr(hidden_draft if with_draft else None), _ptr(weight_draft if with_draft else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, Dt, Dd, float(temperature),
            int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream)]
    L = _lib.load()
    with torch.cuda.device(dev):
        if diagnostics:
            out = {"out_tokens": out_tokens, "num_accepted": num_accepted,
                   "lse_t": torch.full((B, K + 1), float("nan"), dtype=torch.float64, device=dev),
                   "lse_d": torch.full((B, K), float("nan"), dtype=torch.float64, device=dev),
                   "log_ratio": torch.full((B, K), float("nan"), dtype=torch.float64,
                                           device=dev),
                   "seq_status": torch.full((B,), -7, dtype=torch.int32, device=dev)}
            _check(L.spec_verify_lmhead_debug(*args, _ptr(out["lse_t"]), _ptr(out["lse_d"]),
                                              _ptr(out["log_ratio"]), _ptr(out["seq_status"])),
                   "spec_verify_lmhead_debug")
            return out
        if events is None:
            _check(L.spec_verify_lmhead(*args), "spec_verify_lmhead")
        else:
            for e in events:
                if not e.cuda_event:  # created lazily by torch on the first record
                    e.record(stream)
            handles = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
            _check(L.spec_verify_lmhead_timed(*args, handles, len(events)),
                   "spec_verify_lmhead_timed")
    return out_tokens, num_accepted


def spec_verify_lmhead_debug(hidden_target, weight_target, hidden_draft, weight_draft,
                             draft_tokens, temperature: float = 1.0, seed: int = 0,
                             mode="sample", **kw) -> dict:
    """spec_verify_lmhead plus the per-row normalisers, log-ratios and status."""
    return spec_verify_lmhead(hidden_target, weight_target, hidden_draft, weight_draft,
                              draft_tokens, temperature, seed, mode, diagnostics=True, **kw)


def spec_verify_lmhead_timed(hidden_target, weight_target, hidden_draft, weight_draft,
                             draft_tokens, events, temperature: float = 1.0, seed: int = 0,
                             mode="sample", **kw):
    """spec_verify_lmhead with its 5 timing events (see there)."""
    return spec_verify_lmhead(hidden_target, weight_target, hidden_draft, weight_draft,
                              draft_tokens, temperature, seed, mode, events=events, **kw)


def spec_verify_gated(target_logits, draft_logits, draft_tokens, gate, temperature: float = 1.0,
                      seed: int = 0, mode="sample", *, stage: int = 1, top_k: int = 0,
                      top_p: float = 1.0, workspace=None, stream=None) -> dict:
    """Test hook for the timeout paths: spec_verify_filtered (spec_verify with
    the cuts off) with one stage's copies held until the device int32 ``gate``
    (one element) is nonzero: stage 1 = pass 1 (or the thresholds kernel),
    stage 2 = the sampler. Returns out_tokens, num_accepted and seq_status."""
    if gate.dtype != torch.int32 or not gate.is_cuda or gate.numel() < 1:
        raise ValueError("gate must be an int32 CUDA tensor")
    m = mode_code(mode)
    B, K, V = _shapes(target_logits, draft_logits, draft_tokens, m)
    dev = target_logits.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    d = dtype_code(target_logits.dtype)
    if workspace is None:
        workspace = workspace_for(dev, stream, sv_filtered_workspace_bytes(B, K, V, d, m))
    out = {"out_tokens": torch.empty((B, K + 1), dtype=torch.int32, device=dev),
           "num_accepted": torch.empty((B,), dtype=torch.int32, device=dev),
           "seq_status": torch.full((B,), -7, dtype=torch.int32, device=dev)}
    with torch.cuda.device(dev):
        _check(_lib.load().spec_verify_gated(
            _ptr(target_logits), _ptr(draft_logits if m == SV_SAMPLE else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, d, float(temperature), int(top_k),
            float(top_p), int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out["out_tokens"]),
            _ptr(out["num_accepted"]), _ptr(workspace), workspace.numel(),
            ctypes.c_void_p(stream.cuda_stream), _ptr(out["seq_status"]), int(stage), _ptr(gate)),
            "spec_verify_gated")
    return out


def spec_verify_lmhead_gated(hidden_target, weight_target, hidden_draft, weight_draft,
                             draft_tokens, gate, temperature: float = 1.0, seed: int = 0,
                             mode="sample", *, workspace=None, stream=None) -> dict:
    """Test hook for the timeout path: spec_verify_lmhead with the statistics
    GEMM's loads held until the device int32 ``gate`` (one element) is nonzero.
    Returns out_tokens, num_accepted and seq_status."""
    m = mode_code(mode)
    B, K, V, Dt, Dd = _lm_shapes(hidden_target, weight_target, hidden_draft, weight_draft,
                                 draft_tokens, m)
    if gate.dtype != torch.int32 or not gate.is_cuda or gate.numel() < 1:
        raise ValueError("gate must be an int32 CUDA tensor")
    dev = hidden_target.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = workspace_for(dev, stream, sv_lmhead_workspace_bytes(B, K, V, Dt, Dd, m))
    out = {"out_tokens": torch.empty((B, K + 1), dtype=torch.int32, device=dev),
           "num_accepted": torch.empty((B,), dtype=torch.int32, device=dev),
           "seq_status": torch.full((B,), -7, dtype=torch.int32, device=dev)}
    with_draft = m == SV_SAMPLE and K > 0
    with torch.cuda.device(dev):
        _check(_lib.load().spec_verify_lmhead_gated(
            _ptr(hidden_target), _ptr(weight_target),
            _ptr(hidden_draft if with_draft else None), _ptr(weight_draft if with_draft else None),
            _ptr(draft_tokens if K > 0 else None), B, K, V, Dt, Dd, float(temperature),
            int(seed) & 0xFFFFFFFFFFFFFFFF, m, _ptr(out["out_tokens"]), _ptr(out["num_accepted"]),
            _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream),
            _ptr(out["seq_status"]), _ptr(gate)), "spec_verify_lmhead_gated")
    return out


def sv_lmhead_logits(hidden, weight, out=None, err=None, stream=None) -> torch.Tensor:
    """The LM head alone: hidden [R, D] x weight [V, D]^T as float32 [R, V]
    (bfloat16 operands). ``err``: a device int32 tensor of one element that the
    kernel sets to 1 if a bounded wait runs out; checked here when given None."""
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise ValueError("hidden and weight must be bfloat16")
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden must be [R, D] and weight [V, D]")
    if not (hidden.is_cuda and weight.is_cuda and hidden.is_contiguous()
            and weight.is_contiguous()):
        raise ValueError("hidden and weight must be contiguous CUDA tensors")
    R, D = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    if out is None:
        out = torch.empty((R, V), dtype=torch.float32, device=dev)
    check = err is None
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        _check(_lib.load().sv_lmhead_logits(_ptr(hidden), _ptr(weight), R, D, V, _ptr(out),
                                            _ptr(err), ctypes.c_void_p(stream.cuda_stream)),
               "sv_lmhead_logits")
    if check and int(err.item()) != 0:
        raise RuntimeError("sv_lmhead_logits: a bounded wait inside the kernel ran out")
    return out


def sv_philox(seed: int, counters: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """The device Philox4x32-10 words of each counter: counters is an [n, 4]
    int32 CUDA tensor (the words' bit patterns), the result the same shape."""
    if counters.dim() != 2 or counters.shape[1] != 4 or counters.dtype != torch.int32:
        raise ValueError("counters must be an [n, 4] int32 tensor")
    if not counters.is_cuda or not counters.is_contiguous():
        raise ValueError("counters must be a contiguous CUDA tensor")
    dev = counters.device
    if out is None:
        out = torch.empty_like(counters)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        _check(_lib.load().sv_philox(int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(counters), _ptr(out),
                                     counters.shape[0], ctypes.c_void_p(stream.cuda_stream)),
               "sv_philox")
    return out


def version() -> int:
    return int(_lib.load().sv_version())
