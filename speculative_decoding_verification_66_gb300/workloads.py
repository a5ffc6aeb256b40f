"""Seeded synthetic inputs for speculative-decoding verification.

This module only draws inputs. It holds none of the verification arithmetic
(no acceptance ratio, residual or sampling rule), so that both the CUDA path
and the CPU oracle can be fed from it without sharing any of the method.

The pages' own workload (a TinyLlama draft and a Llama-2-7B target on 50-100
token prompts) needs trained weights and prompts that are not available. The
five workloads below stand in for it. Their logits are synthetic, with the
shapes and value distributions listed in ``WORKLOADS``. Each draft row is a
noisy copy of its target row. Draft tokens are drawn from the draft's own
temperature-scaled softmax, as a draft model would draw them. Greedy drafts
are the argmax of a noisy copy.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    V: int
    dtype: str          # "f32" or "bf16": logits storage type
    mode: str           # "sample" or "greedy"
    temperature: float
    target_std: float
    spike: float        # added at one uniformly drawn index of every target row (0 = none)
    draft_scale: float  # draft = draft_scale * target + N(0, draft_noise^2)
    draft_noise: float

    @property
    def label(self) -> str:
        t = f" T={self.temperature:g}" if self.mode == "sample" else ""
        return f"B={self.B} K={self.K} V={self.V} {self.dtype} {self.mode}{t}"

    def resized(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # B=8, K=4, V=32000 fp32: target ~ N(0, 2^2); draft = target + N(0, 0.5^2); T = 1.
    "small_f32": Workload("small_f32", 8, 4, 32000, "f32", "sample", 1.0, 2.0, 0.0, 1.0, 0.5),
    # B=64, K=4, V=32000 bf16: target ~ N(0, 3^2) + 8 at one index per row; draft = target + N(0, 1).
    "spiky_bf16": Workload("spiky_bf16", 64, 4, 32000, "bf16", "sample", 1.0, 3.0, 8.0, 1.0, 1.0),
    # B=256, K=8, V=128256 bf16, T = 0.7 on both: target ~ N(0, 2.5^2); draft = 0.8 target + N(0, 1).
    "llama3_bf16": Workload("llama3_bf16", 256, 8, 128256, "bf16", "sample", 0.7, 2.5, 0.0, 0.8, 1.0),
    # B=32, K=16, V=152064 bf16: target ~ N(0, 2^2); draft = target + N(0, 0.3^2) (long accepted runs).
    "qwen_long_bf16": Workload("qwen_long_bf16", 32, 16, 152064, "bf16", "sample", 1.0, 2.0, 0.0,
                               1.0, 0.3),
    # B=512, K=4, V=128256 bf16 greedy: target ~ N(0, 2^2); drafts = argmax(target + N(0, 1.5^2)).
    "greedy_bf16": Workload("greedy_bf16", 512, 4, 128256, "bf16", "greedy", 1.0, 2.0, 0.0, 1.0, 1.5),
}

# The workload whose throughput is the headline figure.
HEADLINE = "llama3_bf16"


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_inputs(wl: Workload, seed: int, device="cpu", top_k: int = 0, top_p: float = 1.0) -> dict:
    """Draw one batch for ``wl``.

    Returns dict(target [B, K+1, V], draft [B, K, V] or None, tokens [B, K] int32),
    all on ``device``. Noise is drawn in float32 from a generator seeded with
    ``seed`` on ``device``, then stored in the workload's dtype. Draft tokens are
    drawn from the *stored* draft logits, so they follow the draft distribution
    the verifier sees; with ``top_k`` / ``top_p`` (0 / 1.0: no cut) from that
    distribution cut the same way.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    B, K, V = wl.B, wl.K, wl.V
    dt = torch_dtype(wl.dtype)
    tgt = torch.randn((B, K + 1, V), generator=g, device=dev, dtype=torch.float32)
    tgt.mul_(wl.target_std)
    if wl.spike != 0.0 and B * (K + 1) > 0:
        idx = torch.randint(0, V, (B, K + 1, 1), generator=g, device=dev)
        tgt.scatter_add_(2, idx, torch.full((B, K + 1, 1), wl.spike, device=dev))
    target = tgt.to(dt)
    if wl.mode == "greedy":
        noisy = tgt[:, :K] + wl.draft_noise * torch.randn((B, K, V), generator=g, device=dev)
        tokens = noisy.argmax(dim=-1).to(torch.int32) if K > 0 else torch.zeros(
            (B, 0), dtype=torch.int32, device=dev)
        del tgt, noisy
        return {"target": target, "draft": None, "tokens": tokens.contiguous()}
    drf = tgt[:, :K] * wl.draft_scale
    drf.add_(wl.draft_noise * torch.randn((B, K, V), generator=g, device=dev))
    draft = drf.to(dt)
    del tgt, drf
    tokens = draw_from_logits(draft, wl.temperature, g, top_k, top_p)
    return {"target": target, "draft": draft, "tokens": tokens}


def _draft_sampler_probs(x: torch.Tensor, temperature: float, top_k: int, top_p: float):
    """The draft model's own sampling distribution over rows x [n, V] (float32):
    softmax(x / T), cut to the top_k largest logits and then to the smallest
    upper set of logit values holding top_p of the rest, as a serving stack's
    sampler does before it draws. Input generation only."""
    probs = torch.softmax(x / temperature, dim=-1)
    V = x.shape[-1]
    if 0 < top_k < V:
        kth = torch.topk(x, top_k, dim=-1).values[:, -1:]
        probs = probs * (x >= kth)
    if top_p < 1.0:
        xs, order = torch.sort(x, dim=-1, descending=True)
        ps = torch.gather(probs, -1, order)
        csum = torch.cumsum(ps, dim=-1)
        need = top_p * csum[:, -1:]
        first = torch.searchsorted(csum.contiguous(), need.contiguous()).clamp_(max=V - 1)
        thr = torch.gather(xs, -1, first)
        probs = probs * (x >= thr)
    return probs / probs.sum(dim=-1, keepdim=True)


def draw_from_logits(logits: torch.Tensor, temperature: float, g: torch.Generator,
                     top_k: int = 0, top_p: float = 1.0) -> torch.Tensor:
    """One token per row from softmax(logits / T) (optionally top-k / top-p cut):
    what a draft model's sampler does."""
    B, K, V = logits.shape
    if B * K == 0:
        return torch.zeros((B, K), dtype=torch.int32, device=logits.device)
    out = torch.empty((B * K,), dtype=torch.int64, device=logits.device)
    flat = logits.reshape(B * K, V)
    step = max(1, (1 << 28) // max(V, 1))
    if top_k > 0 or top_p < 1.0:
        step = max(1, step // 4)
    for s in range(0, B * K, step):
        probs = _draft_sampler_probs(flat[s:s + step].float(), temperature, top_k, top_p)
        out[s:s + step] = torch.multinomial(probs, 1, generator=g).squeeze(1)
    return out.view(B, K).to(torch.int32)


def bf16_bits(t: torch.Tensor):
    """Host numpy view of a bfloat16 tensor's raw 16-bit patterns (uint16)."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_host_arrays(inputs: dict):
    """(target, draft, tokens) as numpy arrays in the layout the oracle reads."""
    import numpy as np

    def conv(t):
        if t is None:
            return None
        if t.dtype == torch.bfloat16:
            return bf16_bits(t)
        return t.detach().cpu().contiguous().numpy().astype(np.float32, copy=False)

    return conv(inputs["target"]), conv(inputs["draft"]), \
        inputs["tokens"].detach().cpu().numpy().astype(np.int32)


@dataclasses.dataclass(frozen=True)
class LmWorkload:
    """Hidden states and output matrices for verification from the models'
    last layer (the LM head computes the logits). Synthetic: no trained
    weights exist here. Target: h ~ N(0, 1) per coordinate, W ~ N(0,
    target_std^2 / d_target), so every target logit is ~ N(0, target_std^2).
    Draft: the first m = min(d_draft, d_target) coordinates of the target's
    hidden state plus N(0, draft_noise^2), and the first m columns of W scaled
    by sqrt(d_target / m), so a draft logit has about the same spread and a
    correlation of about sqrt(m / d_target) with the target's (a wider draft
    gets fresh coordinates with small weights)."""
    name: str
    B: int
    K: int
    V: int
    d_target: int
    d_draft: int
    mode: str
    temperature: float
    target_std: float
    draft_noise: float

    @property
    def label(self) -> str:
        t = f" T={self.temperature:g}" if self.mode == "sample" else ""
        return (f"B={self.B} K={self.K} V={self.V} D={self.d_target}/{self.d_draft} "
                f"{self.mode}{t}")

    def resized(self, **kw) -> "LmWorkload":
        return dataclasses.replace(self, **kw)


LM_WORKLOADS = {
    # Small: several row blocks, vocabulary tiles and k-blocks, ragged at every edge.
    "lm_small": LmWorkload("lm_small", 64, 4, 1000, 200, 136, "sample", 1.0, 2.0, 0.3),
    # Llama-3-8B target (hidden 4096) with a Llama-3.2-1B-sized draft (hidden
    # 2048), vocabulary 128256, B=256, K=8, T=0.7.
    "lm_llama3_bf16": LmWorkload("lm_llama3_bf16", 256, 8, 128256, 4096, 2048, "sample", 0.7,
                                 2.5, 0.3),
    # Greedy on the same target head.
    "lm_greedy_bf16": LmWorkload("lm_greedy_bf16", 256, 8, 128256, 4096, 2048, "greedy", 1.0,
                                 2.5, 0.3),
}


def make_lmhead_inputs(lw: LmWorkload, seed: int, device="cpu") -> dict:
    """One batch for ``lw``: hidden_t [B, K+1, Dt], weight_t [V, Dt], hidden_d
    [B, K, Dd], weight_d [V, Dd] (bfloat16; the draft pair None in greedy mode)
    and tokens [B, K] int32. Draft tokens are drawn from the draft head's own
    softmax at the workload's temperature (greedy: the argmax of a noisy copy
    of the target logits), computed here in float32 from the stored bfloat16
    operands. Input generation only."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    B, K, V, Dt, Dd = lw.B, lw.K, lw.V, lw.d_target, lw.d_draft
    ht = torch.randn((B, K + 1, Dt), generator=g, device=dev).to(torch.bfloat16)
    wt = (torch.randn((V, Dt), generator=g, device=dev) * (lw.target_std / Dt ** 0.5)).to(
        torch.bfloat16)
    if lw.mode == "greedy":
        tokens = torch.zeros((B, K), dtype=torch.int32, device=dev)
        wtf = wt.float()
        step = max(1, (1 << 26) // max(V * max(K, 1), 1))
        for s in range(0, B if K > 0 else 0, step):
            e = min(B, s + step)
            lg = ht[s:e, :K].float() @ wtf.T
            lg += lw.draft_noise * lw.target_std * torch.randn(lg.shape, generator=g, device=dev)
            tokens[s:e] = lg.argmax(dim=-1).to(torch.int32)
        return {"hidden_t": ht.contiguous(), "weight_t": wt.contiguous(), "hidden_d": None,
                "weight_d": None, "tokens": tokens}
    m = min(Dd, Dt)
    hd = lw.draft_noise * torch.randn((B, K, Dd), generator=g, device=dev)
    hd[..., :m] += ht[:, :K, :m].float()
    if Dd > m:  # a wider draft: its extra coordinates are fresh N(0, 1)
        hd[..., m:] = torch.randn((B, K, Dd - m), generator=g, device=dev)
    hd = hd.to(torch.bfloat16).contiguous()
    wd = torch.empty((V, Dd), device=dev)
    wd[:, :m] = wt[:, :m].float() * (Dt / m) ** 0.5
    if Dd > m:  # small weights on the extra coordinates
        wd[:, m:] = torch.randn((V, Dd - m), generator=g, device=dev) * (
            0.3 * lw.target_std / Dd ** 0.5)
    wd = wd.to(torch.bfloat16).contiguous()
    tokens = torch.zeros((B, K), dtype=torch.int32, device=dev)
    step = max(1, (1 << 26) // max(V * max(K, 1), 1))
    wdf = wd.float()
    for s in range(0, B, step):
        e = min(B, s + step)
        if K == 0:
            break
        lg = (hd[s:e].float() @ wdf.T).contiguous()
        tokens[s:e] = draw_from_logits(lg, lw.temperature, g)
    return {"hidden_t": ht.contiguous(), "weight_t": wt.contiguous(), "hidden_d": hd,
            "weight_d": wd, "tokens": tokens}


def lm_host_arrays(inputs: dict):
    """(hidden_t, weight_t, hidden_d, weight_d, tokens) as the oracle reads
    them: bfloat16 bit patterns (uint16) and int32."""
    def conv(t):
        return None if t is None else bf16_bits(t)

    return (conv(inputs["hidden_t"]), conv(inputs["weight_t"]), conv(inputs["hidden_d"]),
            conv(inputs["weight_d"]), inputs["tokens"].detach().cpu().numpy().astype("int32"))
