"""Seeded synthetic workloads for the SimSD single-forward verification step.

This module only draws random inputs: shapes, sizes and value distributions of the
five workloads below. It holds none of the verification arithmetic (no RoPE, no
mask, no attention, no acceptance test), so that the CUDA path and the CPU oracle
can both consume exactly the same tensors without sharing any of the method's code.

Distributions follow the workload statements: ``N(0, s2)`` is read as mean 0 and
*variance* s2 (so logits ``N(0, 4)`` have standard deviation 2). The cached prompt
keys are drawn directly as N(0, 1): a rotation of an isotropic Gaussian vector is
again isotropic Gaussian, so these are distributed exactly like RoPE-rotated keys
and need no rotation here. Draft tokens are drawn from the draft distribution
(the drafter's own sampling step, which precedes verification).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "fp32" or "bf16" for Q/K/V and the attention output
    batch: int
    Hq: int
    Hkv: int
    D: int
    B: int                # block size: the response span D_1..D_B
    prompt_len: Optional[int]      # fixed prompt length P, or None for ragged
    prompt_len_range: Optional[tuple] = None   # inclusive (lo, hi) for ragged
    rope_theta: float = 1e6
    gamma: int = 4
    V: int = 151936
    logit_std: float = 2.0
    draft_noise_std: float = math.sqrt(0.5)
    temperature: float = 1.0
    identity_tau_frac: float = 0.0   # share of requests whose step labels are 1..B in order
    logit_dtype: str = "fp32"        # "fp32" or "bf16" target / draft logits
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the verification step (one attention layer + acceptance).
WORKLOADS: Dict[str, Workload] = {
    "tiny_fp32": Workload(
        name="tiny_fp32", dtype="fp32", batch=1, Hq=4, Hkv=1, D=64, B=4,
        prompt_len=32, rope_theta=1e4, gamma=4, V=1000,
        logit_std=math.sqrt(2.0), draft_noise_std=math.sqrt(0.5)),
    "gqa8b_bf16": Workload(
        name="gqa8b_bf16", dtype="bf16", batch=16, Hq=32, Hkv=8, D=128, B=4,
        prompt_len=512, rope_theta=1e6, gamma=4, V=151936,
        logit_std=2.0, draft_noise_std=math.sqrt(0.5)),
    "large_block_bf16": Workload(
        name="large_block_bf16", dtype="bf16", batch=32, Hq=32, Hkv=8, D=128, B=32,
        prompt_len=4096, rope_theta=1e6, gamma=32, V=151936,
        logit_std=2.0, draft_noise_std=1.0),
    "long_context_bf16": Workload(
        name="long_context_bf16", dtype="bf16", batch=8, Hq=32, Hkv=8, D=128, B=16,
        prompt_len=32768, rope_theta=1e6, gamma=16, V=151936,
        logit_std=2.0, draft_noise_std=math.sqrt(0.5)),
    "ragged_bf16": Workload(
        name="ragged_bf16", dtype="bf16", batch=256, Hq=32, Hkv=8, D=128, B=8,
        prompt_len=None, prompt_len_range=(128, 8192), rope_theta=1e6, gamma=8,
        V=151936, logit_std=2.0, draft_noise_std=math.sqrt(0.5),
        identity_tau_frac=0.2),
}
WORKLOAD_ORDER = ["tiny_fp32", "gqa8b_bf16", "large_block_bf16",
                  "long_context_bf16", "ragged_bf16"]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_layout_inputs(w: Workload, seed: Optional[int] = None, device="cpu"):
    """Step labels tau [b, B] (int32, a permutation of 1..B per request) and prompt
    lengths [b] (int32)."""
    seed = w.seed if seed is None else seed
    g = _gen(seed, "cpu")          # small; drawn on the CPU so every device agrees
    b, B = w.batch, w.B
    if w.prompt_len is not None:
        plen = torch.full((b,), w.prompt_len, dtype=torch.int32)
    else:
        lo, hi = w.prompt_len_range
        plen = torch.randint(lo, hi + 1, (b,), generator=g, dtype=torch.int64).to(torch.int32)
    tau = torch.stack([torch.randperm(B, generator=g) + 1 for _ in range(b)]).to(torch.int32)
    n_id = int(round(w.identity_tau_frac * b))
    if n_id > 0:
        chosen = torch.randperm(b, generator=g)[:n_id]
        tau[chosen] = torch.arange(1, B + 1, dtype=torch.int32)
    return {"tau": tau.to(device), "prompt_len": plen.to(device)}


def make_attention_inputs(w: Workload, prompt_len: torch.Tensor, seed: Optional[int] = None,
                          device="cpu", cache_layout: str = "NHD"):
    """Q / response K,V / cached prompt K,V for one attention layer.

    q       [b, 2B, Hq, D]   rows 0..B-1 are the data slots D_k, B..2B-1 the mask slots
    k_resp  [b, 2B, Hkv, D]  (pre-RoPE, like q)
    v_resp  [b, 2B, Hkv, D]
    k_cache, v_cache         packed over requests: NHD = [sum P, Hkv, D],
                             HND = [Hkv, sum P, D]; keys already rotated
    cache_offsets [b+1] int64 (token offsets of each request inside the packed cache)
    """
    seed = w.seed if seed is None else seed
    g = _gen(seed + 1, device)
    b, B, Hq, Hkv, D = w.batch, w.B, w.Hq, w.Hkv, w.D
    dt = w.torch_dtype
    plen = prompt_len.to("cpu").to(torch.int64)
    offs = torch.zeros(b + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(plen, 0)
    total = int(offs[-1])

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dt)

    q = randn(b, 2 * B, Hq, D)
    k_resp = randn(b, 2 * B, Hkv, D)
    v_resp = randn(b, 2 * B, Hkv, D)
    if cache_layout == "NHD":
        k_cache = randn(total, Hkv, D)
        v_cache = randn(total, Hkv, D)
    elif cache_layout == "HND":
        k_cache = randn(Hkv, total, D)
        v_cache = randn(Hkv, total, D)
    else:
        raise ValueError(cache_layout)
    return {"q": q, "k_resp": k_resp, "v_resp": v_resp, "k_cache": k_cache,
            "v_cache": v_cache, "cache_offsets": offs.to(device),
            "cache_layout": cache_layout}


def make_accept_inputs(w: Workload, seed: Optional[int] = None, device="cpu",
                       V: Optional[int] = None):
    """Target / draft logits [b, B, V] (indexed by block slot k) in `w.logit_dtype` (bf16:
    the fp32 draws rounded to nearest), draft tokens [b, B] int32 drawn from the draft
    distribution of those logits at temperature T (its argmax at T = 0), and a Philox
    (seed, offset) pair for the acceptance uniforms."""
    seed = w.seed if seed is None else seed
    V = w.V if V is None else V
    g = _gen(seed + 2, device)
    b, B = w.batch, w.B
    target = torch.randn(b, B, V, generator=g, device=device) * w.logit_std
    draft = target + torch.randn(b, B, V, generator=g, device=device) * w.draft_noise_std
    if w.logit_dtype == "bf16":
        target, draft = target.to(torch.bfloat16), draft.to(torch.bfloat16)
    elif w.logit_dtype != "fp32":
        raise ValueError(w.logit_dtype)
    if w.temperature == 0:   # a greedy drafter proposes its own first maximum
        tokens = torch.argmax(draft, dim=-1).to(torch.int32)
    else:
        probs = torch.softmax(draft.float().reshape(b * B, V) / w.temperature, dim=-1)
        tokens = torch.multinomial(probs, 1, generator=g).reshape(b, B).to(torch.int32)
        del probs
    return {"target_logits": target, "draft_logits": draft, "draft_tokens": tokens,
            "philox_seed": 0x5EED0000 + int(seed), "philox_offset": 0}


def algorithmic_bytes(w: Workload, prompt_len: torch.Tensor, target_only: bool = False,
                      with_khat: bool = False) -> dict:
    """Minimum HBM bytes of one verification step: each input read once, each
    output written once (per request: the prompt K/V, the 2B-row Q/K/V/O, and the
    target+draft logit rows of the gamma verified slots; the target rows only at
    temperature 0, where greedy verification reads no draft logits, or with `target_only`
    for coupled-noise verification). `khat_bytes` is the expected-prefix estimate's read of
    the gamma draft rows, added to the total with `with_khat`."""
    esz = 4 if w.dtype == "fp32" else 2
    P_sum = int(prompt_len.to(torch.int64).sum())
    b, B, D = w.batch, w.B, w.D
    kv_prompt = 2 * P_sum * w.Hkv * D * esz
    resp = b * 2 * B * D * esz * (2 * w.Hq + 2 * w.Hkv)   # q + out, k + v
    lsz = 2 if w.logit_dtype == "bf16" else 4
    accept = b * w.gamma * (1 if (w.temperature == 0 or target_only) else 2) * w.V * lsz
    flops = 0
    for P in prompt_len.tolist():
        flops += 4 * 2 * B * w.Hq * (P + B) * D
    khat = b * w.gamma * w.V * lsz
    return {"attn_bytes": kv_prompt + resp, "accept_bytes": accept, "khat_bytes": khat,
            "total_bytes": kv_prompt + resp + accept + (khat if with_khat else 0),
            "attn_flops": flops, "tokens": b * w.gamma}
