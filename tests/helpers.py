"""Shared test helpers: build cases from the seeded workloads, run the CUDA path through
the C interface, run the oracle on the same inputs, and compare."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads

BF16_REL_L2 = 1e-2
BF16_MAX_ABS = 3e-2
FP32_TOL = 1e-5
BF16_LSE_ABS = 3e-2


def ensure_library():
    from diffusion_speculative_verify_gb300 import _build
    _build.build()


def make_case(w, seed=None, device="cuda", cache_layout="NHD", prompt_len=None, tau=None):
    lay = workloads.make_layout_inputs(w, seed=seed, device="cpu")
    if prompt_len is not None:
        lay["prompt_len"] = torch.as_tensor(prompt_len, dtype=torch.int32)
    if tau is not None:
        lay["tau"] = torch.as_tensor(tau, dtype=torch.int32)
    att = workloads.make_attention_inputs(w, lay["prompt_len"], seed=seed, device=device,
                                          cache_layout=cache_layout)
    acc = workloads.make_accept_inputs(w, seed=seed, device=device)
    inputs = {
        "tau": lay["tau"].to(device), "prompt_len": lay["prompt_len"].to(device),
        "q": att["q"], "k_resp": att["k_resp"], "v_resp": att["v_resp"],
        "k_cache": att["k_cache"], "v_cache": att["v_cache"],
        "cache_start": att["cache_offsets"][:-1].contiguous().to(device),
        "target_logits": acc["target_logits"], "draft_logits": acc["draft_logits"],
        "draft_tokens": acc["draft_tokens"],
    }
    meta = {"philox_seed": acc["philox_seed"], "philox_offset": acc["philox_offset"],
            "cache_layout": cache_layout}
    return inputs, meta


def to_np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def oracle_attention(inputs, pos_ids, labels, theta, cache_layout, requests=None,
                     kv_heads=None):
    """Oracle attention on the listed requests / kv heads; each request's cache rows are
    copied to the host on their own (full-size caches never leave the device)."""
    b, twoB, Hq, D = inputs["q"].shape
    Hkv = inputs["k_resp"].shape[2]
    out = np.zeros((b, twoB, Hq, D))
    lse = np.full((b, twoB, Hq), -np.inf)
    starts = inputs["cache_start"].cpu().numpy()
    plens = inputs["prompt_len"].cpu().numpy()
    for r in (range(b) if requests is None else requests):
        P = max(int(plens[r]), 0)
        s0 = int(starts[r])
        if cache_layout == "NHD":
            kc, vc = inputs["k_cache"][s0:s0 + P], inputs["v_cache"][s0:s0 + P]
        else:
            kc, vc = inputs["k_cache"][:, s0:s0 + P], inputs["v_cache"][:, s0:s0 + P]
        o, l = oracle.verify_attention(
            to_np(inputs["q"][r:r + 1]), to_np(inputs["k_resp"][r:r + 1]),
            to_np(inputs["v_resp"][r:r + 1]), to_np(kc), to_np(vc), np.array([0]),
            plens[r:r + 1], to_np(pos_ids[r:r + 1]), to_np(labels[r:r + 1]), theta,
            cache_layout=cache_layout, kv_heads=kv_heads)
        out[r], lse[r] = o[0], l[0]
    return out, lse


def oracle_accept(inputs, labels, gamma, temperature, seed, offset, requests=None):
    """Oracle acceptance on the listed requests, copying only their logit rows."""
    b = inputs["target_logits"].shape[0]
    reqs = list(range(b)) if requests is None else list(requests)
    idx = torch.tensor(reqs, device=inputs["target_logits"].device)
    res = oracle.accept(to_np(inputs["target_logits"][idx]), to_np(inputs["draft_logits"][idx]),
                        to_np(inputs["draft_tokens"][idx]), to_np(labels[idx.to(labels.device)]),
                        gamma, temperature, seed, offset, request_ids=reqs)
    full = {"accepted_len": np.full(b, -7, np.int32), "n_commit": np.full(b, -7, np.int32),
            "out_tokens": np.full((b, inputs["draft_tokens"].shape[1]), -7, np.int32),
            "out_pos": np.full((b, inputs["draft_tokens"].shape[1]), -7, np.int32),
            "err": res["err"], "diag": {}}
    for i, r in enumerate(reqs):
        for k in ("accepted_len", "n_commit", "out_tokens", "out_pos"):
            full[k][r] = res[k][i]
        if i in res["diag"]:
            full["diag"][r] = res["diag"][i]
    return full


def compare_attention(got, ref, dtype, rows_mask=None):
    """got, ref: [..., D] arrays over the compared rows. Returns (rel_l2, max_abs)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    diff = g - r
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(r), 1e-30))
    mx = float(np.abs(diff).max()) if diff.size else 0.0
    if dtype == torch.float32:
        assert rel <= FP32_TOL and mx <= FP32_TOL, (rel, mx)
    else:
        assert rel <= BF16_REL_L2 and mx <= BF16_MAX_ABS, (rel, mx)
    return rel, mx


def select_heads(out, G, heads):
    """Columns of the q-head axis belonging to the listed kv heads."""
    cols = [h * G + g for h in heads for g in range(G)]
    return out[..., cols, :] if out.ndim == 4 else out[..., cols]


def check_accept(res, got, requests, near_tie=1e-5):
    """Bit-exact comparison of accepted_len / n_commit / out_tokens / out_pos; a mismatch
    is tolerated only where the oracle's own decision margin (or race top-2 gap) is below
    `near_tie` relative. Returns the number of tolerated near-ties."""
    ties = 0
    for r in requests:
        same = (got["accepted_len"][r] == res["accepted_len"][r]
                and got["n_commit"][r] == res["n_commit"][r]
                and np.array_equal(got["out_tokens"][r], res["out_tokens"][r])
                and np.array_equal(got["out_pos"][r], res["out_pos"][r]))
        if same:
            continue
        d = res["diag"].get(r, {})
        margins = d.get("margins", [])
        race = d.get("race_top2")
        close = any(m < near_tie for m in margins)
        if race is not None and race[0] > 0:
            close |= (race[0] - race[1]) / race[0] < near_tie
        assert close, (r, got["accepted_len"][r], res["accepted_len"][r],
                       got["out_tokens"][r], res["out_tokens"][r], margins, race)
        ties += 1
    return ties
