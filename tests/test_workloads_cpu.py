"""CPU checks of the seeded input generators: the shapes, types and structure the workloads
state (no method arithmetic is exercised here)."""
import math

import torch

import workloads

W = workloads.WORKLOADS


def test_layout_inputs_are_permutations_with_the_stated_identity_share():
    w = W["ragged_bf16"]
    lay = workloads.make_layout_inputs(w)
    tau, plen = lay["tau"], lay["prompt_len"]
    assert tau.shape == (w.batch, w.B) and tau.dtype == torch.int32
    ident = torch.arange(1, w.B + 1, dtype=torch.int32)
    for r in range(w.batch):
        assert sorted(tau[r].tolist()) == list(range(1, w.B + 1))
    n_id = int((tau == ident).all(dim=1).sum())
    assert n_id >= round(w.identity_tau_frac * w.batch)        # random ones may also be identity
    lo, hi = w.prompt_len_range
    assert int(plen.min()) >= lo and int(plen.max()) <= hi
    again = workloads.make_layout_inputs(w)
    assert torch.equal(again["tau"], tau) and torch.equal(again["prompt_len"], plen)


def test_accept_inputs_types_tokens_and_temperature_zero():
    w = W["tiny_fp32"].with_(batch=6, B=4, gamma=4, V=257)
    acc = workloads.make_accept_inputs(w)
    assert acc["target_logits"].dtype == torch.float32 and acc["target_logits"].shape == (6, 4, 257)
    toks = acc["draft_tokens"]
    assert toks.dtype == torch.int32 and int(toks.min()) >= 0 and int(toks.max()) < 257
    wb = w.with_(logit_dtype="bf16")
    accb = workloads.make_accept_inputs(wb)
    assert accb["target_logits"].dtype == torch.bfloat16 and accb["draft_logits"].dtype == torch.bfloat16
    # bf16 logits are the fp32 draws rounded to nearest
    assert torch.equal(accb["target_logits"], acc["target_logits"].to(torch.bfloat16))
    w0 = w.with_(temperature=0.0)
    acc0 = workloads.make_accept_inputs(w0)
    assert torch.equal(acc0["draft_tokens"], torch.argmax(acc0["draft_logits"], -1).to(torch.int32))


def test_logit_spread_matches_the_stated_variance():
    w = W["gqa8b_bf16"].with_(batch=2, V=20000)
    acc = workloads.make_accept_inputs(w)
    t, d = acc["target_logits"].double(), acc["draft_logits"].double()
    assert abs(float(t.std()) - w.logit_std) < 0.05 * w.logit_std
    assert abs(float((d - t).std()) - w.draft_noise_std) < 0.05 * w.draft_noise_std


def test_algorithmic_bytes_by_logit_type_and_estimator():
    w = W["gqa8b_bf16"]
    plen = workloads.make_layout_inputs(w)["prompt_len"]
    a32 = workloads.algorithmic_bytes(w, plen)
    a16 = workloads.algorithmic_bytes(w.with_(logit_dtype="bf16"), plen)
    assert a32["accept_bytes"] == 2 * w.batch * w.gamma * w.V * 4 == 2 * a16["accept_bytes"]
    assert workloads.algorithmic_bytes(w.with_(temperature=0.0), plen)["accept_bytes"] == a32["accept_bytes"] // 2
    k = workloads.algorithmic_bytes(w, plen, with_khat=True)
    assert k["khat_bytes"] == w.batch * w.gamma * w.V * 4
    assert k["total_bytes"] == a32["total_bytes"] + k["khat_bytes"]
    assert a32["attn_bytes"] == 2 * int(plen.sum()) * w.Hkv * w.D * 2 + \
        w.batch * 2 * w.B * w.D * 2 * (2 * w.Hq + 2 * w.Hkv)
    assert math.isclose(a32["tokens"], w.batch * w.gamma)
