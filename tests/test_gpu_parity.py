"""Parity of the CUDA path (called through the C interface) with the fp64 oracle.

Integer work (layout, accept lengths, committed tokens and slots) must match bit for
bit (accept mismatches are tolerated only at oracle-reported near-ties, which are
counted); attention outputs must match within rel-L2 <= 1e-2 and max-abs <= 3e-2 for
bf16 and 1e-5 for fp32.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import helpers as H

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    H.ensure_library()
    import diffusion_speculative_verify_gb300 as pkg
    pkg.load_library()
    yield


def _pkg():
    import diffusion_speculative_verify_gb300 as pkg
    return pkg


def _step(w, inputs, meta, with_lse=True, **kw):
    pkg = _pkg()
    st = pkg.VerifyStep(inputs, gamma=w.gamma, rope_theta=w.rope_theta,
                        temperature=w.temperature, cache_layout=meta["cache_layout"],
                        with_lse=with_lse, philox_seed=meta["philox_seed"],
                        philox_offset=meta["philox_offset"], **kw)
    st.run()
    torch.cuda.synchronize()
    return st


# ----------------------------------------------------------------------------- layout
@pytest.mark.parametrize("name", workloads.WORKLOAD_ORDER)
def test_layout_bit_exact(name):
    w = W[name]
    lay = workloads.make_layout_inputs(w)
    tau, plen = lay["tau"].cuda(), lay["prompt_len"].cuda()
    b, B = tau.shape
    pos = torch.empty(b, 2 * B, dtype=torch.int32, device="cuda")
    lab = torch.empty(b, 2 * B, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _pkg().simsd_build_layout(tau, plen, pos, lab, err)
    rp, rl, re_ = oracle.build_layout(lay["tau"].numpy(), lay["prompt_len"].numpy())
    assert np.array_equal(pos.cpu().numpy(), rp)
    assert np.array_equal(lab.cpu().numpy(), rl)
    assert int(err.item()) == re_ == 0


@pytest.mark.parametrize("name", ["tiny_fp32", "ragged_bf16"])
def test_layout_physical_positions_bit_exact(name):
    """The ablation layout (mask slots at their own sequence index), later rounds and
    invalid requests included."""
    w = W[name]
    lay = workloads.make_layout_inputs(w)
    tau = _later_round_taus(np.random.default_rng(3), w.batch, w.B, invalid_every=7)
    plen = lay["prompt_len"].numpy().copy()
    plen[5 % w.batch] = -1
    b, B = tau.shape
    pos = torch.empty(b, 2 * B, dtype=torch.int32, device="cuda")
    lab = torch.empty(b, 2 * B, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _pkg().simsd_build_layout(torch.from_numpy(tau).to(torch.int32).cuda(),
                              torch.from_numpy(plen).cuda(), pos, lab, err, flags=1)
    rp, rl, re_ = oracle.build_layout(tau, plen, aligned_rope=False)
    assert np.array_equal(pos.cpu().numpy(), rp)
    assert np.array_equal(lab.cpu().numpy(), rl)
    assert int(err.item()) == re_ != 0


@pytest.mark.parametrize("case", ["fp32", "bf16", "bf16_two_ctas"])
def test_attention_physical_positions_negative_control(case):
    """Attention on the ablation layout against the oracle on the same positions (within
    the usual tolerance), and the negative control: the prediction rows move away from the
    aligned layout's by far more than that tolerance."""
    if case == "fp32":
        w = W["tiny_fp32"].with_(batch=3, B=6, gamma=6)
        plen = [32, 5, 70]
    else:
        w = MEDIUM.with_(B=32, gamma=32, Hq=6, Hkv=2) if case == "bf16_two_ctas" else MEDIUM
        plen = [0, 61, 128, 1000 + 37]
    inputs, meta = H.make_case(w, seed=13, prompt_len=plen)
    aligned = _step(w, inputs, meta)
    base = H.to_np(aligned.out).copy()
    st = _step(w, inputs, meta, aligned_rope=False)
    assert int(st.dev_err.item()) == 0
    P = np.array(plen)[:, None]
    assert np.array_equal(st.pos_ids.cpu().numpy(), P + np.arange(2 * w.B)[None])
    _attention_parity(w, inputs, meta, st)
    got = H.to_np(st.out)
    d = got[:, w.B:] - base[:, w.B:]
    assert np.linalg.norm(d) / np.linalg.norm(base[:, w.B:]) > 0.1   # 0.37-0.53 in the oracle


def test_layout_invalid_requests_and_block_32():
    B = 32
    rng = np.random.default_rng(0)
    tau = np.stack([rng.permutation(B) + 1 for _ in range(5)])
    tau[1, 3] = tau[1, 4]          # duplicate
    tau[2, 0] = 0                  # a committed slot: valid only if 1..31 remain
    tau[3, 7] = 33
    plen = np.array([10, 20, 30, 40, -5])
    pos = torch.empty(5, 2 * B, dtype=torch.int32, device="cuda")
    lab = torch.empty(5, 2 * B, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _pkg().simsd_build_layout(torch.tensor(tau, dtype=torch.int32).cuda(),
                              torch.tensor(plen, dtype=torch.int32).cuda(), pos, lab, err)
    rp, rl, re_ = oracle.build_layout(tau, plen)
    assert np.array_equal(pos.cpu().numpy(), rp)
    assert np.array_equal(lab.cpu().numpy(), rl)
    assert int(err.item()) == re_ == (oracle.ERR_TAU | oracle.ERR_PROMPT_LEN)


def _later_round_taus(rng, b, B, invalid_every=0):
    """Label vectors of later rounds: a random set of committed slots (tau = 0) and a
    permutation of 1..R on the rest; every `invalid_every`-th one gets a gap (invalid)."""
    taus = []
    for r in range(b):
        n_open = int(rng.integers(1, B + 1))
        open_slots = rng.choice(B, size=n_open, replace=False)
        tau = np.zeros(B, dtype=np.int64)
        tau[open_slots] = rng.permutation(n_open) + 1
        if invalid_every and r % invalid_every == invalid_every - 1 and n_open < B:
            tau[tau == n_open] = n_open + 1          # labels 1..R-1, R+1: a gap
        taus.append(tau)
    return np.stack(taus)


@pytest.mark.parametrize("B", [4, 8, 32])
def test_layout_later_rounds_bit_exact(B):
    rng = np.random.default_rng(B)
    b = 64
    tau = _later_round_taus(rng, b, B, invalid_every=5)
    plen = rng.integers(0, 500, b)
    pos = torch.empty(b, 2 * B, dtype=torch.int32, device="cuda")
    lab = torch.empty(b, 2 * B, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _pkg().simsd_build_layout(torch.tensor(tau, dtype=torch.int32).cuda(),
                              torch.tensor(plen, dtype=torch.int32).cuda(), pos, lab, err)
    rp, rl, re_ = oracle.build_layout(tau, plen)
    assert np.array_equal(pos.cpu().numpy(), rp)
    assert np.array_equal(lab.cpu().numpy(), rl)
    assert int(err.item()) == re_ == oracle.ERR_TAU


# -------------------------------------------------------------------------- attention
def _attention_parity(w, inputs, meta, st, requests=None, kv_heads=None):
    ref, ref_lse = H.oracle_attention(inputs, st.pos_ids, st.labels, w.rope_theta,
                                      meta["cache_layout"], requests, kv_heads)
    got = H.to_np(st.out)
    got_lse = st.lse.cpu().numpy()
    reqs = list(range(w.batch)) if requests is None else list(requests)
    heads = list(range(w.Hkv)) if kv_heads is None else list(kv_heads)
    g = H.select_heads(got[reqs], w.G, heads)
    r = H.select_heads(ref[reqs], w.G, heads)
    rel, mx = H.compare_attention(g, r, w.torch_dtype)
    gl = H.select_heads(got_lse[reqs], w.G, heads)
    rl = H.select_heads(ref_lse[reqs], w.G, heads)
    tol = H.FP32_TOL if w.torch_dtype == torch.float32 else H.BF16_LSE_ABS
    assert np.abs(gl - rl).max() <= tol
    return rel, mx


def test_attention_tiny_fp32_full():
    w = W["tiny_fp32"]
    inputs, meta = H.make_case(w)
    st = _step(w, inputs, meta)
    _attention_parity(w, inputs, meta, st)


SAMPLES = {
    "gqa8b_bf16": ([0, 7, 15], [0, 5]),
    "large_block_bf16": ([0, 31], [2, 7]),
    "long_context_bf16": ([0, 5], [1, 6]),
    "ragged_bf16": ([0, 1, 77, 200, 255], [0, 7]),
}


@pytest.mark.parametrize("name", list(SAMPLES))
def test_attention_bf16_full_size_sampled(name):
    w = W[name]
    inputs, meta = H.make_case(w)
    st = _step(w, inputs, meta)
    reqs, heads = SAMPLES[name]
    _attention_parity(w, inputs, meta, st, reqs, heads)
    assert int(st.dev_err.item()) == 0
    # every output row is finite and every lse finite at full size
    assert torch.isfinite(st.out.float()).all()
    assert torch.isfinite(st.lse).all()


MEDIUM = workloads.Workload(
    name="medium_bf16", dtype="bf16", batch=4, Hq=8, Hkv=2, D=128, B=8, prompt_len=None,
    prompt_len_range=(0, 1), rope_theta=1e6, gamma=8, V=4096)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("B", [1, 4, 8, 16, 32])
def test_attention_bf16_ragged_tiles_full_compare(layout, B):
    w = MEDIUM.with_(B=B, gamma=B)
    plen = [0, 61, 128, 1000 + 37][: w.batch]
    inputs, meta = H.make_case(w, seed=B, cache_layout=layout, prompt_len=plen)
    st = _step(w, inputs, meta)
    _attention_parity(w, inputs, meta, st)


@pytest.mark.parametrize("Hq,Hkv,B", [(6, 2, 32), (10, 2, 13), (8, 1, 9)])
def test_attention_bf16_two_ctas_partial_second_block(Hq, Hkv, B):
    # 2B*G rows per (request, kv-head) pair between 129 and 255: the pair runs on a CTA pair
    # (2-CTA cluster) whose second CTA holds a partial row block (64, 2 and 16 rows)
    w = MEDIUM.with_(Hq=Hq, Hkv=Hkv, B=B, gamma=B)
    assert 128 < 2 * B * (Hq // Hkv) < 256
    inputs, meta = H.make_case(w, seed=100 + B, prompt_len=[0, 61, 128, 1000 + 37])
    st = _step(w, inputs, meta)
    _attention_parity(w, inputs, meta, st)
    assert int(st.dev_err.item()) == 0


@pytest.mark.parametrize("Hq,Hkv,B,P", [(8, 1, 4, 20000), (32, 4, 16, 8000)])
def test_attention_bf16_one_pair_split_over_the_grid(Hq, Hkv, B, P):
    # One request whose pair(s) span nearly every schedule unit: a pair split into many
    # pieces (about one tile each), merged inside the kernel by the CTA holding its first
    # piece through many rounds of staged partials. (8, 1, 4): one 64-row pair on the
    # single-CTA kernel over about 150 units; (32, 4, 16): four 256-row pairs on CTA pairs.
    w = MEDIUM.with_(batch=1, Hq=Hq, Hkv=Hkv, B=B, gamma=B)
    inputs, meta = H.make_case(w, seed=300 + B, prompt_len=[P])
    st = _step(w, inputs, meta)
    _attention_parity(w, inputs, meta, st)
    assert int(st.dev_err.item()) == 0
    assert torch.isfinite(st.out.float()).all() and torch.isfinite(st.lse).all()


@pytest.mark.parametrize("B", [4, 16])
def test_attention_bf16_later_rounds(B):
    # committed slots (tau = 0) are seen by every open row through their data slot and by
    # none through their mask slot
    w = MEDIUM.with_(B=B, gamma=B)
    tau = _later_round_taus(np.random.default_rng(50 + B), w.batch, B)
    inputs, meta = H.make_case(w, seed=B, prompt_len=[0, 61, 128, 1000 + 37], tau=tau)
    st = _step(w, inputs, meta)
    assert int(st.dev_err.item()) == 0
    _attention_parity(w, inputs, meta, st)


def test_attention_fp32_later_rounds():
    w = W["tiny_fp32"].with_(batch=3, Hq=4, Hkv=2, D=128, B=8, gamma=8, rope_theta=1e6)
    tau = _later_round_taus(np.random.default_rng(7), 3, 8)
    inputs, meta = H.make_case(w, seed=9, prompt_len=[0, 33, 777], tau=tau)
    st = _step(w, inputs, meta)
    _attention_parity(w, inputs, meta, st)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_accept_later_rounds_bit_exact(T):
    """Later rounds verify min(gamma, R) steps of their R open slots (gamma = B here, so
    most requests verify fewer than gamma)."""
    w = W["gqa8b_bf16"].with_(B=8, gamma=8, batch=24, temperature=T)
    tau = _later_round_taus(np.random.default_rng(11), w.batch, w.B)
    inputs, meta = H.make_case(w, seed=13, tau=tau)
    st = _step(w, inputs, meta, with_lse=False)
    res = H.oracle_accept(inputs, st.labels, w.gamma, T, meta["philox_seed"], 0)
    got, err = _accept_outputs("workspace", inputs["target_logits"], inputs["draft_logits"],
                               inputs["draft_tokens"], st.labels, w.gamma, T, meta["philox_seed"])
    assert err == 0
    reqs = list(range(w.batch))
    assert H.check_accept(res, got, reqs) <= 1
    R = (tau != 0).sum(axis=1)
    assert (got["accepted_len"] <= R).all() and (got["n_commit"] <= R).all()


def test_attention_bf16_identity_tau_and_d64():
    w = MEDIUM.with_(D=64, B=4, gamma=4)
    tau = [[1, 2, 3, 4]] * w.batch
    inputs, meta = H.make_case(w, seed=3, prompt_len=[5, 300, 0, 64], tau=tau)
    st = _step(w, inputs, meta)
    _attention_parity(w, inputs, meta, st)


def test_attention_fp32_ragged_and_long_positions():
    w = W["tiny_fp32"].with_(batch=3, Hq=4, Hkv=2, D=128, B=8, gamma=8, rope_theta=1e6)
    inputs, meta = H.make_case(w, seed=9, prompt_len=[0, 33, 777])
    st = _step(w, inputs, meta)
    _attention_parity(w, inputs, meta, st)
    # large absolute positions (RoPE angle accuracy): shift the prompt start
    w2 = W["tiny_fp32"].with_(batch=1, B=4, gamma=4)
    inputs, meta = H.make_case(w2, seed=10, prompt_len=[40000])
    st = _step(w2, inputs, meta)
    _attention_parity(w2, inputs, meta, st)


def test_attention_invalid_request_rows_are_zero():
    w = MEDIUM.with_(B=4, gamma=4)
    tau = [[1, 2, 3, 4], [1, 1, 3, 4], [2, 1, 4, 3], [4, 3, 2, 1]]
    inputs, meta = H.make_case(w, seed=4, prompt_len=[10, 20, 30, 40], tau=tau)
    st = _step(w, inputs, meta)
    assert int(st.dev_err.item()) & oracle.ERR_TAU
    assert torch.count_nonzero(st.out[1].float()) == 0
    assert torch.isneginf(st.lse[1]).all()
    _attention_parity(w, inputs, meta, st, requests=[0, 2, 3])


@pytest.mark.parametrize("case", ["one_cta_per_pair", "split_pairs_two_ctas"])
def test_attention_bounded_wait_gives_up_and_next_call_is_exact(case):
    """The kernel's warps wait on one another (copies, MMAs, softmax), each wait bounded by
    wait_limit_ns. A limit of 1 ns makes those waits run out (the pipeline takes microseconds),
    which exercises the give-up path without hanging anything: the call returns, the error
    word carries SIMSD_DEVERR_TIMEOUT, every output row is either the row a normal call
    produces (bit for bit: same schedule, same arithmetic) or all NaN, and the next call with
    the default limit, on the same context, reproduces the normal output."""
    pkg = _pkg()
    if case == "one_cta_per_pair":
        w = MEDIUM.with_(B=8, gamma=8)
        plen = [0, 61, 128, 1000 + 37]
    else:  # 192 rows per pair (two CTAs each) and long prompts: pairs split across units
        w = MEDIUM.with_(Hq=6, Hkv=2, B=32, gamma=32)
        plen = [20000, 61, 128, 9000]
    inputs, meta = H.make_case(w, seed=21, prompt_len=plen)
    st = _step(w, inputs, meta)
    assert int(st.dev_err.item()) == 0
    _attention_parity(w, inputs, meta, st)
    ref_out, ref_lse = st.out.clone(), st.lse.clone()

    st.params.wait_limit_ns = 1
    st.dev_err.zero_()
    st.out.fill_(7.0)
    st.lse.fill_(7.0)
    st.attention()
    torch.cuda.synchronize()
    err = int(st.dev_err.item())
    assert err & pkg.DEVERR_TIMEOUT, err
    out = st.out.float().reshape(-1, w.D)
    ref = ref_out.float().reshape(-1, w.D)
    nan_rows = torch.isnan(out).all(dim=1)
    same_rows = (out == ref).all(dim=1)
    assert bool((nan_rows | same_rows).all())
    assert int(nan_rows.sum()) > 0
    lse, rlse = st.lse.reshape(-1), ref_lse.reshape(-1)
    assert bool((torch.isnan(lse) | (lse == rlse)).all())
    assert bool((torch.isnan(lse) == nan_rows).all())

    st.params.wait_limit_ns = 0   # the default limit: a normal call on the same context
    st.dev_err.zero_()
    st.attention()
    torch.cuda.synchronize()
    assert int(st.dev_err.item()) == 0
    assert torch.equal(st.out, ref_out) and torch.equal(st.lse, ref_lse)


def test_masked_slots_do_not_influence_prediction_rows():
    w = MEDIUM.with_(batch=1, B=8, gamma=8)
    tau = [[3, 8, 1, 6, 2, 7, 4, 5]]
    inputs, meta = H.make_case(w, seed=5, prompt_len=[300], tau=tau)
    st = _step(w, inputs, meta)
    base = st.out.clone()
    t = tau[0]
    i = 3                                   # prediction slot D~_3, tau = 6
    for j in range(8):
        for seg in (0, 1):
            invisible = (t[j] >= t[i]) if seg == 0 else (t[j] < t[i])
            if not invisible:
                continue
            inputs["k_resp"][0, seg * 8 + j] += 1.0
            inputs["v_resp"][0, seg * 8 + j] -= 1.0
    st.run()
    torch.cuda.synchronize()
    assert torch.equal(st.out[0, 8 + i], base[0, 8 + i])
    # a visible response slot (the data slot decided at step 1) does change it
    j = t.index(1)
    inputs["v_resp"][0, j] += 1.0
    st.run()
    torch.cuda.synchronize()
    assert not torch.equal(st.out[0, 8 + i], base[0, 8 + i])


# ----------------------------------------------------------------------------- accept
ACC_SAMPLE = {"tiny_fp32": None, "gqa8b_bf16": None, "large_block_bf16": None,
              "long_context_bf16": None, "ragged_bf16": list(range(0, 256, 4))}


@pytest.mark.parametrize("name", workloads.WORKLOAD_ORDER)
def test_accept_bit_exact(name):
    w = W[name]
    inputs, meta = H.make_case(w)
    st = _step(w, inputs, meta, with_lse=False)
    reqs = ACC_SAMPLE[name] or list(range(w.batch))
    res = H.oracle_accept(inputs, st.labels, w.gamma, w.temperature, meta["philox_seed"],
                          meta["philox_offset"], requests=reqs)
    got = {k: getattr(st, k).cpu().numpy() for k in
           ("accepted_len", "n_commit", "out_tokens", "out_pos")}
    ties = H.check_accept(res, got, reqs)
    assert ties <= max(1, len(reqs) // 100)
    assert int(st.dev_err.item()) == 0


def test_accept_equal_logits_accept_everything():
    w = W["gqa8b_bf16"].with_(batch=8, V=5000)
    inputs, meta = H.make_case(w, seed=2)
    inputs["draft_logits"].copy_(inputs["target_logits"])
    st = _step(w, inputs, meta, with_lse=False)
    assert st.accepted_len.tolist() == [w.gamma] * 8
    assert st.n_commit.tolist() == [w.gamma] * 8


@pytest.mark.parametrize("T", [0.7, 1.0, 1.5])
def test_accept_temperatures_and_odd_vocab(T):
    w = W["tiny_fp32"].with_(batch=64, B=8, gamma=6, V=1001, temperature=T)
    inputs, meta = H.make_case(w, seed=11)
    st = _step(w, inputs, meta, with_lse=False)
    reqs = list(range(w.batch))
    res = H.oracle_accept(inputs, st.labels, w.gamma, T, meta["philox_seed"],
                          meta["philox_offset"])
    got = {k: getattr(st, k).cpu().numpy() for k in
           ("accepted_len", "n_commit", "out_tokens", "out_pos")}
    H.check_accept(res, got, reqs)
    assert (st.accepted_len.cpu().numpy() < w.gamma).any()


@pytest.mark.parametrize("V", [5001, 4096])
def test_accept_more_requests_than_finish_ctas(V):
    """More requests than the finish kernel's resident CTAs (700 against at most 304 on
    GB300): its (request, group of 4 entries) ranges are cut across request boundaries, so
    one CTA walks two or three requests in turn and most requests' races straddle two CTAs.
    Every 37th request has a malformed step order; its sentinel outputs come from the CTA
    holding its first group. V = 5001 takes the unvectorised loads."""
    b, B = 700, 8
    g = torch.Generator().manual_seed(71 + V)
    tl = 2.0 * torch.randn(b, B, V, generator=g)
    dl = tl + 0.7 * torch.randn(b, B, V, generator=g)
    toks = torch.randint(0, V, (b, B), generator=g, dtype=torch.int32)
    tau = torch.stack([torch.randperm(B, generator=g) + 1 for _ in range(b)]).to(torch.uint8)
    bad = list(range(0, b, 37))
    for r in bad:
        tau[r, 1] = tau[r, 0]  # a repeated step: not a permutation
    labels = torch.cat([tau, tau | 0x80], dim=1)
    got, err = _accept_outputs("workspace", tl.cuda(), dl.cuda(), toks.cuda(), labels.cuda(), B,
                               1.0, 123)
    res = oracle.accept(tl.numpy(), dl.numpy(), toks.numpy(), labels.numpy(), B, 1.0, 123, 0)
    assert err == res["err"] == oracle.ERR_TAU
    assert all(got["accepted_len"][r] == -1 for r in bad)
    ties = H.check_accept(res, got, range(b))
    assert ties <= 7
    assert (got["accepted_len"] < B).sum() > b // 2  # most requests race


BF16_ACCEPT_CASES = {
    "tiny_fp32": dict(),
    "tiny_odd_vocab": dict(base="tiny_fp32", batch=64, B=8, gamma=6, V=1001),
    "gqa8b_bf16": dict(),
    "gqa8b_t07": dict(base="gqa8b_bf16", temperature=0.7),
    "large_block_bf16": dict(),
    "ragged_bf16": dict(),
}


@pytest.mark.parametrize("case", list(BF16_ACCEPT_CASES))
def test_accept_bf16_logits_bit_exact(case):
    """bf16 target / draft logits through the step: against the oracle on their exactly
    widened values, and identical to the fp32 call on those widened arrays (the kernels
    widen each entry on load and change nothing else). Odd V takes the unvectorised loads."""
    kw = dict(BF16_ACCEPT_CASES[case])
    name = kw.pop("base", case)
    w = W[name].with_(logit_dtype="bf16", **kw)
    inputs, meta = H.make_case(w, seed=51)
    assert inputs["target_logits"].dtype == torch.bfloat16
    st = _step(w, inputs, meta, with_lse=False)
    reqs = ACC_SAMPLE.get(name) or list(range(w.batch))
    res = H.oracle_accept(inputs, st.labels, w.gamma, w.temperature, meta["philox_seed"],
                          meta["philox_offset"], requests=reqs)
    got = {k: getattr(st, k).cpu().numpy() for k in
           ("accepted_len", "n_commit", "out_tokens", "out_pos")}
    ties = H.check_accept(res, got, reqs)
    assert ties <= max(1, len(reqs) // 100)
    assert int(st.dev_err.item()) == 0
    got32, err = _accept_outputs("workspace", inputs["target_logits"].float(),
                                 inputs["draft_logits"].float(), inputs["draft_tokens"],
                                 st.labels, w.gamma, w.temperature, meta["philox_seed"])
    assert err == 0
    for k in got:
        assert np.array_equal(got[k], got32[k]), k


def test_accept_invalid_labels_and_tokens():
    pkg = _pkg()
    B, V = 4, 100
    tl = torch.randn(3, B, V, device="cuda")
    toks = torch.tensor([[1, 2, 3, 4], [1, 2, 300, 4], [0, 0, 0, 0]], dtype=torch.int32,
                        device="cuda")
    labels = torch.tensor([[1, 2, 3, 4, 129, 130, 131, 132],
                           [1, 2, 3, 4, 129, 130, 131, 132],
                           [1, 1, 3, 4, 129, 129, 131, 132]], dtype=torch.uint8, device="cuda")
    out = {k: torch.full((3,), 7, dtype=torch.int32, device="cuda")
           for k in ("accepted_len", "n_commit")}
    ot = torch.zeros(3, B, dtype=torch.int32, device="cuda")
    op = torch.zeros(3, B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(pkg.simsd_accept_workspace(3, B, B, V), dtype=torch.uint8, device="cuda")
    pkg.simsd_accept(tl, tl, toks, labels, B, 1.0, 1, 0, out["accepted_len"], ot, op,
                     out["n_commit"], ws, err)
    torch.cuda.synchronize()
    res = oracle.accept(tl.cpu().numpy(), tl.cpu().numpy(), toks.cpu().numpy(),
                        labels.cpu().numpy(), B, 1.0, 1, 0)
    assert out["accepted_len"].tolist() == res["accepted_len"].tolist() == [4, -1, -1]
    assert out["n_commit"].tolist() == res["n_commit"].tolist()
    assert np.array_equal(ot.cpu().numpy(), res["out_tokens"])
    assert np.array_equal(op.cpu().numpy(), res["out_pos"])
    assert int(err.item()) == res["err"] == (oracle.ERR_TAU | oracle.ERR_TOKEN)


def _accept_outputs(path, tl, dl, toks, labels, gamma, T, seed, ws=None):
    """Runs one acceptance entry point: "workspace" (simsd_accept on a caller workspace,
    `ws` or a fresh zeroed one), "bf16" (simsd_accept_ex on bf16 logits, same workspace
    rule) or "fixed" (simsd_accept_noalloc on the library's array)."""
    pkg = _pkg()
    b, B, V = tl.shape
    out = {k: torch.full((b,), -7, dtype=torch.int32, device="cuda")
           for k in ("accepted_len", "n_commit")}
    out |= {k: torch.full((b, B), -7, dtype=torch.int32, device="cuda")
            for k in ("out_tokens", "out_pos")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (tl, dl, toks, labels, gamma, T, seed, 0, out["accepted_len"], out["out_tokens"],
            out["out_pos"], out["n_commit"])
    if path in ("workspace", "bf16"):
        if ws is None:
            ws = torch.zeros(pkg.simsd_accept_workspace(b, B, gamma, V), dtype=torch.uint8,
                             device="cuda")
        (pkg.simsd_accept_ex if path == "bf16" else pkg.simsd_accept)(*args, ws, err)
    else:
        pkg.simsd_accept_noalloc(*args, err)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, int(err.item())


def _slot_order(labels_row, B):
    tau = [int(x) & 0x7F for x in labels_row[:B]]
    return [tau.index(t) for t in range(1, B + 1)]


@pytest.mark.parametrize("path", ["workspace", "fixed", "bf16"])
@pytest.mark.parametrize("name", ["tiny_fp32", "gqa8b_bf16", "large_block_bf16"])
def test_accept_greedy_bit_exact(name, path):
    """Greedy verification (temperature 0) against the oracle, bit-exact: draft tokens
    agree with the target's first-maximum choice on a prefix of every length 0..gamma, and
    some rows hold an exact tie of their maximum at an index half the vocabulary away
    (another chunk), so the first-index rule is exercised across the chunk merge. With
    bf16 logits (8-bit mantissa) many rows also tie by rounding."""
    w = W[name]
    inputs, meta = H.make_case(w, seed=31)
    st = _step(w, inputs, meta, with_lse=False)
    b, B, V = inputs["target_logits"].shape
    tl = inputs["target_logits"].clone()
    dl = inputs["draft_logits"]
    if path == "bf16":
        tl, dl = tl.to(torch.bfloat16), dl.to(torch.bfloat16)
    labels = H.to_np(st.labels)
    tl_cpu = H.to_np(tl)
    for r in range(0, b, 3):                      # ties: the maximum copied elsewhere
        for k in range(B):
            c = int(np.argmax(tl_cpu[r, k]))
            far = (c + V // 2) % V
            tl_cpu[r, k, far] = tl_cpu[r, k, c]
    tl.copy_(torch.from_numpy(tl_cpu))
    toks = inputs["draft_tokens"].cpu().clone()
    for r in range(b):
        order = _slot_order(labels[r], B)
        L = r % (w.gamma + 1)
        for t in range(w.gamma):
            k = order[t]
            c = oracle.greedy_choice(tl_cpu[r, k])
            toks[r, k] = c if t < L else (c + 1 + r) % V
    toks = toks.cuda()
    case = dict(inputs, target_logits=tl, draft_tokens=toks)
    res = H.oracle_accept(case, st.labels, w.gamma, 0.0, meta["philox_seed"], 0)
    got, err = _accept_outputs(path, tl, dl, toks, st.labels, w.gamma, 0.0, meta["philox_seed"])
    assert err == 0
    assert H.check_accept(res, got, list(range(b))) == 0
    assert set(res["accepted_len"].tolist()) == set(range(min(b, w.gamma + 1)))


@pytest.mark.parametrize("ldt", ["fp32", "bf16"])
@pytest.mark.parametrize("V", [5000, 5001])
def test_accept_greedy_masked_rows(V, ldt):
    """Greedy verification on masked vocabularies (-inf entries): a fully masked row (its
    first index is the choice), rows masked except a few entries, the maximum at the first
    or the last entry, and a maximum repeated across chunks; V = 5001 takes the unvectorised
    loads. Bit-exact against the oracle."""
    b, B, gamma = 12, 4, 4
    g = torch.Generator(device="cpu").manual_seed(61)
    tl = torch.randn(b, B, V, generator=g) * 2
    tl[0] = -math.inf                                   # every row of request 0 fully masked
    keep = torch.rand(b, B, V, generator=g) < 0.01
    tl[1][~keep[1]] = -math.inf                         # request 1: 1 % of the entries left
    tl[2, :, 0] = 50.0                                  # maximum at the first entry
    tl[3, :, V - 1] = 50.0                              # ... at the last entry
    tl[4, :, 7] = 40.0
    tl[4, :, V - 3] = 40.0                              # repeated far apart: the first wins
    tl[5, :, : V // 2] = -math.inf                      # first half masked
    if ldt == "bf16":
        tl = tl.to(torch.bfloat16)
    tl_cpu = H.to_np(tl)
    tau = torch.stack([torch.randperm(B, generator=g) + 1 for _ in range(b)]).to(torch.int32)
    labels = torch.cat([tau, tau + 128], 1).to(torch.uint8)
    toks = torch.zeros(b, B, dtype=torch.int32)
    for r in range(b):
        order = _slot_order(labels[r].numpy(), B)
        L = r % (gamma + 1)
        for t in range(gamma):
            k = order[t]
            c = oracle.greedy_choice(tl_cpu[r, k])
            toks[r, k] = c if t < L else (c + 1) % V
    res = oracle.accept(tl_cpu, tl_cpu, toks.numpy(), labels.numpy(), gamma, 0.0, 3, 0)
    path = "bf16" if ldt == "bf16" else "workspace"
    got, err = _accept_outputs(path, tl.cuda(), tl.cuda(), toks.cuda(), labels.cuda(), gamma,
                               0.0, 3)
    assert err == 0
    assert H.check_accept(res, got, list(range(b))) == 0
    assert res["accepted_len"][0] == 0 and 0 in res["out_tokens"][0].tolist()


def _coupled_outputs(tl, toks, labels, pos, gamma, T, seed):
    pkg = _pkg()
    b, B, V = tl.shape
    out = {k: torch.full((b,), -7, dtype=torch.int32, device="cuda")
           for k in ("accepted_len", "n_commit")}
    out |= {k: torch.full((b, B), -7, dtype=torch.int32, device="cuda")
            for k in ("out_tokens", "out_pos")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(pkg.simsd_accept_workspace(b, B, gamma, V), dtype=torch.uint8, device="cuda")
    call = pkg.simsd_accept_coupled_ex if tl.dtype == torch.bfloat16 else pkg.simsd_accept_coupled
    call(tl, toks, labels, pos, gamma, T, seed, 0, out["accepted_len"], out["out_tokens"],
         out["out_pos"], out["n_commit"], ws, err)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, int(err.item())


@pytest.mark.parametrize("name,T,later,ldt", [
    ("tiny_fp32", 1.0, False, "fp32"), ("gqa8b_bf16", 1.0, False, "fp32"),
    ("gqa8b_bf16", 0.8, True, "fp32"), ("gqa8b_bf16", 0.0, False, "fp32"),
    ("gqa8b_bf16", 1.0, True, "bf16"), ("tiny_fp32", 0.0, False, "bf16")])
def test_accept_coupled_bit_exact(name, T, later, ldt):
    """Coupled-noise verification against the oracle. Half of the requests propose the
    drafter's coupled choice (draft logits, same noise), the others the target's own (all
    accepted); bit-exact except where the oracle's two best keys are within 1e-4. With bf16
    logits the oracle runs on their exactly widened values."""
    w = W[name].with_(temperature=T if T > 0 else 1.0, logit_dtype=ldt)
    tau = _later_round_taus(np.random.default_rng(23), w.batch, w.B) if later else None
    inputs, meta = H.make_case(w, seed=41, tau=tau)
    st = _step(w, inputs, meta, with_lse=False)
    b, B, V = inputs["target_logits"].shape
    seed = meta["philox_seed"]
    labels = H.to_np(st.labels)
    pos = H.to_np(st.pos_ids)
    tl_cpu = H.to_np(inputs["target_logits"])
    dl_cpu = H.to_np(inputs["draft_logits"])
    toks = inputs["draft_tokens"].cpu().clone()
    for r in range(b):
        src = tl_cpu if r % 2 else dl_cpu
        for k in range(B):
            if int(labels[r, k]) & 0x7F:
                toks[r, k] = oracle.coupled_choice(src[r, k], T, seed, 0, r, int(pos[r, k]))[0]
    toks = toks.cuda()
    res = oracle.accept_coupled(tl_cpu, toks.cpu().numpy(), labels, pos, w.gamma, T, seed, 0)
    got, err = _coupled_outputs(inputs["target_logits"], toks, st.labels, st.pos_ids, w.gamma, T, seed)
    assert err == 0
    ties = 0
    for r in range(b):
        same = all(np.array_equal(got[k][r], res[k][r])
                   for k in ("accepted_len", "n_commit", "out_tokens", "out_pos"))
        if not same:
            assert min(res["diag"][r]["key_gaps"]) < 1e-4, (r, got["accepted_len"][r], res["accepted_len"][r])
            ties += 1
    assert ties <= max(1, b // 16)
    for r in range(1, b, 2):   # the target as its own drafter: everything open is accepted
        R = int(sum(1 for k in range(B) if int(labels[r, k]) & 0x7F))
        assert res["accepted_len"][r] == min(w.gamma, R)


@pytest.mark.parametrize("name,T", [("tiny_fp32", 1.0), ("gqa8b_bf16", 1.0),
                                    ("gqa8b_bf16", 0.7)])
def test_accept_fixed_scratch_entry_bit_exact(name, T):
    """The allocation-free entry point (its scratch a fixed array in the library) against
    the oracle."""
    w = W[name].with_(temperature=T)
    inputs, meta = H.make_case(w, seed=21)
    st = _step(w, inputs, meta, with_lse=False)
    reqs = list(range(w.batch))
    res = H.oracle_accept(inputs, st.labels, w.gamma, T, meta["philox_seed"], 0)
    got, err = _accept_outputs("fixed", inputs["target_logits"], inputs["draft_logits"],
                               inputs["draft_tokens"], st.labels, w.gamma, T,
                               meta["philox_seed"])
    ties = H.check_accept(res, got, reqs)
    assert ties <= max(1, len(reqs) // 100)
    assert err == 0


@pytest.mark.parametrize("path", ["workspace", "fixed"])
def test_accept_residual_vanishing_in_fp32_races_on_p(path):
    """Target and draft logits equal except at the draft tokens, which sit far below every
    other logit (-20 in the draft, -30 in the target): step 1 is rejected (p/q = e^-10 at
    the token) while in fp32 the two softmaxes agree everywhere else, so max(0, p - q) is
    0 at every entry and the race runs on p. In fp64 the residual is e^(t_v) (1/S_t - 1/S_d)
    for v != token, i.e. proportional to p there, so the oracle draws the same winner."""
    b, B, V = 16, 4, 5000
    g = torch.Generator(device="cpu").manual_seed(31)
    dl = torch.randn(b, B, V, generator=g)
    tl = dl.clone()
    toks = torch.randint(0, V, (b, B), generator=g, dtype=torch.int32)
    for r in range(b):
        for k in range(B):
            dl[r, k, toks[r, k]] = -20.0
            tl[r, k, toks[r, k]] = -30.0
    tau = torch.tensor([3, 1, 4, 2], dtype=torch.int32)
    labels = torch.cat([tau, tau + 128]).to(torch.uint8).repeat(b, 1)
    res = oracle.accept(tl.numpy(), dl.numpy(), toks.numpy(), labels.numpy(), B, 1.0, 5, 0)
    got, err = _accept_outputs(path, tl.cuda(), dl.cuda(), toks.cuda(), labels.cuda(), B, 1.0, 5)
    assert (res["accepted_len"] < B).all()
    H.check_accept(res, got, list(range(b)))
    assert err == 0


def test_accept_one_workspace_across_shapes():
    """One workspace, zeroed once, serving calls of different shapes in a row (batch, B,
    gamma and V all change, so every scratch region moves): each call against the oracle.
    The per-request state is cleared by every call; only the barrier words at the head of
    the workspace carry over."""
    pkg = _pkg()
    shapes = [(4, 4, 4, 5000), (16, 8, 6, 1000), (2, 32, 32, 30000), (24, 4, 3, 2048)]
    need = max(pkg.simsd_accept_workspace(b, B, g, V) for b, B, g, V in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    gen = torch.Generator(device="cpu").manual_seed(41)
    for i, (b, B, gamma, V) in enumerate(shapes):
        tl = torch.randn(b, B, V, generator=gen)
        dl = tl + 0.7 * torch.randn(b, B, V, generator=gen)
        toks = torch.randint(0, V, (b, B), generator=gen, dtype=torch.int32)
        tau = torch.stack([torch.randperm(B, generator=gen) + 1 for _ in range(b)]).to(torch.int32)
        labels = torch.cat([tau, tau + 128], 1).to(torch.uint8)
        res = oracle.accept(tl.numpy(), dl.numpy(), toks.numpy(), labels.numpy(), gamma, 1.0,
                            100 + i, 0)
        got, err = _accept_outputs("workspace", tl.cuda(), dl.cuda(), toks.cuda(), labels.cuda(),
                                   gamma, 1.0, 100 + i, ws=ws)
        H.check_accept(res, got, list(range(b)))
        assert err == 0


def test_accept_monte_carlo_commits_follow_target():
    """2^16 requests with identical logits and draft tokens drawn from q: the committed
    token of step 1 follows p (chi-square), E[accepted] matches the 1 - TV closed form."""
    from scipy import stats
    pkg = _pkg()
    N, B, V = 1 << 16, 4, 16
    g = torch.Generator(device="cpu").manual_seed(77)
    tl1 = torch.randn(B, V, generator=g) * 1.5
    dl1 = tl1 + torch.randn(B, V, generator=g)
    p = torch.softmax(tl1.double(), -1).numpy()
    q = torch.softmax(dl1.double(), -1).numpy()
    tau = torch.tensor([2, 4, 1, 3], dtype=torch.int32)
    order = [int((tau == t).nonzero()) for t in range(1, B + 1)]
    toks = torch.stack([torch.multinomial(torch.tensor(q[k]), N, replacement=True, generator=g)
                        for k in range(B)], 1).to(torch.int32)
    labels = torch.cat([tau, tau + 128]).to(torch.uint8).repeat(N, 1)
    tl = tl1.repeat(N, 1, 1).cuda()
    dl = dl1.repeat(N, 1, 1).cuda()
    al = torch.empty(N, dtype=torch.int32, device="cuda")
    nc = torch.empty_like(al)
    ot = torch.empty(N, B, dtype=torch.int32, device="cuda")
    op = torch.empty_like(ot)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(pkg.simsd_accept_workspace(N, B, B, V), dtype=torch.uint8, device="cuda")
    pkg.simsd_accept(tl, dl, toks.cuda(), labels.cuda(), B, 1.0, 99, 0, al, ot, op, nc, ws, err)
    torch.cuda.synchronize()
    a = al.cpu().numpy()
    ot = ot.cpu().numpy()
    beta = 1 - 0.5 * np.abs(p - q).sum(1)
    bs = [beta[k] for k in order]
    expected = sum(np.prod(bs[:k + 1]) for k in range(B))
    assert abs(a.mean() - expected) < 4 * a.std() / math.sqrt(N) + 1e-3
    for step, sel in ((0, np.ones(N, bool)), (1, a >= 1)):
        counts = np.bincount(ot[sel, step], minlength=V)
        e = p[order[step]] * sel.sum()
        keep = e > 5
        chi2 = ((counts[keep] - e[keep]) ** 2 / e[keep]).sum()
        assert stats.chi2.sf(chi2, keep.sum() - 1) > 1e-4
    # and bit-exact against the oracle on a slice of the same requests
    reqs = list(range(0, N, 512))
    res = oracle.accept(tl1.numpy()[None].repeat(N, 0), dl1.numpy()[None].repeat(N, 0),
                        toks.numpy(), labels.numpy(), B, 1.0, 99, 0, requests=reqs)
    got = {"accepted_len": a, "n_commit": nc.cpu().numpy(), "out_tokens": ot,
           "out_pos": op.cpu().numpy()}
    H.check_accept(res, got, reqs)


# ------------------------------------------------------------------ routing estimator (K^)
ALPHA_TOL = 2e-5   # fp32 sums of e^(z - m) over a row: alpha of the entropy estimator


def _khat_gpu(dl, labels, gamma, T, mode, tau_margin, beta, with_alpha=True):
    pkg = _pkg()
    b, B, V = dl.shape
    khat = torch.full((b,), -7.0, device="cuda")
    al = torch.full((b, gamma), -7.0, device="cuda") if with_alpha else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkg.simsd_expected_prefix_workspace(b, B, gamma, V), dtype=torch.uint8,
                     device="cuda")
    pkg.simsd_expected_prefix(dl, labels, gamma, T, mode, tau_margin, beta, khat, al, ws, err)
    torch.cuda.synchronize()
    return khat.cpu().numpy(), (al.cpu().numpy() if with_alpha else None), int(err.item())


def _check_khat(res, khat, alpha, reqs, mode, tau_margin):
    """Entropy estimator: alpha within ALPHA_TOL and K^ within L(L+1)/2 ALPHA_TOL (each
    prefix product moves by at most the sum of its factors' errors). Margin estimator: the
    decisions and K^ exact, except for a request with a margin within a relative 1e-5 of
    tau_margin (counted and returned)."""
    near = 0
    for r in reqs:
        L = int(np.sum(~np.isnan(res["margin"][r])))
        if res["khat"][r] == -1:
            assert khat[r] == -1 and (alpha is None or (alpha[r] == 0).all())
            continue
        if alpha is not None:
            assert (alpha[r, L:] == 0).all()
        if mode == oracle.KHAT_MARGIN:
            close = np.abs(res["margin"][r, :L] - tau_margin) <= 1e-5 * abs(tau_margin) + 1e-12
            if close.any():
                near += 1
                continue
            if alpha is not None:
                assert np.array_equal(alpha[r, :L], res["alpha"][r, :L]), r
            assert khat[r] == res["khat"][r], (r, khat[r], res["khat"][r])
        else:
            if alpha is not None:
                assert np.abs(alpha[r, :L] - res["alpha"][r, :L]).max(initial=0) <= ALPHA_TOL, r
            assert abs(khat[r] - res["khat"][r]) <= L * (L + 1) / 2 * ALPHA_TOL, (r, khat[r], res["khat"][r])
    return near


def _spread_logits(b, B, V, seed):
    """Rows from flat to peaked (logit scale 0.3 .. 40), so margins and entropies cover
    (0, 1)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    scale = torch.exp(torch.linspace(math.log(0.3), math.log(40.0), b * B))
    scale = scale[torch.randperm(b * B, generator=g)].reshape(b, B, 1)
    return torch.randn(b, B, V, generator=g) * scale


@pytest.mark.parametrize("ldt", ["fp32", "bf16"])
@pytest.mark.parametrize("mode,T", [(0, 1.0), (0, 0.7), (1, 1.0), (1, 1.3)])
def test_expected_prefix_spread_rows(mode, T, ldt):
    """Margin and entropy estimators on rows from flat to peaked, first and later rounds
    (committed slots skipped, R < gamma for some requests), against the oracle."""
    b, B, gamma, V = 40, 8, 6, 32000
    dl = _spread_logits(b, B, V, 71)
    if ldt == "bf16":
        dl = dl.to(torch.bfloat16)
    labels = torch.from_numpy(oracle.build_layout(
        _later_round_taus(np.random.default_rng(72), b, B), np.full(b, 100))[1])
    tau_margin, beta = 0.3, 2.0
    res = oracle.expected_prefix(H.to_np(dl), labels.numpy(), gamma, T, mode, tau_margin, beta)
    khat, alpha, err = _khat_gpu(dl.cuda(), labels.cuda(), gamma, T, mode, tau_margin, beta)
    assert err == 0
    near = _check_khat(res, khat, alpha, range(b), mode, tau_margin)
    assert near <= 2
    assert len(set(np.round(res["khat"], 6))) > (5 if mode == oracle.KHAT_ENTROPY else 3)


@pytest.mark.parametrize("name", ["tiny_fp32", "gqa8b_bf16", "large_block_bf16", "ragged_bf16"])
def test_expected_prefix_in_the_step(name):
    """The estimator inside VerifyStep (between the layout and the attention) on the
    workloads' draft logits, entropy estimator at the workload's temperature; the ragged
    workload is checked on a sample of its requests."""
    w = W[name]
    inputs, meta = H.make_case(w, seed=81)
    st = _step(w, inputs, meta, with_lse=False, khat_mode=oracle.KHAT_ENTROPY, beta=1.5,
               khat_temperature=w.temperature)
    reqs = ACC_SAMPLE.get(name) or list(range(w.batch))
    idx = torch.tensor(reqs, device="cuda")
    res = oracle.expected_prefix(H.to_np(inputs["draft_logits"][idx]), H.to_np(st.labels[idx]),
                                 w.gamma, w.temperature, oracle.KHAT_ENTROPY, beta=1.5)
    khat = st.khat.cpu().numpy()[reqs]
    alpha = st.alpha.cpu().numpy()[reqs]
    _check_khat(res, khat, alpha, range(len(reqs)), oracle.KHAT_ENTROPY, 0.0)
    assert int(st.dev_err.item()) == 0


@pytest.mark.parametrize("ldt", ["fp32", "bf16"])
def test_expected_prefix_edges(ldt):
    """Odd V (unvectorised loads), masked entries, a request with invalid labels (K^ = -1,
    tau error bit), one with every slot committed (K^ = 0), a peaked row per request, no
    alpha output; and V = 1 (margin 1, entropy 0: K^ = L)."""
    b, B, gamma, V = 6, 4, 4, 1001
    dl = _spread_logits(b, B, V, 91)
    dl[1, :, : V // 2] = -math.inf
    dl[2, :, 5] = 40.0
    if ldt == "bf16":
        dl = dl.to(torch.bfloat16)
    taus = np.array([[2, 1, 4, 3], [1, 2, 3, 4], [0, 0, 0, 0], [3, 0, 1, 2], [1, 1, 2, 3],
                     [4, 3, 2, 1]])
    pos, lab, lerr = oracle.build_layout(taus, np.full(b, 10))
    assert lerr == oracle.ERR_TAU
    for mode in (oracle.KHAT_MARGIN, oracle.KHAT_ENTROPY):
        res = oracle.expected_prefix(H.to_np(dl), lab, gamma, 0.9, mode, 0.05, 0.8)
        assert res["khat"][2] == 0 and res["khat"][4] == -1
        for with_alpha in (True, False):
            khat, alpha, err = _khat_gpu(dl.cuda(), torch.from_numpy(lab).cuda(), gamma, 0.9,
                                         mode, 0.05, 0.8, with_alpha)
            assert err == oracle.ERR_TAU
            _check_khat(res, khat, alpha, range(b), mode, 0.05)
    one = torch.randn(3, B, 1)
    if ldt == "bf16":
        one = one.to(torch.bfloat16)
    khat, alpha, err = _khat_gpu(one.cuda(), torch.from_numpy(lab[:2]).cuda().repeat(2, 1)[:3],
                                 gamma, 1.0, oracle.KHAT_ENTROPY, 0.0, 3.0)
    assert err == 0 and khat.tolist() == [4.0, 4.0, 4.0] and (alpha == 1).all()
