"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

* Philox4x32-10 against the published known-answer vectors.
* The masked single forward against a brute-force rebuild of every denoising state
  (SimSD notes, item 2: at the prediction slot D~_i the model sees the prompt, the data
  slots decided before step tau(i) and the still-masked slots -- exactly the
  autoregressive prefix view), with an independent complex-number RoPE.
* Perturbation invariance, B = 1 against a textbook attention routine (torch SDPA),
  identity tau = the 2L / AR verification view (S2D2 page, "2L 技巧"), RoPE shift
  invariance and the D = 2 rotation, the key count of every row.
* Acceptance: special cases, the closed form E[a] = sum_k prod_{r<=k} (1 - TV(p_r, q_r))
  (total-variation bound on the SPOT page), and Monte Carlo: committed tokens follow the
  target distribution (speculative decoding is lossless, S2D2 / SPOT pages).
* Routing estimator K^ (S2D2 page, step (4)): the expectation of the accepted-prefix
  length under independent acceptances, enumerated outcome by outcome; entropy against
  scipy; closed forms for uniform and two-level distributions; a hand-worked margin case
  in a permuted step order; later rounds.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- Philox
def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat_rows())
def test_philox_known_answers(row):
    out = philox.philox4x32_10(np.array(row[:4], np.uint32), np.array(row[4:6], np.uint32))
    assert [int(x) for x in out] == row[6:]
    assert philox.philox_scalar(row[:4], row[4:6]) == row[6:]


def test_philox_vector_matches_scalar_random_inputs():
    rng = np.random.default_rng(1)
    ctr = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(64, 2), dtype=np.uint64).astype(np.uint32)
    out = philox.philox4x32_10(ctr, key)
    for i in range(64):
        assert [int(x) for x in out[i]] == philox.philox_scalar(ctr[i], key[i])


def test_uniforms_open_interval_and_exact_in_fp32():
    u = philox.resample_uniforms(seed=123, offset=7, request=3, V=200_000)
    assert u.min() > 0.0 and u.max() < 1.0
    assert np.all(u.astype(np.float32).astype(np.float64) == u)
    # uniformity (Kolmogorov-Smirnov against U(0,1))
    from scipy import stats
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # accept and resample streams differ; requests and offsets differ
    a = philox.accept_uniforms(123, 7, 3, 8)
    b = philox.accept_uniforms(123, 7, 4, 8)
    c = philox.accept_uniforms(123, 8, 3, 8)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    assert not np.array_equal(a, u[:8])


# --------------------------------------------------------------------------- layout
def test_layout_positions_and_labels():
    tau = np.array([[2, 3, 1], [1, 2, 3]])
    plen = np.array([5, 0])
    pos, labels, err = oracle.build_layout(tau, plen)
    assert err == 0
    assert pos.tolist() == [[5, 6, 7, 5, 6, 7], [0, 1, 2, 0, 1, 2]]
    assert labels.tolist() == [[2, 3, 1, 130, 131, 129], [1, 2, 3, 129, 130, 131]]


def test_layout_invalid_requests():
    tau = np.array([[1, 1, 3], [1, 2, 3], [0, 2, 3]])
    plen = np.array([4, -1, 2])
    pos, labels, err = oracle.build_layout(tau, plen)
    assert err == (oracle.ERR_TAU | oracle.ERR_PROMPT_LEN)
    for r in range(3):
        assert pos[r].tolist() == [-1] * 6
        assert labels[r].tolist() == [0xFF] * 6


# ---------------------------------------------------------------- attention helpers
def _complex_rope(x, pos, theta):
    """Independent restatement of RoPE: pairs (d, d + D/2) as one complex number,
    multiplied by exp(i * pos * theta^(-2d/D))."""
    D = x.shape[-1]
    half = D // 2
    z = x[..., :half] + 1j * x[..., half:]
    w = np.exp(1j * np.outer(pos, theta ** (-2.0 * np.arange(half) / D)))
    z = z * w.reshape(w.shape[0], *([1] * (z.ndim - 2)), half)
    return np.concatenate([z.real, z.imag], axis=-1)


def _random_case(rng, b, B, Hq, Hkv, D, plens, taus=None):
    q = rng.standard_normal((b, 2 * B, Hq, D))
    k = rng.standard_normal((b, 2 * B, Hkv, D))
    v = rng.standard_normal((b, 2 * B, Hkv, D))
    total = int(sum(plens))
    kc = rng.standard_normal((total, Hkv, D))
    vc = rng.standard_normal((total, Hkv, D))
    offs = np.concatenate([[0], np.cumsum(plens)]).astype(np.int64)
    if taus is None:
        taus = np.stack([rng.permutation(B) + 1 for _ in range(b)])
    pos, labels, err = oracle.build_layout(taus, plens)
    assert err == 0
    return dict(q=q, k_resp=k, v_resp=v, k_cache=kc, v_cache=vc, cache_offsets=offs,
                prompt_len=np.array(plens), pos_ids=pos, labels=labels, tau=taus)


def _run(case, theta, **kw):
    return oracle.verify_attention(case["q"], case["k_resp"], case["v_resp"], case["k_cache"],
                                   case["v_cache"], case["cache_offsets"], case["prompt_len"],
                                   case["pos_ids"], case["labels"], theta, **kw)


def _softmax_attend(qv, K, V, scale):
    s = K @ qv * scale
    s = s - s.max()
    e = np.exp(s)
    return e @ V / e.sum()


# ----------------------------------------------------- P1: explicit-state brute force
@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_single_forward_equals_explicit_denoising_states(B):
    rng = np.random.default_rng(10 + B)
    Hq, Hkv, D, P, theta = 4, 2, 8, 5, 100.0
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    for perm in itertools.permutations(range(1, B + 1)):
        case = _random_case(rng, 1, B, Hq, Hkv, D, [P], taus=np.array([perm]))
        out, _ = _run(case, theta)
        tau = list(perm)
        q_rot = _complex_rope(case["q"][0], np.array(case["pos_ids"][0], float), theta)
        pos_slot = P + np.arange(B)
        kD = _complex_rope(case["k_resp"][0, :B], pos_slot.astype(float), theta)
        kM = _complex_rope(case["k_resp"][0, B:], pos_slot.astype(float), theta)
        vD, vM = case["v_resp"][0, :B], case["v_resp"][0, B:]
        for i in range(2 * B):
            slot = i % B
            t = tau[slot]
            # state seen by row i: slot k holds its decided token if tau(k) < t for a
            # prediction slot (D~), or tau(k) <= t for a data slot (D)
            decided = [(tau[k] < t) if i >= B else (tau[k] <= t) for k in range(B)]
            for h in range(Hkv):
                K = np.concatenate([case["k_cache"][:P, h],
                                    np.stack([kD[k, h] if decided[k] else kM[k, h]
                                              for k in range(B)])])
                Vv = np.concatenate([case["v_cache"][:P, h],
                                     np.stack([vD[k, h] if decided[k] else vM[k, h]
                                               for k in range(B)])])
                for g in range(G):
                    hq = h * G + g
                    ref = _softmax_attend(q_rot[i, hq], K, Vv, scale)
                    np.testing.assert_allclose(out[0, i, hq], ref, rtol=0, atol=1e-12)


def _partial_label_sets(B):
    """Every label vector of a later round of a B-slot block: a set of committed slots
    (tau = 0) and a permutation of 1..R on the others."""
    for committed in itertools.product([False, True], repeat=B):
        open_slots = [k for k in range(B) if not committed[k]]
        for perm in itertools.permutations(range(1, len(open_slots) + 1)):
            tau = [0] * B
            for k, t in zip(open_slots, perm):
                tau[k] = t
            yield tau


@pytest.mark.parametrize("B", [2, 3, 4])
def test_later_rounds_equal_explicit_denoising_states(B):
    # a slot committed in an earlier round (tau = 0) holds its token in every state, like
    # the prompt: the brute-force rebuild below marks it decided for every row of step >= 1
    rng = np.random.default_rng(40 + B)
    Hq, Hkv, D, P, theta = 2, 1, 8, 3, 100.0
    scale = 1.0 / math.sqrt(D)
    n = 0
    for tau in _partial_label_sets(B):
        if all(t == 0 for t in tau) or all(t != 0 for t in tau):
            continue
        n += 1
        case = _random_case(rng, 1, B, Hq, Hkv, D, [P], taus=np.array([tau]))
        out, _ = _run(case, theta)
        q_rot = _complex_rope(case["q"][0], np.array(case["pos_ids"][0], float), theta)
        pos_slot = (P + np.arange(B)).astype(float)
        kD = _complex_rope(case["k_resp"][0, :B], pos_slot, theta)
        kM = _complex_rope(case["k_resp"][0, B:], pos_slot, theta)
        vD, vM = case["v_resp"][0, :B], case["v_resp"][0, B:]
        for i in range(2 * B):
            t = tau[i % B]
            if t == 0:
                continue          # rows of committed slots are not predictions
            decided = [(tau[k] < t) if i >= B else (tau[k] <= t) for k in range(B)]
            K = np.concatenate([case["k_cache"][:P, 0],
                                np.stack([kD[k, 0] if decided[k] else kM[k, 0] for k in range(B)])])
            Vv = np.concatenate([case["v_cache"][:P, 0],
                                 np.stack([vD[k, 0] if decided[k] else vM[k, 0] for k in range(B)])])
            for hq in range(Hq):
                ref = _softmax_attend(q_rot[i, hq], K, Vv, scale)
                np.testing.assert_allclose(out[0, i, hq], ref, rtol=0, atol=1e-12)
    assert n > 0


def test_layout_of_later_rounds():
    taus = np.array([[0, 2, 0, 1], [0, 0, 0, 0], [3, 0, 1, 2], [0, 2, 3, 0], [1, 1, 0, 2], [5, 0, 1, 2]])
    pos, labels, err = oracle.build_layout(taus, np.array([4, 4, 4, 4, 4, 4]))
    assert err == oracle.ERR_TAU                 # rows 3 (gap), 4 (duplicate), 5 (> B)
    assert labels[0].tolist() == [0, 2, 0, 1, 128, 130, 128, 129]
    assert labels[1].tolist() == [0, 0, 0, 0, 128, 128, 128, 128]
    assert pos[0].tolist() == [4, 5, 6, 7, 4, 5, 6, 7]
    for r in (3, 4, 5):
        assert (labels[r] == oracle.INVALID_LABEL).all() and (pos[r] == -1).all()


def test_later_round_accepts_like_the_block_of_its_open_slots():
    # committed slots take no part in acceptance: the block with committed slots and the
    # smaller block made of its open slots alone (same step labels, same request ids, so
    # the same uniforms) give the same decisions and commits
    rng = np.random.default_rng(12)
    b, B, V = 5, 6, 40
    tl = rng.standard_normal((b, B, V)) * 2
    dl = tl + rng.standard_normal((b, B, V)) * 0.7
    toks = rng.integers(0, V, (b, B))
    taus, subs = [], []
    for r in range(b):
        open_slots = sorted(rng.choice(B, size=int(rng.integers(1, B + 1)), replace=False).tolist())
        perm = rng.permutation(len(open_slots)) + 1
        tau = [0] * B
        for k, t in zip(open_slots, perm):
            tau[k] = int(t)
        taus.append(tau)
        subs.append(open_slots)
    for T in (1.0, 0.0):
        gamma = B
        full = _accept_case(tl, dl, toks, taus, gamma, seed=4, T=T)
        for r in range(b):
            sl = subs[r]
            R = len(sl)
            _, lab, err = oracle.build_layout(np.array([[taus[r][k] for k in sl]]), np.zeros(1, int))
            assert err == 0
            sub = oracle.accept(tl[r:r + 1, sl], dl[r:r + 1, sl], toks[r:r + 1, sl], lab, R, T, 4, 0,
                                request_ids=[r])
            assert full["accepted_len"][r] == sub["accepted_len"][0] <= R
            assert full["n_commit"][r] == sub["n_commit"][0]
            n = int(sub["n_commit"][0])
            assert full["out_tokens"][r, :n].tolist() == sub["out_tokens"][0, :n].tolist()
            assert full["out_pos"][r, :n].tolist() == [sl[k] for k in sub["out_pos"][0, :n]]
            assert (full["out_pos"][r, n:] == -1).all()


# ------------------------------------------------------ P2: perturbation invariance
def test_perturbing_invisible_slots_leaves_prediction_rows_unchanged():
    rng = np.random.default_rng(2)
    B, Hq, Hkv, D, P, theta = 4, 2, 1, 16, 6, 1e4
    case = _random_case(rng, 1, B, Hq, Hkv, D, [P], taus=np.array([[3, 1, 4, 2]]))
    base, _ = _run(case, theta)
    tau = case["tau"][0]
    for j in range(B):
        for seg in (0, 1):
            pert = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in case.items()}
            pert["k_resp"][0, seg * B + j] += 3.0
            pert["v_resp"][0, seg * B + j] -= 2.0
            out, _ = _run(pert, theta)
            for i in range(B):
                row = B + i          # D~_i
                if seg == 0:
                    invisible = tau[j] >= tau[i]       # future or own data token
                else:
                    invisible = tau[j] < tau[i]        # mask slot already decided
                same = np.array_equal(out[0, row], base[0, row])
                assert same == invisible, (i, j, seg)
    # the prompt is visible to every row
    pert = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in case.items()}
    pert["v_cache"][0] += 1.0
    out, _ = _run(pert, theta)
    for row in range(2 * B):
        assert not np.array_equal(out[0, row], base[0, row])


# -------------------------------------------------- P3: B = 1 is prefix attention
def test_block_of_one_is_plain_prefix_attention():
    rng = np.random.default_rng(3)
    Hq, Hkv, D, theta = 4, 2, 32, 1e4
    plens = [7, 0, 12]
    case = _random_case(rng, 3, 1, Hq, Hkv, D, plens)
    out, lse = _run(case, theta)
    for r, P in enumerate(plens):
        off = int(case["cache_offsets"][r])
        q_rot = _complex_rope(case["q"][r], np.array([P, P], float), theta)
        k_rot = _complex_rope(case["k_resp"][r], np.array([P, P], float), theta)
        for row in range(2):
            for hq in range(Hq):
                h = hq // (Hq // Hkv)
                K = np.concatenate([case["k_cache"][off:off + P, h], k_rot[row:row + 1, h]])
                V = np.concatenate([case["v_cache"][off:off + P, h],
                                    case["v_resp"][r, row:row + 1, h]])
                ref = torch.nn.functional.scaled_dot_product_attention(
                    torch.tensor(q_rot[row, hq])[None, None, None],
                    torch.tensor(K)[None, None], torch.tensor(V)[None, None])[0, 0, 0].numpy()
                np.testing.assert_allclose(out[r, row, hq], ref, rtol=0, atol=1e-12)
                s = torch.tensor(K) @ torch.tensor(q_rot[row, hq]) / math.sqrt(D)
                assert abs(lse[r, row, hq] - torch.logsumexp(s, 0).item()) < 1e-12


# --------------------------------------------- P4: identity tau is the 2L / AR view
def test_identity_tau_is_autoregressive_prefix_view():
    B = 5
    A = oracle.temporal_causal_mask(list(range(1, B + 1)))
    for i in range(B):
        # prediction slot D~_i: data tokens strictly before i, mask slots from i on
        assert A[B + i, :B].tolist() == [j < i for j in range(B)]
        assert A[B + i, B:].tolist() == [j >= i for j in range(B)]
        # data slot D_i: data tokens up to and including i, mask slots after i
        assert A[i, :B].tolist() == [j <= i for j in range(B)]
        assert A[i, B:].tolist() == [j > i for j in range(B)]


# ------------------------------------------------------------- P5: RoPE properties
def test_rope_matches_complex_rotation_and_d2_case():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 3, 16))
    pos = np.array([0, 1, 5, 100, 4096, 32790])
    np.testing.assert_allclose(oracle.rope(x, pos, 1e6), _complex_rope(x, pos, 1e6),
                               atol=1e-12, rtol=0)
    x2 = rng.standard_normal((4, 1, 2))
    p2 = np.array([0.0, 1.0, 2.5, 7.0])
    got = oracle.rope(x2, p2, 1e4)
    for n in range(4):
        c, s = math.cos(p2[n]), math.sin(p2[n])
        exp = np.array([[c, -s], [s, c]]) @ x2[n, 0]
        np.testing.assert_allclose(got[n, 0], exp, atol=1e-14)


def test_attention_invariant_to_a_common_position_shift():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D, P, theta = 3, 2, 1, 16, 9, 1e4
    case = _random_case(rng, 1, B, Hq, Hkv, D, [P])
    raw_k = rng.standard_normal((P, Hkv, D))
    outs = []
    for shift in (0, 37):
        c = dict(case)
        c["k_cache"] = oracle.rope(raw_k, np.arange(P) + shift, theta)
        c["pos_ids"] = case["pos_ids"] + shift
        outs.append(_run(c, theta)[0])
    np.testing.assert_allclose(outs[0], outs[1], atol=1e-10, rtol=0)


def test_unaligned_positions_change_prediction_rows():
    """The ablation layout (SimSD notes' table, "Without Aligned RoPE"): the position ids are
    the physical indices P .. P + 2B - 1 of the response slots, and the prediction rows no
    longer match the explicit-state view that the aligned layout reproduces."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, P, theta = 4, 2, 1, 16, 6, 1e4
    case = _random_case(rng, 1, B, Hq, Hkv, D, [P])
    base, _ = _run(case, theta)
    pos, labels, err = oracle.build_layout(case["tau"], [P], aligned_rope=False)
    assert err == 0 and np.array_equal(labels, case["labels"])
    assert pos.tolist() == [list(range(P, P + 2 * B))]
    c = dict(case)
    c["pos_ids"] = pos
    out, _ = _run(c, theta)
    assert np.abs(out[0, B:] - base[0, B:]).max() > 1e-3


# ---------------------------------------------------------- P6: keys seen per row
@pytest.mark.parametrize("B", [1, 2, 5, 8, 16, 32])
def test_every_row_sees_exactly_B_response_keys(B):
    rng = np.random.default_rng(B)
    A = oracle.temporal_causal_mask(rng.permutation(B) + 1)
    assert np.all(A.sum(axis=1) == B)
    # exactly one of (D_k, D~_k) is visible to each row, for every slot k
    assert np.all(A[:, :B] ^ A[:, B:])


# ------------------------------------------------------------- P7: accept cases
def _accept_case(tl, dl, toks, tau, gamma, seed=1, offset=0, T=1.0):
    _, labels, err = oracle.build_layout(np.array(tau), np.zeros(len(tau), int))
    assert err == 0
    return oracle.accept(np.array(tl), np.array(dl), np.array(toks), labels, gamma, T,
                         seed, offset)


def test_equal_distributions_accept_everything():
    rng = np.random.default_rng(8)
    b, B, V = 6, 5, 50
    tl = rng.standard_normal((b, B, V)) * 2
    toks = rng.integers(0, V, (b, B))
    tau = [list(rng.permutation(B) + 1) for _ in range(b)]
    res = _accept_case(tl, tl.copy(), toks, tau, B)
    assert res["accepted_len"].tolist() == [B] * b
    assert res["n_commit"].tolist() == [B] * b
    for r in range(b):
        order = [tau[r].index(t) for t in range(1, B + 1)]
        assert res["out_pos"][r].tolist() == order
        assert res["out_tokens"][r].tolist() == [int(toks[r, k]) for k in order]


def test_one_hot_target_disagreeing_with_draft_rejects_and_resamples_argmax():
    B, V = 3, 20
    tl = np.full((1, B, V), -1e4)
    tl[0, :, 7] = 10.0                       # p is one-hot on token 7 in fp64
    dl = np.zeros((1, B, V))
    toks = np.array([[3, 3, 3]])
    res = _accept_case(tl, dl, toks, [[2, 1, 3]], B)
    assert res["accepted_len"][0] == 0
    assert res["n_commit"][0] == 1
    assert res["out_pos"][0].tolist() == [1, -1, -1]   # slot with tau = 1
    assert res["out_tokens"][0].tolist() == [7, -1, -1]


def test_one_hot_draft_on_a_certain_target_token_accepts():
    B, V = 2, 10
    tl = np.full((1, B, V), -1e4)
    tl[0, :, 4] = 5.0
    dl = tl.copy()
    dl[0, 1, 4] = 4.0   # still one-hot after softmax in fp64
    res = _accept_case(tl, dl, np.array([[4, 4]]), [[1, 2]], B)
    assert res["accepted_len"][0] == 2


def test_invalid_tau_and_token_sentinels():
    B, V = 3, 10
    tl = np.zeros((2, B, V))
    labels = np.array([[1, 1, 3, 129, 129, 131], [1, 2, 3, 129, 130, 131]], dtype=np.uint8)
    toks = np.array([[0, 0, 0], [0, 12, 0]])
    res = oracle.accept(tl, tl, toks, labels, B, 1.0, 0, 0)
    assert res["err"] == (oracle.ERR_TAU | oracle.ERR_TOKEN)
    assert res["accepted_len"].tolist() == [-1, -1]
    assert res["n_commit"].tolist() == [0, 0]
    assert (res["out_tokens"] == -1).all() and (res["out_pos"] == -1).all()


def test_temperature_scales_logits():
    B, V = 1, 6
    rng = np.random.default_rng(9)
    tl = rng.standard_normal((1, B, V))
    p_t2 = oracle.softmax(tl[0, 0], 2.0)
    p_half = oracle.softmax(tl[0, 0] / 2.0, 1.0)
    np.testing.assert_allclose(p_t2, p_half, atol=1e-15)


# ------------------------------------------- greedy verification (temperature 0)
def _greedy_case(seed, b=8, B=6, V=60):
    """Target logits with a clear winner per row (gap >= 3: every other entry of the fp64
    softmax at T = 1e-3 underflows to 0), a greedy drafter (draft token = argmax of the
    draft logits) that agrees with the target on a random prefix of steps."""
    rng = np.random.default_rng(seed)
    tl = rng.standard_normal((b, B, V)) * 2
    dl = tl + rng.standard_normal((b, B, V))
    for r in range(b):
        for k in range(B):
            tl[r, k, int(np.argmax(tl[r, k]))] += 3.0
            dl[r, k, int(np.argmax(dl[r, k]))] += 3.0
    tau = [list(rng.permutation(B) + 1) for _ in range(b)]
    for r in range(b):
        agree = int(rng.integers(0, B + 1))
        for t in range(1, B + 1):
            k = tau[r].index(t)
            if t <= agree:
                dl[r, k] = tl[r, k]            # the drafter's choice is the target's
            elif int(np.argmax(dl[r, k])) == int(np.argmax(tl[r, k])):
                w = (int(np.argmax(tl[r, k])) + 1) % V
                dl[r, k, w] = dl[r, k].max() + 3.0
    toks = np.argmax(dl, axis=-1)
    return tl, dl, toks, tau


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_greedy_is_the_zero_temperature_limit_of_the_stochastic_rule(seed):
    # at T -> 0 p and q are one-hot; min(1, p/q) accepts exactly when the draft token is
    # the target's argmax, and the residual max(0, p - q) is one-hot on that argmax, so
    # the race commits it: the fp64 softmax + race path at T = 1e-3 must agree with the
    # argmax path at T = 0 on every output
    tl, dl, toks, tau = _greedy_case(seed)
    B = tl.shape[1]
    cold = _accept_case(tl, dl, toks, tau, B, T=1e-3)
    greedy = _accept_case(tl, dl, toks, tau, B, T=0.0)
    for key in ("accepted_len", "n_commit", "out_tokens", "out_pos"):
        np.testing.assert_array_equal(greedy[key], cold[key])
    assert 0 < int(greedy["accepted_len"].sum()) < B * tl.shape[0]   # both branches used


def test_greedy_ignores_draft_logits_and_seed_and_takes_the_first_maximum():
    B, V = 3, 12
    tl = np.zeros((1, B, V))
    tl[0, :, 5] = 2.0
    tl[0, :, 9] = 2.0                          # tie: the first index (5) is the choice
    toks = np.array([[5, 9, 5]])
    base = _accept_case(tl, np.zeros_like(tl), toks, [[1, 2, 3]], B, seed=1, T=0.0)
    assert base["accepted_len"][0] == 1
    assert base["out_tokens"][0].tolist() == [5, 5, -1]
    assert base["out_pos"][0].tolist() == [0, 1, -1]
    other = _accept_case(tl, np.random.default_rng(3).standard_normal(tl.shape), toks,
                         [[1, 2, 3]], B, seed=77, offset=5, T=0.0)
    for key in ("accepted_len", "n_commit", "out_tokens", "out_pos"):
        np.testing.assert_array_equal(base[key], other[key])


# ------------------------------------------ coupled-noise verification (SPOT page)
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_coupled_choice_is_a_sample_of_p(T):
    # Gumbel-max identity (SPOT page, "Gumbel-Max 技巧与随机耦合"): over independent noise
    # rows (one per absolute position) argmax_v (log p_v + G_v) follows p
    z = np.array([1.2, -0.3, 0.4, 2.0, -1.1, 0.0])
    p = oracle.softmax(z, T)
    n = 20000
    counts = np.zeros(len(z))
    for a in range(n):
        counts[oracle.coupled_choice(z, T, 7, 3, 0, a)[0]] += 1
    sigma = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(counts / n - p) < 4.5 * sigma + 1e-4)


def test_coupled_drafter_agreement_meets_the_total_variation_bound():
    # SPOT page, same section: under shared noise two samplers of p and q agree with
    # probability at least (1 - delta) / (1 + delta), delta = TV(p, q)
    rng = np.random.default_rng(4)
    V, n = 12, 6000
    zt = rng.standard_normal(V) * 1.5
    zd = zt + rng.standard_normal(V) * 0.8
    p, q = oracle.softmax(zt, 1.0), oracle.softmax(zd, 1.0)
    delta = 0.5 * np.abs(p - q).sum()
    agree = sum(oracle.coupled_choice(zt, 1.0, 5, 0, 2, a)[0] == oracle.coupled_choice(zd, 1.0, 5, 0, 2, a)[0]
                for a in range(n))
    bound = (1 - delta) / (1 + delta)
    assert agree / n >= bound - 4.0 * math.sqrt(bound * (1 - bound) / n)
    assert agree / n <= 1.0 - delta + 4.0 * math.sqrt(delta * (1 - delta) / n)   # never above 1 - TV


def test_coupled_verification_at_small_temperature_is_greedy():
    tl, dl, toks, tau = _greedy_case(3)
    b, B, V = tl.shape
    pos, labels, err = oracle.build_layout(np.array(tau), np.full(b, 9))
    assert err == 0
    cold = oracle.accept_coupled(tl, toks, labels, pos, B, 1e-3, 11, 0)
    greedy = oracle.accept(tl, dl, toks, labels, B, 0.0, 11, 0)
    for key in ("accepted_len", "n_commit", "out_tokens", "out_pos"):
        np.testing.assert_array_equal(cold[key], greedy[key])


def test_coupled_verification_with_the_target_as_drafter_accepts_everything():
    rng = np.random.default_rng(6)
    b, B, V = 4, 5, 30
    tl = rng.standard_normal((b, B, V)) * 2
    tau = [list(rng.permutation(B) + 1) for _ in range(b)]
    pos, labels, _ = oracle.build_layout(np.array(tau), np.array([0, 3, 17, 40]))
    toks = np.array([[oracle.coupled_choice(tl[r, k], 0.8, 9, 1, r, pos[r, k])[0] for k in range(B)]
                     for r in range(b)])
    res = oracle.accept_coupled(tl, toks, labels, pos, B, 0.8, 9, 1)
    assert res["accepted_len"].tolist() == [B] * b
    other = oracle.accept_coupled(tl, toks, labels, pos, B, 0.8, 10, 1)   # other noise
    assert other["accepted_len"].sum() < B * b


# ----------------------------------------------- P8: Monte Carlo, lossless accept
def test_monte_carlo_commits_follow_target_and_mean_length_closed_form():
    from scipy import stats
    rng = np.random.default_rng(11)
    B = gamma = 4
    V = 16
    tl1 = rng.standard_normal((B, V)) * 1.5
    dl1 = tl1 + rng.standard_normal((B, V)) * 1.0
    p = np.stack([oracle.softmax(tl1[k], 1.0) for k in range(B)])
    q = np.stack([oracle.softmax(dl1[k], 1.0) for k in range(B)])
    N = 40_000
    tau = np.array([3, 1, 4, 2])
    order = [int(np.where(tau == t)[0][0]) for t in range(1, B + 1)]
    toks = np.stack([rng.choice(V, size=N, p=q[k]) for k in range(B)], axis=1)
    _, labels1, _ = oracle.build_layout(tau[None], np.array([0]))
    labels = np.broadcast_to(labels1, (N, 2 * B))
    tl = np.broadcast_to(tl1, (N, B, V))
    dl = np.broadcast_to(dl1, (N, B, V))
    res = oracle.accept(tl, dl, toks, labels, gamma, 1.0, seed=2024, offset=0)
    a = res["accepted_len"]
    beta = 1.0 - 0.5 * np.abs(p - q).sum(axis=1)          # per slot
    beta_steps = [beta[k] for k in order]
    expected = sum(np.prod(beta_steps[:k + 1]) for k in range(gamma))
    se = a.std() / math.sqrt(N)
    assert abs(a.mean() - expected) < 4 * se + 1e-3
    # step 1 commit ~ p at slot o_1; step 2 commit (given step 1 accepted) ~ p at o_2
    for step in (0, 1):
        sel = a >= step if step > 0 else np.ones(N, bool)
        if step > 0:
            sel = a >= 1
        counts = np.bincount(res["out_tokens"][sel, step], minlength=V)
        exp_p = p[order[step]] * sel.sum()
        keep = exp_p > 5
        chi2 = ((counts[keep] - exp_p[keep]) ** 2 / exp_p[keep]).sum()
        pval = stats.chi2.sf(chi2, keep.sum() - 1)
        assert pval > 1e-3, (step, pval)
    # a plausible mistake -- resampling from p instead of the residual -- is detectable
    counts_rej = np.bincount(res["out_tokens"][a == 0, 0], minlength=V)
    resid = np.maximum(p[order[0]] - q[order[0]], 0)
    resid /= resid.sum()
    exp_rej = resid * (a == 0).sum()
    keep = exp_rej > 5
    chi2 = ((counts_rej[keep] - exp_rej[keep]) ** 2 / exp_rej[keep]).sum()
    assert stats.chi2.sf(chi2, keep.sum() - 1) > 1e-3


# --------------------------------------------------------------------- routing estimator
def _labels_from_tau(tau):
    tau = np.asarray(tau, dtype=np.int64)
    return np.concatenate([tau, tau + 128], axis=-1).astype(np.uint8)


def _prefix_expectation_by_enumeration(alphas):
    """E[number of leading accepts] when step i is accepted independently with
    probability alphas[i]: every accept/reject pattern weighted by its probability."""
    total = 0.0
    for pattern in itertools.product([0, 1], repeat=len(alphas)):
        w = 1.0
        for a, x in zip(alphas, pattern):
            w *= a if x else 1.0 - a
        lead = 0
        while lead < len(pattern) and pattern[lead]:
            lead += 1
        total += w * lead
    return total


@pytest.mark.parametrize("B,gamma", [(4, 4), (8, 6), (6, 6)])
def test_khat_entropy_is_expected_prefix_of_independent_acceptances(B, gamma):
    """Entropy estimator with a permuted step order: alpha_i = exp(-beta H(p_i) / ln V),
    the entropies taken by scipy in the oracle's step order, then K^ against the
    enumeration of every acceptance pattern."""
    from scipy import stats
    rng = np.random.default_rng(5)
    V, T, beta = 50, 0.8, 1.7
    dl = rng.normal(0, 2, (3, B, V))
    tau = np.stack([rng.permutation(B) + 1 for _ in range(3)])
    res = oracle.expected_prefix(dl, _labels_from_tau(tau), gamma, T, oracle.KHAT_ENTROPY,
                                 beta=beta)
    assert res["err"] == 0
    for r in range(3):
        slots = [int(np.where(tau[r] == i)[0][0]) for i in range(1, gamma + 1)]
        alphas = []
        for k in slots:
            z = dl[r, k] / T
            p = np.exp(z - z.max())
            p /= p.sum()
            alphas.append(math.exp(-beta * stats.entropy(p) / math.log(V)))
        np.testing.assert_allclose(res["alpha"][r], alphas, rtol=1e-12)
        assert abs(res["khat"][r] - _prefix_expectation_by_enumeration(alphas)) < 1e-12


def test_khat_uniform_and_one_hot_closed_forms():
    """Uniform draft logits: H~ = 1 and margin 0, so K^ = sum_{k=1..L} e^(-beta k) with the
    entropy estimator and 0 with a positive margin threshold (L with threshold 0). A
    near-one-hot distribution: H~ -> 0, margin -> 1, K^ -> L."""
    B, V, beta = 5, 64, 0.9
    tau = np.array([[2, 5, 1, 4, 3]])
    lab = _labels_from_tau(tau)
    uni = np.zeros((1, B, V))
    e = oracle.expected_prefix(uni, lab, B, 1.0, oracle.KHAT_ENTROPY, beta=beta)
    geo = math.exp(-beta) * (1 - math.exp(-beta * B)) / (1 - math.exp(-beta))
    assert abs(e["khat"][0] - geo) < 1e-12
    np.testing.assert_allclose(e["entropy"][0], 1.0, rtol=1e-12)
    np.testing.assert_allclose(e["margin"][0], 0.0, atol=1e-15)
    assert oracle.expected_prefix(uni, lab, B, 1.0, oracle.KHAT_MARGIN, tau_margin=0.01)["khat"][0] == 0
    assert oracle.expected_prefix(uni, lab, B, 1.0, oracle.KHAT_MARGIN, tau_margin=0.0)["khat"][0] == B
    hot = np.zeros((1, B, V))
    hot[..., 7] = 60.0
    h = oracle.expected_prefix(hot, lab, B, 1.0, oracle.KHAT_ENTROPY, beta=beta)
    assert abs(h["khat"][0] - B) < 1e-12 and np.all(h["entropy"][0] < 1e-20)
    np.testing.assert_allclose(h["margin"][0], 1.0, rtol=1e-20)


@pytest.mark.parametrize("n_hi", [1, 2, 7])
def test_khat_two_level_distribution(n_hi):
    """n entries at logit a and V - n at logit c: p_hi = e^a / (n e^a + (V - n) e^c), and
    the entropy and margin follow in closed form (margin 0 when the maximum is shared)."""
    V, a, c, T = 40, 3.0, -1.0, 1.5
    x = np.full(V, c)
    x[[3 * i + 1 for i in range(n_hi)]] = a
    ea, ec = math.exp(a / T), math.exp(c / T)
    Z = n_hi * ea + (V - n_hi) * ec
    ph, pl = ea / Z, ec / Z
    H = -(n_hi * ph * math.log(ph) + (V - n_hi) * pl * math.log(pl))
    m, hn = oracle.draft_confidence(x, T)
    assert abs(hn - H / math.log(V)) < 1e-13
    assert abs(m - ((ph - pl) if n_hi == 1 else 0.0)) < 1e-15


def test_khat_margin_follows_the_step_order():
    """Margin estimator, worked by hand. Slots 0 and 2 confident (margin near 1), slot 1
    flat (margin 0). tau = (2, 3, 1): steps visit slots 2, 0, 1, so alpha = (1, 1, 0) and
    K^ = 1 + 1 + 0 = 2; with tau = identity alpha = (1, 0, 1) and K^ = 1."""
    V = 16
    dl = np.zeros((2, 3, V))
    dl[:, 0, 4] = dl[:, 2, 9] = 30.0
    lab = _labels_from_tau([[2, 3, 1], [1, 2, 3]])
    res = oracle.expected_prefix(dl, lab, 3, 1.0, oracle.KHAT_MARGIN, tau_margin=0.5)
    assert res["alpha"].tolist() == [[1.0, 1.0, 0.0], [1.0, 0.0, 1.0]]
    assert res["khat"].tolist() == [2.0, 1.0]


def test_khat_later_rounds_temperature_and_invalid_labels():
    """Committed slots (tau = 0) are skipped and L = min(gamma, R); logits / T at T = 1
    equal logits at T; invalid labels give K^ = -1 and the tau error bit; masked (-inf)
    entries hold no probability."""
    rng = np.random.default_rng(9)
    B, V, beta = 6, 30, 2.0
    dl = rng.normal(0, 1.5, (3, B, V))
    dl[0, :, :5] = -np.inf
    lab = _labels_from_tau([[0, 2, 0, 1, 3, 0], [3, 1, 2, 4, 6, 5], [1, 1, 2, 3, 4, 5]])
    res = oracle.expected_prefix(dl, lab, 4, 0.7, oracle.KHAT_ENTROPY, beta=beta)
    assert res["err"] == oracle.ERR_TAU and res["khat"][2] == -1
    slots0 = [3, 1, 4]                      # R = 3 < gamma: steps 1..3
    a0 = [math.exp(-beta * oracle.draft_confidence(dl[0, k], 0.7)[1]) for k in slots0]
    assert abs(res["khat"][0] - (a0[0] + a0[0] * a0[1] + a0[0] * a0[1] * a0[2])) < 1e-12
    assert res["alpha"][0, 3] == 0 and np.isnan(res["entropy"][0, 3])
    scaled = oracle.expected_prefix(dl / 0.7, lab, 4, 1.0, oracle.KHAT_ENTROPY, beta=beta)
    np.testing.assert_allclose(scaled["khat"][:2], res["khat"][:2], rtol=1e-12)
    p = oracle.softmax(dl[0, 0], 0.7)
    assert np.all(p[:5] == 0) and abs(p.sum() - 1) < 1e-12
