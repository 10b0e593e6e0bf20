"""Plain fp64 CPU oracle of the SimSD single-forward speculative verification step.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg are the only code that may import this module. The CUDA library
shares no code with it (no kernels, headers, helpers, tables or constants) and the
product path never calls it.

Each function restates a definition from the pages, in their notation:

* layout    -- SimSD notes, "关键设计" items 1 and 3 (paired data/mask layout; RoPE copy);
               gist.science SimSD summary, sections 1 and 3.
* mask      -- SimSD notes, item 2, the four-case equation for A_ij; step labels tau are
               a permutation of 1..B (gist.science summary, section 2, "Mapa de Passo");
               in a later round of the same block, slots committed earlier carry tau = 0
               like the prompt, and the R remaining positions (SimSD notes, item 4) a
               permutation of 1..R.
* attention -- one softmax-attention layer over [prompt | D | D~] under A_ij, with the
               RoPE ids of D~_k copied from D_k (SimSD notes items 2-3).
* accept    -- SimSD notes item 4, equation for alpha_r = min(1, p_theta / p_phi), walked in
               the draft's time order; the first rejected slot is resampled from the
               normalised residual max(0, p - q) (S2D2 page, "方法步骤详情" step (5));
               the race draw is the Gumbel-max / exponential-race identity (SPOT page,
               "Gumbel-Max 技巧与随机耦合").
* routing   -- S2D2 page, "方法步骤详情" step (4) (the score-threshold routing policy of
               its Algorithm 4): the expected accepted-prefix length
               K^ = sum_{k=1..L} prod_{i=1..k} alpha_i with a margin-based
               alpha_i = 1[m_i >= tau_margin] or an entropy-based alpha_i = exp(-beta H~_i).

Readings taken where the pages are silent (all listed in the design notes):
  prompt tokens carry tau = 0 and are visible to every response row; RoPE pairs are
  half-split (d, d + D/2) with omega_d = theta^(-2d/D); the prompt keys arrive already
  rotated; softmax scale 1/sqrt(D); q-head h uses kv-head h // G; every slot of D and
  D~ is computed; no bonus token when all gamma drafts are accepted; a request with
  R < gamma remaining positions (which the SimSD notes hand to the regular denoising path)
  verifies its R steps.
"""
from __future__ import annotations

import math

import numpy as np

from . import philox

SEG_DATA = 0        # D_k   (reference data slot)
SEG_MASK = 1        # D~_k  ([MASK] prediction slot)
INVALID_LABEL = 0xFF

# Error bits of the per-call device error word (same meaning as the C interface).
ERR_TAU = 1          # step labels are not a permutation of 1..B
ERR_PROMPT_LEN = 2   # negative prompt length
ERR_TOKEN = 4        # draft token id outside [0, V)

# Estimators of the per-step acceptance alpha_i (same values as the C interface).
KHAT_MARGIN = 0      # alpha_i = 1[m_i >= tau_margin]
KHAT_ENTROPY = 1     # alpha_i = exp(-beta * H~_i)


# ----------------------------------------------------------------------------- layout
def build_layout(tau, prompt_len, aligned_rope=True):
    """Paired layout [prompt | D_1..D_B | D~_1..D~_B].

    Position ids: prompt token j -> j (implicit); D_k -> P + k; D~_k copies D_k's id
    (0-based k). With aligned_rope=False, the ablation of the SimSD notes' table ("Without
    Aligned RoPE", positions increasing physically), D~_k takes its own index in the
    sequence, P + B + k. Labels: one byte per response slot, (segment << 7) | tau, segment 0
    for D and 1 for D~. tau = 0 marks a slot committed in an earlier round of the same
    block (its token is known, like the prompt's); the other slots' labels must be a
    permutation of 1..R, R = their count (R = B in a block's first round). A request
    breaking this, or with a negative prompt length, gets pos = -1 and labels = 0xFF on
    all 2B slots and raises the matching error bit.
    """
    tau = np.asarray(tau, dtype=np.int64)
    prompt_len = np.asarray(prompt_len, dtype=np.int64)
    b, B = tau.shape
    pos = np.zeros((b, 2 * B), dtype=np.int32)
    labels = np.zeros((b, 2 * B), dtype=np.uint8)
    err = 0
    for r in range(b):
        P = int(prompt_len[r])
        bad = 0
        open_steps = sorted(t for t in tau[r].tolist() if t != 0)
        if any(t < 0 or t > B for t in tau[r].tolist()) or open_steps != list(range(1, len(open_steps) + 1)):
            bad |= ERR_TAU
        if P < 0:
            bad |= ERR_PROMPT_LEN
        err |= bad
        for k in range(B):
            if bad:
                pos[r, k] = pos[r, B + k] = -1
                labels[r, k] = labels[r, B + k] = INVALID_LABEL
                continue
            pos[r, k] = P + k            # data slot D_k: next response position
            pos[r, B + k] = P + k if aligned_rope else P + B + k   # D~_k: D_k's id, or its own
            labels[r, k] = (SEG_DATA << 7) | int(tau[r, k])
            labels[r, B + k] = (SEG_MASK << 7) | int(tau[r, k])
    return pos, labels, err


# ------------------------------------------------------------------------------- mask
def temporal_causal_mask(tau_row):
    """A_ij over the 2B response slots (index < B: D, index >= B: D~), the four cases
    of the SimSD mask equation written out literally."""
    tau_row = [int(t) for t in tau_row]
    B = len(tau_row)
    A = np.zeros((2 * B, 2 * B), dtype=bool)
    for i in range(2 * B):
        for j in range(2 * B):
            ti, tj = tau_row[i % B], tau_row[j % B]
            i_in_D, j_in_D = i < B, j < B
            if i_in_D and j_in_D:
                A[i, j] = tj <= ti
            elif i_in_D and not j_in_D:
                A[i, j] = tj > ti
            elif not i_in_D and j_in_D:
                A[i, j] = tj < ti
            else:
                A[i, j] = tj >= ti
    return A


# ------------------------------------------------------------------------------- RoPE
def rope(x, pos, theta):
    """Rotate x [n, H, D] at positions pos [n]: pairs (d, d + D/2) turn by
    pos * theta^(-2d/D), in fp64."""
    x = np.asarray(x, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    omega = float(theta) ** (-2.0 * np.arange(half, dtype=np.float64) / D)
    ang = pos[:, None] * omega[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


# -------------------------------------------------------------------------- attention
def _cache_rows(cache, layout, start, P, h):
    cache = np.asarray(cache)
    if layout == "NHD":
        return cache[start:start + P, h, :]
    return cache[h, start:start + P, :]


def verify_attention(q, k_resp, v_resp, k_cache, v_cache, cache_offsets, prompt_len,
                     pos_ids, labels, rope_theta, softmax_scale=0.0, cache_layout="NHD",
                     requests=None, kv_heads=None):
    """One attention layer of the verify forward.

    q [b, 2B, Hq, D], k_resp/v_resp [b, 2B, Hkv, D] (pre-RoPE), k_cache/v_cache packed
    (NHD [sumP, Hkv, D] or HND [Hkv, sumP, D], keys already rotated), cache_offsets
    [b+1], prompt_len [b], pos_ids/labels [b, 2B]. Returns (out [b, 2B, Hq, D] fp64,
    lse [b, 2B, Hq] fp64 natural-log sum-exp of the scaled scores). Only the listed
    requests / kv heads are computed (others stay 0 / -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    k_resp = np.asarray(k_resp, dtype=np.float64)
    v_resp = np.asarray(v_resp, dtype=np.float64)
    b, twoB, Hq, D = q.shape
    B = twoB // 2
    Hkv = k_resp.shape[2]
    G = Hq // Hkv
    scale = softmax_scale if softmax_scale and softmax_scale > 0 else 1.0 / math.sqrt(D)
    labels = np.asarray(labels)
    pos_ids = np.asarray(pos_ids)
    out = np.zeros((b, twoB, Hq, D), dtype=np.float64)
    lse = np.full((b, twoB, Hq), -np.inf, dtype=np.float64)
    req_list = range(b) if requests is None else requests
    head_list = range(Hkv) if kv_heads is None else kv_heads
    for r in req_list:
        if int(labels[r, 0]) == INVALID_LABEL or int(prompt_len[r]) < 0:
            continue
        P = int(prompt_len[r])
        start = int(cache_offsets[r])
        tau_row = (labels[r, :B] & 0x7F).astype(np.int64)
        A = temporal_causal_mask(tau_row)
        # every response row sees the whole prompt (tau = 0 < tau(i)), then A_ij
        visible = np.concatenate([np.ones((twoB, P), dtype=bool), A], axis=1)
        q_rot = rope(q[r], pos_ids[r], rope_theta)
        k_rot = rope(k_resp[r], pos_ids[r], rope_theta)
        for h in head_list:
            K = np.concatenate([np.asarray(_cache_rows(k_cache, cache_layout, start, P, h),
                                           dtype=np.float64), k_rot[:, h, :]], axis=0)
            Vm = np.concatenate([np.asarray(_cache_rows(v_cache, cache_layout, start, P, h),
                                            dtype=np.float64), v_resp[r, :, h, :]], axis=0)
            for g in range(G):
                hq = h * G + g
                S = (q_rot[:, hq, :] @ K.T) * scale          # [2B, P + 2B]
                S = np.where(visible, S, -np.inf)
                m = S.max(axis=1, keepdims=True)
                E = np.exp(S - m)
                denom = E.sum(axis=1, keepdims=True)
                out[r, :, hq, :] = (E @ Vm) / denom
                lse[r, :, hq] = (m + np.log(denom))[:, 0]
    return out, lse


# ----------------------------------------------------------------------------- accept
def softmax(logits, temperature):
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def _order_from_labels(labels_row, B):
    """o_r = the slot whose step label is r (r = 1..R, R = the slots not committed in an
    earlier round), or None if those labels are not a permutation of 1..R."""
    if int(labels_row[0]) == INVALID_LABEL:
        return None
    tau = [int(x) & 0x7F for x in labels_row[:B]]
    open_steps = sorted(t for t in tau if t != 0)
    if open_steps != list(range(1, len(open_steps) + 1)):
        return None
    order = [0] * len(open_steps)
    for k, t in enumerate(tau):
        if t:
            order[t - 1] = k
    return order


def greedy_choice(logits):
    """The target's own deterministic next token at temperature 0: the first index of the
    largest logit (SPOT page, verification step of Algorithm 2: at T = 0 the target's
    transition is Phi_0)."""
    return int(np.argmax(np.asarray(logits, dtype=np.float64)))


def coupled_choice(logits, temperature, seed, offset, request, position):
    """The target's own transition under the shared noise table (SPOT page, "Gumbel-Max
    技巧与随机耦合" and the coupled-noise verification of Algorithm 2): with p =
    softmax(logits / T) and Gumbel noise G_{a,v} = -ln(-ln u_{a,v}) indexed by the
    absolute output position a, Phi_G = argmax_v (log p_v + G_{a,v}), which by the
    Gumbel-max identity is a sample of p. log p_v differs from logits_v / T by a constant,
    so the keys are logits_v / T + G_{a,v}. Returns (token, gap between the two largest
    keys). T = 0 is Phi_0, the first maximum of the logits (gap: of the logits)."""
    z = np.asarray(logits, dtype=np.float64)
    if float(temperature) == 0.0:
        keys = z
    else:
        u = philox.noise_uniforms(seed, offset, request, position, z.shape[-1])
        keys = z / float(temperature) - np.log(-np.log(u))
    y = int(np.argmax(keys))          # first maximum
    top2 = np.sort(keys)[-2:] if keys.shape[-1] > 1 else np.array([-np.inf, keys[0]])
    return y, float(top2[1] - top2[0])


def accept_coupled(target_logits, draft_tokens, labels, pos_ids, gamma, temperature, seed,
                   offset, requests=None, request_ids=None):
    """Coupled-noise verification (SPOT page, Algorithm 2 and the coupled-noise
    verification paragraph): the drafter and the target share the Gumbel noise table,
    conditioned on which the target's transition Phi_G is deterministic; step r (slot
    k = o_r, absolute position a = pos_ids[k]) is accepted iff the draft token equals
    Phi_G at k, and at the first mismatch the target's own Phi_G is committed. Verifies
    min(gamma, R) steps like `accept`. No draft logits are read."""
    tl = np.asarray(target_logits)
    toks = np.asarray(draft_tokens)
    labels = np.asarray(labels)
    pos_ids = np.asarray(pos_ids)
    b, B, V = tl.shape
    acc_len = np.full(b, -1, dtype=np.int32)
    n_commit = np.zeros(b, dtype=np.int32)
    out_tokens = np.full((b, B), -1, dtype=np.int32)
    out_pos = np.full((b, B), -1, dtype=np.int32)
    err = 0
    diag = {}
    req_list = range(b) if requests is None else requests
    for r in req_list:
        order = _order_from_labels(labels[r], B)
        if order is None:
            err |= ERR_TAU
            continue
        steps = order[:gamma]
        if any(not (0 <= int(toks[r, k]) < V) for k in steps):
            err |= ERR_TOKEN
            continue
        rid = r if request_ids is None else int(request_ids[r])
        a, gaps, choice = 0, [], None
        for k in steps:
            choice, gap = coupled_choice(tl[r, k], temperature, seed, offset, rid, int(pos_ids[r, k]))
            gaps.append(gap)
            if int(toks[r, k]) != choice:
                break
            a += 1
        for step in range(a):
            out_tokens[r, step] = int(toks[r, steps[step]])
            out_pos[r, step] = steps[step]
        if a < len(steps):
            out_tokens[r, a] = choice
            out_pos[r, a] = steps[a]
        acc_len[r] = a
        n_commit[r] = a + (1 if a < len(steps) else 0)
        diag[r] = {"key_gaps": gaps}
    return {"accepted_len": acc_len, "n_commit": n_commit, "out_tokens": out_tokens,
            "out_pos": out_pos, "err": err, "diag": diag}


def accept(target_logits, draft_logits, draft_tokens, labels, gamma, temperature,
           seed, offset, requests=None, request_ids=None):
    """Speculative acceptance along the draft's time order, then residual resampling.

    A request verifies gamma_r = min(gamma, R) steps, R = its slots not committed in an
    earlier round (tau != 0); n_commit = a + [a < gamma_r].

    temperature == 0 is greedy verification (SPOT page, Algorithm 2 and its verification
    paragraph: at T = 0 the target's own next commit is the deterministic Phi_0; an edge is
    accepted iff the draft agrees with it, otherwise the target's own result is
    committed): step r is accepted iff x = argmax of the target logits at k; at the first
    mismatch the committed token is that argmax. Draft logits and uniforms are unused.

    For steps r = 1..gamma: slot k = o_r, x = draft token at k, p = softmax(target
    logits at k / T), q = softmax(draft logits at k / T); accept if p_x >= q_x, else
    accept iff u_r * q_x < p_x (u_r uniform in (0,1)); stop at the first rejection.
    At the first rejected slot draw y from max(0, p - q) (normalised) by the race
    argmax_v r_v / E_v, E_v = -ln(u_v) (ties: smallest v; if the residual is all zero,
    race on p instead). Returns dict with accepted_len [b], n_commit [b], out_tokens
    [b, B], out_pos [b, B] (slot index, step order, -1 past n_commit), err, and
    per-request diagnostics (decision margins, race top-2 keys). ``request_ids`` maps
    batch rows to the request index used in the Philox counters (default: the row).
    """
    tl = np.asarray(target_logits)
    dl = np.asarray(draft_logits)
    toks = np.asarray(draft_tokens)
    labels = np.asarray(labels)
    b, B, V = tl.shape
    acc_len = np.full(b, -1, dtype=np.int32)
    n_commit = np.zeros(b, dtype=np.int32)
    out_tokens = np.full((b, B), -1, dtype=np.int32)
    out_pos = np.full((b, B), -1, dtype=np.int32)
    err = 0
    diag = {}
    req_list = range(b) if requests is None else requests
    greedy = float(temperature) == 0.0
    for r in req_list:
        order = _order_from_labels(labels[r], B)
        if order is None:
            err |= ERR_TAU
            continue
        steps = order[:gamma]
        if any(not (0 <= int(toks[r, k]) < V) for k in steps):
            err |= ERR_TOKEN
            continue
        rid = r if request_ids is None else int(request_ids[r])
        if greedy:
            a = 0
            for k in steps:
                if int(toks[r, k]) != greedy_choice(tl[r, k]):
                    break
                a += 1
            for step in range(a):
                out_tokens[r, step] = int(toks[r, steps[step]])
                out_pos[r, step] = steps[step]
            if a < len(steps):
                out_tokens[r, a] = greedy_choice(tl[r, steps[a]])
                out_pos[r, a] = steps[a]
            acc_len[r] = a
            n_commit[r] = a + (1 if a < len(steps) else 0)
            diag[r] = {"margins": [], "race_top2": None}
            continue
        u = philox.accept_uniforms(seed, offset, rid, gamma)
        a = 0
        margins = []
        p = q = None
        for step, k in enumerate(steps):
            x = int(toks[r, k])
            p = softmax(tl[r, k], temperature)
            q = softmax(dl[r, k], temperature)
            px, qx = p[x], q[x]
            margins.append(abs(u[step] * qx - px) / qx if qx > 0 else np.inf)
            if px >= qx or u[step] * qx < px:
                a += 1
                continue
            break
        for step in range(a):
            out_tokens[r, step] = int(toks[r, steps[step]])
            out_pos[r, step] = steps[step]
        race = None
        if a < len(steps):
            k = steps[a]
            p = softmax(tl[r, k], temperature)
            q = softmax(dl[r, k], temperature)
            res = np.maximum(p - q, 0.0)
            if not np.any(res > 0):
                res = p
            uv = philox.resample_uniforms(seed, offset, rid, V)
            keys = res / (-np.log(uv))
            y = int(np.argmax(keys))          # first maximum = smallest v on ties
            top2 = np.sort(keys)[-2:] if V > 1 else np.array([0.0, keys[0]])
            race = (float(top2[1]), float(top2[0]))
            out_tokens[r, a] = y
            out_pos[r, a] = k
        acc_len[r] = a
        n_commit[r] = a + (1 if a < len(steps) else 0)
        diag[r] = {"margins": margins, "race_top2": race}
    return {"accepted_len": acc_len, "n_commit": n_commit, "out_tokens": out_tokens,
            "out_pos": out_pos, "err": err, "diag": diag}


# ----------------------------------------------------------------------------- routing
def draft_confidence(logits, temperature):
    """Confidence of the draft at one position, from its distribution p = softmax(logits / T):
    the margin m = p_(1) - p_(2) between its two largest probabilities, and the entropy
    normalised by its largest possible value, H~ = H(p) / ln V (0 when V = 1). These are the
    m_i and H~_i of the routing estimators (S2D2 page, "方法步骤详情" step (4))."""
    p = softmax(logits, temperature)
    V = p.shape[-1]
    top = np.sort(p)[::-1]
    margin = float(top[0] - (top[1] if V > 1 else 0.0))
    nz = p[p > 0]                     # 0 log 0 = 0 (masked entries)
    H = float(-np.sum(nz * np.log(nz)))
    return margin, (H / math.log(V) if V > 1 else 0.0)


def expected_prefix(draft_logits, labels, gamma, temperature, mode, tau_margin=0.0, beta=1.0,
                    requests=None):
    """Expected accepted-prefix length of every request (S2D2 page, "方法步骤详情" step (4)):

        K^ = sum_{k=1..L} prod_{i=1..k} alpha_i

    over the L = min(gamma, R) steps that verification would walk, in the draft's time order
    (step i is the slot o_i labelled i; left to right when tau is the identity), with
    alpha_i = 1[m_i >= tau_margin] (mode KHAT_MARGIN) or exp(-beta H~_i) (KHAT_ENTROPY), m_i
    and H~_i from `draft_confidence` at temperature T > 0.

    Returns khat [b] (-1 for a request whose labels are invalid, which also sets ERR_TAU),
    alpha, margin and entropy [b, gamma] (step order; alpha 0 and margin / entropy NaN past
    L or for an invalid request) and the error word."""
    dl = np.asarray(draft_logits)
    labels = np.asarray(labels)
    b, B, V = dl.shape
    khat = np.full(b, -1.0)
    alpha = np.zeros((b, gamma))
    margin = np.full((b, gamma), np.nan)
    entropy = np.full((b, gamma), np.nan)
    err = 0
    for r in (range(b) if requests is None else requests):
        order = _order_from_labels(labels[r], B)
        if order is None:
            err |= ERR_TAU
            continue
        for i, k in enumerate(order[:gamma]):
            margin[r, i], entropy[r, i] = draft_confidence(dl[r, k], temperature)
            if mode == KHAT_MARGIN:
                alpha[r, i] = 1.0 if margin[r, i] >= tau_margin else 0.0
            else:
                alpha[r, i] = math.exp(-beta * entropy[r, i])
        L = min(gamma, len(order))
        khat[r] = sum(float(np.prod(alpha[r, : k + 1])) for k in range(L))
    return {"khat": khat, "alpha": alpha, "margin": margin, "entropy": entropy, "err": err}
