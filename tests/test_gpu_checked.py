"""The bounds-checked build (libsimsd_checked.so, compiled with SIMSD_CHECKED).

A memory checker cannot run on these GPUs, so the library has a build in which every kernel
checks the index of each global access against the extent of the array it addresses and
reports a violation in the device error word (SIMSD_DEVERR_BOUNDS) instead of making the
access. These tests swap that build in under the same Python binding and run small cases of
every entry point (layout, bf16 attention with one and two CTAs per pair and with pairs
split across CTAs or CTA pairs, NHD and HND caches, fp32 attention, acceptance at T = 1 and T = 0 with
fp32 and bf16 logits and an odd vocabulary, coupled-noise verification, the
expected-prefix estimate, the allocation-free acceptance entry): each must raise no error
bit and still match the fp64 oracle. A last case checks that the checks fire: a request
whose cache_start points past the end of the cache (an error in device data that the host
cannot see) gives SIMSD_DEVERR_BOUNDS, and the rows of the other requests stay right.
"""
import contextlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import helpers as H

pytestmark = pytest.mark.gpu

MEDIUM = workloads.Workload(
    name="medium_bf16", dtype="bf16", batch=4, Hq=8, Hkv=2, D=128, B=8, prompt_len=None,
    prompt_len_range=(0, 1), rope_theta=1e6, gamma=8, V=4096)


@contextlib.contextmanager
def _checked_library():
    from diffusion_speculative_verify_gb300 import _binding, _build
    path = _build.build(checked=True)
    saved = _binding._lib
    _binding._lib = None
    try:
        yield _binding.load_library(path)
    finally:
        _binding._lib = saved


def _run(w, inputs, meta, **kw):
    import diffusion_speculative_verify_gb300 as pkg
    st = pkg.VerifyStep(inputs, gamma=w.gamma, rope_theta=w.rope_theta, temperature=w.temperature,
                        cache_layout=meta["cache_layout"], with_lse=True,
                        philox_seed=meta["philox_seed"], philox_offset=meta["philox_offset"], **kw)
    st.run()
    torch.cuda.synchronize()
    return st


def _attention_matches(w, inputs, meta, st, requests=None):
    ref, _ = H.oracle_attention(inputs, st.pos_ids, st.labels, w.rope_theta, meta["cache_layout"],
                                requests)
    reqs = list(range(w.batch)) if requests is None else list(requests)
    H.compare_attention(H.to_np(st.out)[reqs], ref[reqs], w.torch_dtype)


def _accept_matches(w, inputs, meta, st):
    res = H.oracle_accept(inputs, st.labels, w.gamma, w.temperature, meta["philox_seed"],
                          meta["philox_offset"])
    got = {k: getattr(st, k).cpu().numpy() for k in ("accepted_len", "n_commit", "out_tokens", "out_pos")}
    assert H.check_accept(res, got, list(range(w.batch))) <= 1


CASES = {
    # name: (workload, prompt lengths, cache layout)
    "one_cta_per_pair_nhd": (MEDIUM, [0, 61, 128, 1037], "NHD"),
    "one_cta_per_pair_hnd": (MEDIUM, [0, 61, 128, 1037], "HND"),
    "two_ctas_per_pair": (MEDIUM.with_(Hq=6, Hkv=2, B=32, gamma=32), [0, 61, 128, 1037], "NHD"),
    "split_pairs": (MEDIUM.with_(Hq=6, Hkv=2, B=16, gamma=16), [20000, 61, 128, 9000], "NHD"),
    # 256-row pairs on CTA pairs, split across 2-CTA clusters and merged in the kernel
    "split_pairs_two_ctas_hnd": (MEDIUM.with_(Hq=8, Hkv=1, B=16, gamma=16), [20000, 61, 128, 9000], "HND"),
    "fp32": (workloads.WORKLOADS["tiny_fp32"].with_(batch=3, B=8, gamma=8), [0, 33, 300], "NHD"),
}


@pytest.mark.parametrize("case", list(CASES))
def test_checked_build_attention_layout_and_estimate_raise_nothing(case):
    import diffusion_speculative_verify_gb300 as pkg
    w, plen, layout = CASES[case]
    inputs, meta = H.make_case(w, seed=31, prompt_len=plen, cache_layout=layout)
    with _checked_library():
        st = _run(w, inputs, meta, khat_mode=pkg.KHAT_ENTROPY, beta=1.0)
        err = int(st.dev_err.item())
        assert err == 0, err
        _attention_matches(w, inputs, meta, st)
        _accept_matches(w, inputs, meta, st)
        kref = oracle.expected_prefix(H.to_np(inputs["draft_logits"]), st.labels.cpu().numpy(),
                                      w.gamma, 1.0, oracle.KHAT_ENTROPY, beta=1.0)["khat"]
        assert np.abs(st.khat.cpu().numpy() - kref).max() <= w.gamma * (w.gamma + 1) / 2 * 2e-5


@pytest.mark.parametrize("T,ldt,V,coupled", [(1.0, "fp32", 5001, False), (1.0, "bf16", 4096, False),
                                             (0.0, "fp32", 4096, False), (0.0, "bf16", 5001, False),
                                             (1.0, "fp32", 4096, True)])
def test_checked_build_acceptance_raises_nothing(T, ldt, V, coupled):
    w = workloads.WORKLOADS["gqa8b_bf16"].with_(batch=6, V=V, temperature=T, logit_dtype=ldt)
    inputs, meta = H.make_case(w, seed=37)
    with _checked_library():
        st = _run(w, inputs, meta, coupled=coupled)
        assert int(st.dev_err.item()) == 0
        f64 = H.to_np
        if coupled:
            res = oracle.accept_coupled(f64(inputs["target_logits"]), f64(inputs["draft_tokens"]),
                                        st.labels.cpu().numpy(), st.pos_ids.cpu().numpy(), w.gamma, T,
                                        meta["philox_seed"], meta["philox_offset"])
        else:
            res = oracle.accept(f64(inputs["target_logits"]), f64(inputs["draft_logits"]),
                                f64(inputs["draft_tokens"]), st.labels.cpu().numpy(), w.gamma, T,
                                meta["philox_seed"], meta["philox_offset"])
        got = {k: getattr(st, k).cpu().numpy() for k in ("accepted_len", "n_commit", "out_tokens", "out_pos")}
        if not coupled:
            assert H.check_accept(res, got, list(range(w.batch))) <= 1
            return
        for r in range(w.batch):  # coupled keys: equal unless the oracle's two best are near-tied
            if not all(np.array_equal(got[k][r], res[k][r]) for k in got):
                assert min(res["diag"][r]["key_gaps"]) < 1e-4, r


def test_checked_build_noalloc_acceptance_raises_nothing():
    import diffusion_speculative_verify_gb300 as pkg
    w = workloads.WORKLOADS["gqa8b_bf16"].with_(batch=6, V=4096)
    inputs, meta = H.make_case(w, seed=41)
    with _checked_library():
        st = _run(w, inputs, meta)
        b, B = st.labels.shape[0], w.B
        out = {k: torch.full((b,), -7, dtype=torch.int32, device="cuda") for k in ("accepted_len", "n_commit")}
        out |= {k: torch.full((b, B), -7, dtype=torch.int32, device="cuda") for k in ("out_tokens", "out_pos")}
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkg.simsd_accept_noalloc(inputs["target_logits"], inputs["draft_logits"], inputs["draft_tokens"],
                                 st.labels, w.gamma, w.temperature, meta["philox_seed"], meta["philox_offset"],
                                 out["accepted_len"], out["out_tokens"], out["out_pos"], out["n_commit"], err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for k in out:
            assert torch.equal(out[k], getattr(st, k)), k


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_checked_build_reports_a_cache_start_past_the_cache(dtype):
    """Request 1's cache_start points beyond the packed cache: the checked kernels skip
    those rows and raise SIMSD_DEVERR_BOUNDS; the other requests' rows are still right."""
    import diffusion_speculative_verify_gb300 as pkg
    w = MEDIUM if dtype == "bf16" else workloads.WORKLOADS["tiny_fp32"].with_(batch=3, B=8, gamma=8)
    plen = [0, 61, 128, 1037][: w.batch]
    inputs, meta = H.make_case(w, seed=43, prompt_len=plen)
    tokens = inputs["k_cache"].shape[0]
    with _checked_library():
        bad = inputs["cache_start"].clone()
        bad[1] = tokens + 4096
        good_start = inputs["cache_start"]
        inputs["cache_start"] = bad
        st = _run(w, inputs, meta)
        err = int(st.dev_err.item())
        assert err & pkg.DEVERR_BOUNDS, err
        inputs["cache_start"] = good_start
        others = [r for r in range(w.batch) if r != 1]
        _attention_matches(w, inputs, meta, st, requests=others)
