"""The allocation-free acceptance entry point (simsd_accept_noalloc) against simsd_accept.

simsd_accept_noalloc exists for callers that cannot allocate device memory (plugin hosts
that only hand over input/output buffers, runtimes that forbid allocation after start-up);
it uses a fixed scratch array inside the library instead of a caller workspace, and runs
the two-launch acceptance (stats, then finish), while simsd_accept runs the one-launch
cluster kernel: two implementations of the same arithmetic. On random inputs their results
must be identical, and stay so on consecutive calls that reuse the shared array. This file sorts last so that a stop-at-first-failure run has already
run every other test when it gets here.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _outputs(b, B, dev):
    return {k: torch.full((b,), -7, dtype=torch.int32, device=dev)
            for k in ("accepted_len", "n_commit")} | {
        k: torch.full((b, B), -7, dtype=torch.int32, device=dev) for k in ("out_tokens", "out_pos")}


def test_noalloc_accept_matches_workspace_accept_on_consecutive_calls():
    H.ensure_library()
    import diffusion_speculative_verify_gb300 as pkg
    pkg.load_library()
    assert pkg.simsd_accept_noalloc_max_scratch() > 0
    dev = torch.device("cuda")
    w = workloads.WORKLOADS["gqa8b_bf16"]
    for call, seed in enumerate((5, 6)):   # two calls in a row, different inputs
        lay = workloads.make_layout_inputs(w, seed=seed)
        acc = workloads.make_accept_inputs(w, seed=seed, device=dev)
        b, B = lay["tau"].shape
        pos = torch.empty(b, 2 * B, dtype=torch.int32, device=dev)
        labels = torch.empty(b, 2 * B, dtype=torch.uint8, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        pkg.simsd_build_layout(lay["tau"].to(dev), lay["prompt_len"].to(dev), pos, labels, err)
        ref = _outputs(b, B, dev)
        ws = torch.zeros(pkg.simsd_accept_workspace(b, B, w.gamma, w.V), dtype=torch.uint8,
                         device=dev)
        pkg.simsd_accept(acc["target_logits"], acc["draft_logits"], acc["draft_tokens"], labels,
                         w.gamma, w.temperature, acc["philox_seed"], 0, ref["accepted_len"],
                         ref["out_tokens"], ref["out_pos"], ref["n_commit"], ws, err)
        got = _outputs(b, B, dev)
        err2 = torch.zeros(1, dtype=torch.int32, device=dev)
        pkg.simsd_accept_noalloc(acc["target_logits"], acc["draft_logits"], acc["draft_tokens"],
                                 labels, w.gamma, w.temperature, acc["philox_seed"], 0,
                                 got["accepted_len"], got["out_tokens"], got["out_pos"],
                                 got["n_commit"], err2)
        torch.cuda.synchronize()
        for k in ref:   # integer outputs: identical
            assert torch.equal(got[k], ref[k]), (call, k)
        assert int(err.item()) == int(err2.item()) == 0
        assert (ref["accepted_len"] >= 0).all()


def test_noalloc_accept_rejects_sizes_beyond_its_scratch():
    H.ensure_library()
    import diffusion_speculative_verify_gb300 as pkg
    lib = pkg.load_library()
    # a plan needing more than the fixed array: many requests x long blocks
    b, B, V = 1 << 16, 32, 1000
    assert pkg.simsd_accept_workspace(b, B, B, V) > pkg.simsd_accept_noalloc_max_scratch()
    st = lib.simsd_accept_noalloc(None, None, None, None, b, B, B, V, 1.0, 0, 0,
                                  None, None, None, None, None, None)
    assert st == 3   # SIMSD_ERR_WORKSPACE, nothing launched
