"""The allocation-free acceptance entry point, simsd_accept_noalloc.

Some callers cannot allocate device memory: plugin hosts that hand the library only its
input and output buffers, and serving runtimes that forbid allocation once they have
started (an allocation can synchronise the device). simsd_accept_noalloc serves them. It
runs the same acceptance kernels as simsd_accept, with the scratch those kernels need in a
fixed array inside the library instead of a caller workspace.

These tests call it through the C interface twice in a row, on different inputs, so that
the second call finds the shared array holding the first call's contents, once with
rejection sampling (T = 1) and once with greedy verification (T = 0; that mode's scratch
plan is a different one). Each call's outputs must equal those of simsd_accept on the same
inputs and those of the fp64 oracle (bit for bit; a mismatch with the oracle is allowed only
at a decision the oracle itself reports as a near-tie). A last test checks that sizes whose
scratch exceeds the array are refused before anything is launched.

The file sorts last, so a run that stops at the first failure has already run every other
test when it gets here.
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


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_noalloc_accept_matches_accept_and_oracle_on_consecutive_calls(T):
    H.ensure_library()
    import diffusion_speculative_verify_gb300 as pkg
    pkg.load_library()
    assert pkg.simsd_accept_noalloc_max_scratch() > 0
    dev = torch.device("cuda")
    w = workloads.WORKLOADS["gqa8b_bf16"].with_(temperature=T)
    assert pkg.simsd_accept_workspace(w.batch, w.B, w.gamma, w.V) <= \
        pkg.simsd_accept_noalloc_max_scratch()
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
                         w.gamma, T, acc["philox_seed"], 0, ref["accepted_len"],
                         ref["out_tokens"], ref["out_pos"], ref["n_commit"], ws, err)
        got = _outputs(b, B, dev)
        err2 = torch.zeros(1, dtype=torch.int32, device=dev)
        pkg.simsd_accept_noalloc(acc["target_logits"], acc["draft_logits"], acc["draft_tokens"],
                                 labels, w.gamma, T, acc["philox_seed"], 0,
                                 got["accepted_len"], got["out_tokens"], got["out_pos"],
                                 got["n_commit"], err2)
        torch.cuda.synchronize()
        assert int(err.item()) == int(err2.item()) == 0
        for k in ref:   # integer outputs of the two entry points: identical
            assert torch.equal(got[k], ref[k]), (call, k)
        inputs = {"target_logits": acc["target_logits"], "draft_logits": acc["draft_logits"],
                  "draft_tokens": acc["draft_tokens"]}
        res = H.oracle_accept(inputs, labels, w.gamma, T, acc["philox_seed"], 0)
        got_np = {k: v.cpu().numpy() for k, v in got.items()}
        assert H.check_accept(res, got_np, list(range(b))) <= 1
        assert (got_np["accepted_len"] >= 0).all()


def test_noalloc_accept_rejects_sizes_beyond_its_scratch():
    H.ensure_library()
    import diffusion_speculative_verify_gb300 as pkg
    lib = pkg.load_library()
    # a plan needing more than the fixed array: many requests x long blocks. The pointers
    # are real device buffers (the argument checks pass) but the size check refuses the
    # call before anything is launched, so nothing reads them.
    b, B, V = 1 << 16, 32, 1000
    assert pkg.simsd_accept_workspace(b, B, B, V) > pkg.simsd_accept_noalloc_max_scratch()
    buf = torch.zeros(1024, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    st = lib.simsd_accept_noalloc(p, p, p, p, b, B, B, V, 1.0, 0, 0, p, p, p, p, p, None)
    assert st == 3   # SIMSD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(buf.abs().sum().item()) == 0
