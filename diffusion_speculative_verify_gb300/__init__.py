"""GB300-native SimSD single-forward speculative verification (sm_103a).

Python side of the C library ``libsimsd.so``: the binding functions carry the C names
(``simsd_build_layout``, ``simsd_verify_attention``, ``simsd_accept``, workspace queries)
and ``VerifyStep`` owns the buffers of one step and issues the three calls on a stream.
PyTorch only supplies device memory and streams.
"""
from __future__ import annotations

import torch

from ._binding import (CACHE_HND, CACHE_NHD, DEVERR_PROMPT_LEN, DEVERR_TAU,  # noqa: F401
                       DEVERR_BOUNDS, DEVERR_TIMEOUT, DEVERR_TOKEN, EXPORTED, KHAT_ENTROPY, KHAT_MARGIN,
                       LAYOUT_PHYSICAL_POSITIONS, LIB_PATH, AttnParams,
                       SimsdError, load_library, make_attn_params, simsd_accept, simsd_accept_coupled,
                       simsd_accept_coupled_ex, simsd_accept_ex, simsd_accept_noalloc, simsd_accept_noalloc_max_scratch,
                       simsd_accept_workspace, simsd_build_layout, simsd_expected_prefix,
                       simsd_expected_prefix_workspace, simsd_last_cuda_error, simsd_status_str,
                       simsd_verify_attention, simsd_verify_attention_workspace,
                       simsd_version)

__all__ = ["VerifyStep", "simsd_build_layout", "simsd_verify_attention", "simsd_accept",
           "simsd_accept_coupled", "simsd_accept_ex", "simsd_accept_coupled_ex",
           "simsd_expected_prefix", "simsd_expected_prefix_workspace",
           "simsd_verify_attention_workspace", "simsd_accept_workspace", "make_attn_params",
           "load_library", "SimsdError"]


class VerifyStep:
    """One verification step (layout -> verify attention -> accept) over fixed inputs.

    ``inputs`` holds device tensors: tau, prompt_len, q, k_resp, v_resp, k_cache, v_cache,
    cache_start (int64 [b]), target_logits, draft_logits (both fp32 or both bf16),
    draft_tokens. With ``khat_mode`` set (KHAT_MARGIN or KHAT_ENTROPY) the step also
    estimates every request's expected accepted-prefix length from the draft logits
    (``khat``, ``alpha``) between the layout and the attention. Outputs live in
    this object (``pos_ids``, ``labels``, ``out``, ``lse``, ``accepted_len``, ``n_commit``,
    ``out_tokens``, ``out_pos``, ``dev_err``) and are overwritten by every ``run``.
    """

    def __init__(self, inputs: dict, gamma: int, rope_theta: float, temperature: float = 1.0,
                 cache_layout: str = "NHD", softmax_scale: float = 0.0, with_lse: bool = True,
                 philox_seed: int = 0, philox_offset: int = 0, coupled: bool = False,
                 khat_mode=None, tau_margin: float = 0.5, beta: float = 1.0,
                 khat_temperature: float = 1.0, aligned_rope: bool = True):
        load_library()
        dev = inputs["q"].device
        b, twoB, Hq, D = inputs["q"].shape
        B = twoB // 2
        V = inputs["target_logits"].shape[-1]
        self.b, self.B, self.V, self.gamma = b, B, V, gamma
        self.temperature = temperature
        self.coupled = coupled  # coupled-noise verification instead of rejection sampling
        self.seed, self.offset = philox_seed, philox_offset
        self.inputs = inputs
        self.pos_ids = torch.empty(b, twoB, dtype=torch.int32, device=dev)
        self.labels = torch.empty(b, twoB, dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(inputs["q"])
        self.lse = torch.empty(b, twoB, Hq, dtype=torch.float32, device=dev) if with_lse else None
        self.accepted_len = torch.empty(b, dtype=torch.int32, device=dev)
        self.n_commit = torch.empty(b, dtype=torch.int32, device=dev)
        self.out_tokens = torch.empty(b, B, dtype=torch.int32, device=dev)
        self.out_pos = torch.empty(b, B, dtype=torch.int32, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.params = make_attn_params(
            inputs["q"], inputs["k_resp"], inputs["v_resp"], inputs["k_cache"],
            inputs["v_cache"], inputs["cache_start"], inputs["prompt_len"], self.pos_ids,
            self.labels, self.out, self.dev_err, rope_theta, softmax_scale, self.lse,
            cache_layout)
        ws_attn = simsd_verify_attention_workspace(self.params)
        if ws_attn == 0:
            raise SimsdError(1, "simsd_verify_attention_workspace")
        self.ws_attn = torch.empty(ws_attn, dtype=torch.uint8, device=dev)
        ws_acc = simsd_accept_workspace(b, B, gamma, V)
        if ws_acc == 0:
            raise SimsdError(1, "simsd_accept_workspace")
        self.ws_accept = torch.empty(ws_acc, dtype=torch.uint8, device=dev)
        self.khat_mode = khat_mode
        # aligned_rope=False: the mask slots keep their physical positions (ablation)
        self.layout_flags = 0 if aligned_rope else LAYOUT_PHYSICAL_POSITIONS
        if khat_mode is not None:
            self.khat_args = (khat_temperature, int(khat_mode), tau_margin, beta)
            self.khat = torch.empty(b, dtype=torch.float32, device=dev)
            self.alpha = torch.empty(b, gamma, dtype=torch.float32, device=dev)
            ws_k = simsd_expected_prefix_workspace(b, B, gamma, V)
            if ws_k == 0:
                raise SimsdError(1, "simsd_expected_prefix_workspace")
            self.ws_khat = torch.empty(ws_k, dtype=torch.uint8, device=dev)

    def layout(self, stream=None):
        simsd_build_layout(self.inputs["tau"], self.inputs["prompt_len"], self.pos_ids,
                           self.labels, self.dev_err, stream, self.layout_flags)

    def expected_prefix(self, stream=None):
        simsd_expected_prefix(self.inputs["draft_logits"], self.labels, self.gamma,
                              *self.khat_args, self.khat, self.alpha, self.ws_khat,
                              self.dev_err, stream)

    def attention(self, stream=None):
        simsd_verify_attention(self.params, self.ws_attn, stream)

    def accept(self, stream=None):
        i = self.inputs
        if self.coupled:
            simsd_accept_coupled_ex(i["target_logits"], i["draft_tokens"], self.labels, self.pos_ids,
                                    self.gamma, self.temperature, self.seed, self.offset,
                                    self.accepted_len, self.out_tokens, self.out_pos,
                                    self.n_commit, self.ws_accept, self.dev_err, stream)
            return
        simsd_accept_ex(i["target_logits"], i["draft_logits"], i["draft_tokens"], self.labels,
                        self.gamma, self.temperature, self.seed, self.offset,
                        self.accepted_len, self.out_tokens, self.out_pos, self.n_commit,
                        self.ws_accept, self.dev_err, stream)

    def run(self, stream=None):
        self.layout(stream)
        if self.khat_mode is not None:
            self.expected_prefix(stream)
        self.attention(stream)
        self.accept(stream)
