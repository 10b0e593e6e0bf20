"""fp64 CPU oracle of the SimSD verification step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. It is independent of the CUDA library: the two share no
code, and neither imports the other.
"""
from .simsd import (ERR_PROMPT_LEN, ERR_TAU, ERR_TOKEN, INVALID_LABEL, KHAT_ENTROPY,  # noqa: F401
                    KHAT_MARGIN, SEG_DATA, SEG_MASK, accept, accept_coupled, build_layout,
                    coupled_choice, draft_confidence, expected_prefix, greedy_choice, rope,
                    softmax, temporal_causal_mask, verify_attention)
from . import philox  # noqa: F401
