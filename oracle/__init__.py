"""Float64 CPU oracle for the DCOCO hot path -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never uses it.
"""
from .dcoco import (LN_EPS, canonical, candidate_repr, cycle, cycle_lm, layer_norm, lm_head_topk,  # noqa: F401
                    lm_logits, pair_state,
                    residual_draw, select, select_discounted, silu, topk, transition_scores, verify_greedy,
                    verify_speculative, verify_stochastic)
