"""Planted mistakes in the oracle (on the CPU) must trip at least one pin.

Each case swaps a piece of the oracle for a plausible wrong variant and runs the
pin that is meant to catch it.
"""
import numpy as np
import pytest

import oracle
import oracle.dcoco as od
import test_oracle_pins as pins


def _unbiased_ln(x, eps=od.LN_EPS):
    mu = x.mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(x.var(axis=-1, ddof=1, keepdims=True) + eps)


def _eps_outside_ln(x, eps=od.LN_EPS):
    mu = x.mean(axis=-1, keepdims=True)
    return (x - mu) / (np.sqrt(((x - mu) ** 2).mean(axis=-1, keepdims=True)) + eps)


def _argmax_last(x):
    y = od.canonical(x)
    return int(len(y) - 1 - np.argmax(y[::-1]))


def _swap(w, a, b):
    w = dict(w)
    w[a], w[b] = w[b], w[a]
    return w


ORIG_TS = od.transition_scores
ORIG_CR = od.candidate_repr
ORIG_TOPK = od.topk


def _ts_swapped_logit_weights(z, s, vals, w):
    return ORIG_TS(z, s, vals, _swap(w, "u_a", "u_b"))


def _ts_swapped_UV(z, s, vals, w):
    return ORIG_TS(z, s, vals, _swap(w, "U", "V"))


def _cr_concat_order(ids, emb, h, w):
    w = dict(w)
    r = w["W_f"].shape[0]
    w["W_f"] = np.hstack([w["W_f"][:, r:], w["W_f"][:, :r]])
    return ORIG_CR(ids, emb, h, w)


def _cr_transposed_gather(ids, emb, h, w):
    # gathers by candidate position instead of token id
    pos = np.broadcast_to(np.arange(ids.shape[-1]), ids.shape)
    return ORIG_CR(pos, emb, h, w)


def _topk_ties_high(logits, K):
    x = od.canonical(np.asarray(logits, dtype=np.float64))
    order = np.argsort(-x[..., ::-1], axis=-1, kind="stable")[..., :K]
    order = x.shape[-1] - 1 - order
    return np.take_along_axis(x, order, axis=-1), order


def _ts_dropped_b1(z, s, vals, w):
    w = dict(w)
    w["b1"] = np.zeros_like(w["b1"])
    return ORIG_TS(z, s, vals, w)


def _ts_flipped_correction(z, s, vals, w):
    # S = l - Delta instead of l + Delta
    base = np.broadcast_to(vals[:, 1:, None, :], (z.shape[0], z.shape[1] - 1, z.shape[2], z.shape[2]))
    return 2 * base - ORIG_TS(z, s, vals, w)


def _select_transposed(S, vals, ids):
    # walks the column S_p(., k_p) instead of the row S_p(k_p, .)
    return ORIG_SELECT(np.swapaxes(S, -1, -2), vals, ids)


def _select_first_slot_assumed_zero(S, vals, ids):
    # takes candidate 0 for slot 0 instead of the argmax of the drafter's logits
    v = np.array(vals, dtype=np.float64, copy=True)
    v[:, 0, :] = 0.0
    v[:, 0, 0] = 1.0
    return ORIG_SELECT(S, v, ids)


def _verify_greedy_commits_draft(draft, t):
    out = ORIG_VG(draft, t)
    com = out["committed"].copy()
    for n, A in enumerate(out["accept_len"]):
        if A < draft.shape[1]:
            com[n, A] = draft[n, A]
    return {**out, "committed": com}


def _verify_stochastic_non_strict(draft, q, u):
    # accepts when u == q(y)
    return ORIG_VS(draft, q, np.nextafter(u, -np.inf))


def _residual_keeps_draft(q, u, exclude):
    return ORIG_RD(q, u, -1)


ORIG_SELECT = od.select
ORIG_SD = od.select_discounted


def _sd_wrong_power(S, vals, ids, lam):
    # weights lam^p instead of lam^(p+1): the first transition is not discounted
    return ORIG_SD(S / lam, vals, ids, lam) if lam != 1.0 else ORIG_SD(S, vals, ids, lam)


def _sd_first_slot_fixed(S, vals, ids, lam):
    # keeps the drafter's top candidate at slot 0 instead of optimising it with the rest
    v = np.array(vals, dtype=np.float64, copy=True)
    top = np.argmax(v[:, 0, :], axis=1)
    v[:, 0, :] = -1e9
    v[np.arange(v.shape[0]), 0, top] = 0.0
    return ORIG_SD(S, v, ids, lam)
ORIG_VG = od.verify_greedy
ORIG_VS = od.verify_stochastic
ORIG_RD = od.residual_draw
ORIG_VSP = od.verify_speculative


def _vsp_ignores_p(draft, p, q, u):
    # accepts on u < q(y), as if the draft were a point mass
    return ORIG_VSP(draft, np.ones_like(np.asarray(p, dtype=np.float64)), q, u)


def _vsp_unclamped_residual(draft, p, q, u):
    # residual q - p without the clamp at zero: negative mass enters the draw
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    N, B = draft.shape
    out = ORIG_VSP(draft, p, q, u)
    for n in range(N):
        A = int(out["accept_len"][n])
        if A < B:
            out["committed"][n, A] = od._inverse_cdf(q[n, A] - p[n, A], u[n, A, 1], int(draft[n, A]))[0]
    return out

def _lm_transposed(h, W_lm):
    return np.asarray(h, dtype=np.float64) @ np.asarray(W_lm, dtype=np.float64)


def _lm_drops_last_unit(h, W_lm):
    h = np.asarray(h, dtype=np.float64)
    W_lm = np.asarray(W_lm, dtype=np.float64)
    return h[..., :-1] @ W_lm[:, :-1].T


CASES = [
    ("layer_norm", _unbiased_ln, pins.test_layer_norm_spike_closed_form),
    ("layer_norm", _eps_outside_ln, pins.test_layer_norm_spike_closed_form),
    ("_argmax_first", _argmax_last, pins.test_walk_ties_go_to_lower_index),
    ("transition_scores", _ts_swapped_logit_weights,
     lambda: pins.test_scores_single_term_closed_form("u_a")),
    ("transition_scores", _ts_swapped_UV, lambda: pins.test_scores_single_term_closed_form("U")),
    ("candidate_repr", _cr_concat_order, pins.test_candidate_repr_hidden_path_and_concat_order),
    ("candidate_repr", _cr_transposed_gather, pins.test_candidate_repr_embedding_path),
    ("topk", _topk_ties_high, pins.test_topk_all_equal_and_k_equals_v),
    ("transition_scores", _ts_dropped_b1, pins.test_scores_bias_only_closed_form),
    ("transition_scores", _ts_flipped_correction, pins.test_scores_bias_only_closed_form),
    ("select", _select_transposed, lambda: [pins.test_walk_matches_brute_force(i) for i in range(8)]),
    ("select", _select_first_slot_assumed_zero, lambda: [pins.test_walk_matches_brute_force(i) for i in range(8)]),
    ("verify_greedy", _verify_greedy_commits_draft, pins.test_greedy_verify_closed_form),
    ("verify_stochastic", _verify_stochastic_non_strict, pins.test_stochastic_verify_hand_cases),
    ("residual_draw", _residual_keeps_draft, pins.test_stochastic_verify_hand_cases),
    ("verify_speculative", _vsp_ignores_p, pins.test_speculative_hand_cases),
    ("verify_speculative", _vsp_unclamped_residual, pins.test_speculative_hand_cases),
    ("select_discounted", _sd_wrong_power,
     lambda: [pins.test_discounted_path_matches_brute_force(i, 0.5) for i in range(10)]),
    ("lm_logits", _lm_transposed, lambda: [pins.test_lm_head_topk_matches_scalar_loops(i) for i in range(5)]),
    ("lm_logits", _lm_drops_last_unit, lambda: [pins.test_lm_head_topk_matches_scalar_loops(i) for i in range(5)]),
    ("select_discounted", _sd_first_slot_fixed,
     lambda: [pins.test_discounted_path_matches_brute_force(i, 1.0) for i in range(10)]),
]


@pytest.mark.parametrize("name,bad,pin", CASES, ids=[f"{c[0]}:{c[1].__name__}" for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, bad, pin):
    monkeypatch.setattr(od, name, bad)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, bad)
    with pytest.raises(AssertionError):
        pin()
