"""Pins of the float64 oracle against what the pages and the mathematics fix.

Nothing here re-types the oracle's formulas: each check is a brute force, a closed
form evaluated with scalar arithmetic, an invariant, or a value the pages print.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import workloads as wl
from conftest import GOLDEN

# ---------------------------------------------------------------------------
# top-K: brute force
# ---------------------------------------------------------------------------


def _rank_value(x):
    """Value used for ranking: NaN is lowest, -0 == +0."""
    return -math.inf if math.isnan(x) else x + 0.0


def brute_topk(row, K):
    taken, out = set(), []
    for _ in range(K):
        best = None
        for i, x in enumerate(row):
            if i in taken:
                continue
            if best is None or _rank_value(x) > _rank_value(row[best]):
                best = i  # strict '>' keeps the lowest index among equals
        taken.add(best)
        out.append(best)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force_random(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(1, 64))
    K = int(rng.integers(1, V + 1))
    row = np.round(rng.normal(0, 2, V), 1)  # rounding to 0.1 makes ties common
    vals, ids = oracle.topk(row[None], K)
    want = brute_topk(list(row), K)
    assert list(ids[0]) == want
    assert list(vals[0]) == [_rank_value(row[i]) for i in want]


def test_topk_special_values():
    row = [0.0, -0.0, math.inf, -math.inf, math.nan, 1.0, 1.0, -math.inf, math.nan, -0.0, math.inf]
    for K in range(1, len(row) + 1):
        vals, ids = oracle.topk(np.array(row)[None], K)
        assert list(ids[0]) == brute_topk(row, K)
    vals, ids = oracle.topk(np.array(row)[None], len(row))
    # +inf ids 2, 10; 1.0 ids 5, 6; zeros 0, 1, 9 (sign ignored); -inf and NaN tie: 3, 4, 7, 8
    assert list(ids[0]) == [2, 10, 5, 6, 0, 1, 9, 3, 4, 7, 8]
    assert not np.signbit(vals[0][4:7]).any()          # -0 reported as +0
    assert np.all(vals[0][7:] == -math.inf)             # NaN reported as -inf


def test_topk_all_equal_and_k_equals_v():
    row = np.full(40, 3.5)
    _, ids = oracle.topk(row[None], 7)
    assert list(ids[0]) == list(range(7))
    _, ids = oracle.topk(row[None], 40)
    assert list(ids[0]) == list(range(40))


def test_topk_batched_rows_independent():
    rng = np.random.default_rng(11)
    x = np.round(rng.normal(0, 1, (2, 3, 30)), 1)
    vals, ids = oracle.topk(x, 5)
    for n in range(2):
        for i in range(3):
            assert list(ids[n, i]) == brute_topk(list(x[n, i]), 5)


# ---------------------------------------------------------------------------
# Drafter output projection + top-K: scalar loops, one-hot rows, ties
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("seed", range(5))
def test_lm_head_topk_matches_scalar_loops(seed):
    """Each logit as an explicit scalar sum over the hidden units, then brute-force top-K.
    Square shapes (V == d) catch a transposed projection; dyadic values keep every sum exact."""
    rng = np.random.default_rng(100 + seed)
    rows, d = int(rng.integers(1, 4)), int(rng.integers(2, 9))
    V = d if seed % 2 == 0 else int(rng.integers(d + 1, 3 * d + 2))
    K = int(rng.integers(1, V + 1))
    h = rng.integers(-4, 5, (rows, d)) / 4.0
    W = rng.integers(-4, 5, (V, d)) / 8.0
    vals, ids = oracle.lm_head_topk(h, W, K)
    for i in range(rows):
        row = []
        for v in range(V):
            acc = 0.0
            for k in range(d):
                acc += float(h[i, k]) * float(W[v, k])
            row.append(acc)
        want = brute_topk(row, K)
        assert list(ids[i]) == want
        assert list(vals[i]) == [row[v] for v in want]


def test_lm_head_topk_one_hot_rows_select_hidden_units():
    """Row v of W_lm = c_v e_{pi(v)} (c_v > 0, V <= d) makes logit v = c_v h[pi(v)]: the
    top-K follows the scaled hidden units through the permutation."""
    rng = np.random.default_rng(7)
    d, V, K = 12, 9, 4
    pi = rng.permutation(d)[:V]
    c = rng.integers(1, 4, V).astype(np.float64)
    W = np.zeros((V, d))
    W[np.arange(V), pi] = c
    h = rng.integers(-8, 9, (2, d)).astype(np.float64)
    vals, ids = oracle.lm_head_topk(h, W, K)
    for i in range(2):
        scaled = [c[v] * h[i, pi[v]] for v in range(V)]
        assert list(ids[i]) == brute_topk(scaled, K)
        assert list(vals[i]) == sorted(scaled, reverse=True)[:K]


def test_lm_head_topk_duplicate_rows_tie_to_lower_id():
    """Tokens with identical output rows have equal logits; the lower id ranks first."""
    rng = np.random.default_rng(3)
    base = rng.integers(-3, 4, (4, 6)).astype(np.float64)
    W = np.concatenate([base, base[::-1]])   # ids 0..3 and 7..4 repeat the same rows
    h = rng.integers(-3, 4, (1, 6)).astype(np.float64)
    _, ids = oracle.lm_head_topk(h, W, 8)
    logit = {v: float(h[0] @ W[v]) for v in range(8)}
    assert list(ids[0]) == brute_topk([logit[v] for v in range(8)], 8)
    for a, b in zip(ids[0][:-1], ids[0][1:]):
        if logit[a] == logit[b]:
            assert a < b


# ---------------------------------------------------------------------------
# LayerNorm and SiLU: closed forms and invariants
# ---------------------------------------------------------------------------


def ln_single_spike(x0, r, eps=1e-5):
    """LN of [x0, 0, ..., 0] (length r): mean x0/r, biased variance x0^2 (r-1)/r^2."""
    var = x0 * x0 * (r - 1) / (r * r)
    den = math.sqrt(var + eps)
    return [x0 * (r - 1) / r / den] + [-(x0 / r) / den] * (r - 1)


def test_layer_norm_spike_closed_form():
    for x0, r in ((3.0, 4), (-0.02, 32), (1e-3, 8)):
        x = np.zeros(r)
        x[0] = x0
        np.testing.assert_allclose(oracle.layer_norm(x), ln_single_spike(x0, r), rtol=1e-12, atol=1e-15)


def test_layer_norm_invariants():
    rng = np.random.default_rng(3)
    x = rng.normal(0.7, 0.05, (5, 256))
    y = oracle.layer_norm(x)
    var = x.var(axis=1)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=1), var / (var + oracle.LN_EPS), rtol=1e-10)


def test_silu_values():
    s = oracle.silu(np.array([0.0, 1.0, -1.0, 40.0, -40.0, 2.5]))
    want = [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.exp(1)), 40.0, -40 * math.exp(-40) / (1 + math.exp(-40)),
            2.5 / (1 + math.exp(-2.5))]
    np.testing.assert_allclose(s, want, rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([-1000.0]))[0] == 0.0


# ---------------------------------------------------------------------------
# Candidate representation and pair state: structured weights
# ---------------------------------------------------------------------------


def _zero_weights(r, H, d, E):
    return {"W_e": np.zeros((r, E)), "W_h": np.zeros((r, d)), "W_f": np.zeros((r, 2 * r)),
            "W_pair": np.zeros((r, 2 * d)), "U": np.zeros((H, r)), "V": np.zeros((H, r)),
            "W": np.zeros((H, r)), "u_a": np.zeros(H), "u_b": np.zeros(H), "b1": np.zeros(H),
            "w2": np.zeros(H), "b2": np.zeros(1)}


def test_candidate_repr_embedding_path():
    """W_e with one entry w at (row 0, column j): b_ik = LN([w Emb[c_ik, j], 0, ...])."""
    rng = np.random.default_rng(5)
    N, B, K, V, E, d, r, H = 2, 3, 2, 50, 12, 6, 8, 4
    emb = rng.normal(0, 1, (V, E))
    ids = rng.integers(0, V, (N, B, K))
    h = rng.normal(0, 1, (N, B, d))
    w = _zero_weights(r, H, d, E)
    j, wv = 7, 0.37
    w["W_e"][0, j] = wv
    out = oracle.candidate_repr(ids, emb, h, w)
    for n, i, k in itertools.product(range(N), range(B), range(K)):
        x0 = wv * emb[ids[n, i, k], j]
        np.testing.assert_allclose(out["b"][n, i, k], ln_single_spike(x0, r), rtol=1e-10, atol=1e-12)
    # W_h = 0: g is LN of zeros = 0; W_f = 0: z = SiLU(0) = 0
    assert np.all(out["g"] == 0) and np.all(out["z"] == 0)


def test_candidate_repr_hidden_path_and_concat_order():
    rng = np.random.default_rng(6)
    N, B, K, V, E, d, r, H = 1, 4, 3, 20, 5, 9, 6, 4
    emb = rng.normal(0, 1, (V, E))
    ids = rng.integers(0, V, (N, B, K))
    h = rng.normal(0, 1, (N, B, d))
    w = _zero_weights(r, H, d, E)
    w["W_e"] = rng.normal(0, 1, (r, E))
    w["W_h"][2, 4] = -1.3                      # g_i = LN of a spike at feature 2
    # W_f = [I, 0]: z = SiLU(b);   W_f = [0, I]: z = SiLU(g) for every candidate
    w["W_f"] = np.hstack([np.eye(r), np.zeros((r, r))])
    out = oracle.candidate_repr(ids, emb, h, w)
    b = out["b"]
    np.testing.assert_allclose(out["z"], b / (1 + np.exp(-b)), rtol=1e-13)
    for n, i in itertools.product(range(N), range(B)):
        spike = ln_single_spike(-1.3 * h[n, i, 4], r)
        want = np.roll(spike, 2)               # the spike sits at feature 2
        np.testing.assert_allclose(out["g"][n, i], want, rtol=1e-10, atol=1e-12)
    w["W_f"] = np.hstack([np.zeros((r, r)), np.eye(r)])
    out = oracle.candidate_repr(ids, emb, h, w)
    for n, i, k in itertools.product(range(N), range(B), range(K)):
        g = out["g"][n, i]
        np.testing.assert_allclose(out["z"][n, i, k], [x / (1 + math.exp(-x)) for x in g], rtol=1e-13)


def test_pair_state_blocks():
    rng = np.random.default_rng(7)
    N, B, d, r = 2, 5, 4, 4
    h = rng.normal(0, 1, (N, B, d))
    w = {"W_pair": np.hstack([np.eye(d), np.zeros((d, d))])}
    s = oracle.pair_state(h, w)
    assert s.shape == (N, B - 1, r)
    np.testing.assert_array_equal(s, h[:, :-1])
    w = {"W_pair": np.hstack([np.zeros((d, d)), np.eye(d)])}
    np.testing.assert_array_equal(oracle.pair_state(h, w), h[:, 1:])
    w = {"W_pair": np.zeros((3, 2 * d))}
    w["W_pair"][1, d + 2] = 2.0
    s = oracle.pair_state(h, w)
    for n, p in itertools.product(range(N), range(B - 1)):
        assert s[n, p, 1] == 2.0 * h[n, p + 1, 2] and s[n, p, 0] == 0 and s[n, p, 2] == 0


# ---------------------------------------------------------------------------
# Transition scores: zero-output identity and one-term closed forms
# ---------------------------------------------------------------------------

N_, B_, K_, r_, H_ = 2, 4, 3, 5, 6


def _score_inputs(seed=8):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 1, (N_, B_, K_, r_))
    s = rng.normal(0, 1, (N_, B_ - 1, r_))
    vals = rng.normal(0, 2, (N_, B_, K_))
    return rng, z, s, vals


def _sil(x):
    return x / (1 + math.exp(-x))


def test_scores_zero_output_layer_is_drafter_logit():
    """w2 = b2 = 0 (zero-initialised output layer): S_p(a,b) = l_{p+1}(b) exactly."""
    rng, z, s, vals = _score_inputs()
    w = {k: rng.normal(0, 1, v.shape) for k, v in _zero_weights(r_, H_, 1, 1).items()}
    w["w2"][:] = 0
    w["b2"][:] = 0
    S = oracle.transition_scores(z, s, vals, w)
    for n, p, a, b in itertools.product(range(N_), range(B_ - 1), range(K_), range(K_)):
        assert S[n, p, a, b] == vals[n, p + 1, b]


def test_scores_bias_only_closed_form():
    rng, z, s, vals = _score_inputs()
    w = _zero_weights(r_, H_, 1, 1)
    w["b1"] = rng.normal(0, 1, H_)
    w["w2"] = rng.normal(0, 1, H_)
    w["b2"][0] = 0.125
    S = oracle.transition_scores(z, s, vals, w)
    const = sum(w["w2"][h] * _sil(w["b1"][h]) for h in range(H_)) + 0.125
    for n, p, a, b in itertools.product(range(N_), range(B_ - 1), range(K_), range(K_)):
        assert abs(S[n, p, a, b] - (vals[n, p + 1, b] + const)) < 1e-12


@pytest.mark.parametrize("term", ["u_a", "u_b", "U", "V", "W"])
def test_scores_single_term_closed_form(term):
    """One first-layer entry alpha and one output weight beta at hidden unit h0:
    S_p(a,b) = l_{p+1}(b) + beta * SiLU(alpha * x) with x the one input that entry reads."""
    rng, z, s, vals = _score_inputs(9)
    w = _zero_weights(r_, H_, 1, 1)
    h0, j, alpha, beta = 4, 2, 0.8, -1.7
    if term in ("u_a", "u_b"):
        w[term][h0] = alpha
    else:
        w[term][h0, j] = alpha
    w["w2"][h0] = beta
    S = oracle.transition_scores(z, s, vals, w)
    for n, p, a, b in itertools.product(range(N_), range(B_ - 1), range(K_), range(K_)):
        x = {"u_a": vals[n, p, a], "u_b": vals[n, p + 1, b], "U": z[n, p, a, j],
             "V": z[n, p + 1, b, j], "W": s[n, p, j]}[term]
        want = vals[n, p + 1, b] + beta * _sil(alpha * x)
        assert abs(S[n, p, a, b] - want) < 1e-12, (term, n, p, a, b)


# ---------------------------------------------------------------------------
# Prefix-first greedy walk: brute force over all paths
# ---------------------------------------------------------------------------


def brute_walk(S, vals):
    """Prefix-first rule as a search over every path: k_1 is the drafter's top candidate,
    and among all paths the chosen one maximises the sequence
    (S_1(k_1,k_2), -k_2, S_2(k_2,k_3), -k_3, ...) in lexicographic order."""
    B, K = vals.shape
    k1 = max(range(K), key=lambda k: (vals[0, k], -k))
    best, best_key = None, None
    for rest in itertools.product(range(K), repeat=B - 1):
        path = (k1,) + rest
        key = []
        for p in range(B - 1):
            key += [S[p, path[p], path[p + 1]], -path[p + 1]]
        if best_key is None or key > best_key:
            best, best_key = path, key
    return list(best)


@pytest.mark.parametrize("seed", range(8))
def test_walk_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    B, K = int(rng.integers(2, 6)), int(rng.integers(1, 5))
    N = 3
    vals = np.round(rng.normal(0, 1, (N, B, K)), 1)
    S = np.round(rng.normal(0, 1, (N, B - 1, K, K)), 1)   # coarse values: ties happen
    ids = rng.integers(0, 1000, (N, B, K))
    k, tokens = oracle.select(S, vals, ids)
    for n in range(N):
        assert list(k[n]) == brute_walk(S[n], vals[n])
        assert list(tokens[n]) == [ids[n, i, k[n, i]] for i in range(B)]


def test_walk_ties_go_to_lower_index():
    vals = np.array([[[2.0, 2.0, 1.0], [0.0, 0.0, 0.0], [1.0, 3.0, 3.0]]])
    S = np.zeros((1, 2, 3, 3))
    S[0, 1, 0] = [0.5, 0.7, 0.7]
    k, _ = oracle.select(S, vals, np.zeros((1, 3, 3), dtype=np.int64))
    assert list(k[0]) == [0, 0, 1]


def test_walk_with_zero_correction_is_per_slot_argmax():
    rng = np.random.default_rng(12)
    N, B, K = 4, 6, 5
    vals = rng.normal(0, 1, (N, B, K))
    S = np.broadcast_to(vals[:, 1:, None, :], (N, B - 1, K, K))
    k, _ = oracle.select(S, vals, np.zeros((N, B, K), dtype=np.int64))
    np.testing.assert_array_equal(k, vals.argmax(axis=2))


def test_greedy_is_not_global_sum():
    """The prefix-first walk does not trade an early score for later ones."""
    vals = np.array([[1.0, 0.0], [0.0, 0.0], [0.0, 0.0]])
    S = np.zeros((2, 2, 2))
    S[0, 0] = [1.0, 0.9]          # slot 2: candidate 0 is best given slot 1
    S[1, 0] = [0.0, 0.0]
    S[1, 1] = [5.0, 0.0]          # but candidate 1 unlocks a large later score
    k, _ = oracle.select(S[None], vals[None], np.zeros((1, 3, 2), dtype=np.int64))
    assert list(k[0]) == [0, 0, 0]


# ---------------------------------------------------------------------------
# Whole-path rules: Global-Sum (lambda = 1) and the geometric discount (lambda = 0.75)
# ---------------------------------------------------------------------------


def brute_discounted(S, vals, lam):
    """Every path's score l_0(k_0) + sum_p lam^(p+1) S_p(k_p, k_{p+1}); the best one, ties broken
    towards the lowest last index, then the lowest index before it, and so on."""
    B, K = vals.shape
    best, best_key = None, None
    for path in itertools.product(range(K), repeat=B):
        total = vals[0, path[0]] + sum(lam ** (p + 1) * S[p, path[p], path[p + 1]] for p in range(B - 1))
        key = (total, tuple(-c for c in reversed(path)))
        if best_key is None or key > best_key:
            best, best_key = path, key
    return list(best)


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("lam", [1.0, 0.75, 0.5])
def test_discounted_path_matches_brute_force(seed, lam):
    rng = np.random.default_rng(300 + seed)
    B, K, N = int(rng.integers(2, 6)), int(rng.integers(1, 5)), 3
    vals = rng.integers(-6, 7, (N, B, K)) * 0.5     # dyadic values: every total is exact
    S = rng.integers(-6, 7, (N, B - 1, K, K)) * 0.5
    ids = rng.integers(0, 1000, (N, B, K))
    k, tokens = oracle.select_discounted(S, vals, ids, lam)
    for n in range(N):
        assert list(k[n]) == brute_discounted(S[n], vals[n], lam)
        assert list(tokens[n]) == [ids[n, i, k[n, i]] for i in range(B)]


@pytest.mark.parametrize("lam", [1.0, 0.75])
def test_discounted_path_with_zero_correction_is_per_slot_argmax(lam):
    rng = np.random.default_rng(21)
    N, B, K = 4, 7, 5
    vals = rng.normal(0, 1, (N, B, K))
    S = np.broadcast_to(vals[:, 1:, None, :], (N, B - 1, K, K))
    k, _ = oracle.select_discounted(S, vals, np.zeros((N, B, K), dtype=np.int64), lam)
    np.testing.assert_array_equal(k, np.argmax(vals, axis=2))


def test_discounted_path_small_lambda_is_the_greedy_walk():
    """As lambda -> 0 the objective orders the slots lexicographically: the prefix-first walk."""
    rng = np.random.default_rng(22)
    N, B, K = 50, 5, 4
    vals = rng.normal(0, 1, (N, B, K))
    S = rng.normal(0, 1, (N, B - 1, K, K))
    k_greedy, _ = oracle.select(S, vals, np.zeros((N, B, K), dtype=np.int64))
    k_disc, _ = oracle.select_discounted(S, vals, np.zeros((N, B, K), dtype=np.int64), 1e-3)
    np.testing.assert_array_equal(k_disc, k_greedy)


def test_global_sum_trades_an_early_score_for_a_later_one():
    """On the grid where the prefix-first walk keeps [0, 0, 0], the whole-path sum takes the
    candidate that unlocks the large later score."""
    vals = np.array([[1.0, 0.0], [0.0, 0.0], [0.0, 0.0]])
    S = np.zeros((2, 2, 2))
    S[0, 0] = [1.0, 0.9]
    S[1, 1] = [5.0, 0.0]
    k, _ = oracle.select_discounted(S[None], vals[None], np.zeros((1, 3, 2), dtype=np.int64), 1.0)
    assert list(k[0]) == [0, 1, 0]


# ---------------------------------------------------------------------------
# The pages' worked example (B=4, K=3)
# ---------------------------------------------------------------------------


def load_worked_example():
    grid, words, stated = [], [], {}
    with open(os.path.join(GOLDEN, "worked_example.txt")) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "slot":
                toks = parts[2:]
                words.append(toks[0::2])
                grid.append([float(v) for v in toks[1::2]])
            else:
                stated[parts[0]] = parts[1:]
    return np.array(grid), words, stated


def test_worked_example_printed_values_as_drafter_logits():
    """(T1) The printed numbers read as drafter logits with the correction switched off.

    The per-slot argmax is then These / keys / are / missing.  The review's narrative calls
    the drafter's top-1 reading "These key is missing", which these printed numbers do not
    produce (key 0.4 < keys 2.7): the printed values behave like the corrected scores of
    the chosen path.  The test records what the printed numbers give.
    """
    grid, words, stated = load_worked_example()
    vals = grid[None]
    S = np.broadcast_to(vals[:, 1:, None, :], (1, 3, 3, 3))
    k, _ = oracle.select(S, vals, np.zeros((1, 4, 3), dtype=np.int64))
    assert [words[i][k[0, i]] for i in range(4)] == stated["corrected"]
    assert [words[i][k[0, i]] for i in range(4)] != stated["uncorrected"]


def test_worked_example_printed_values_as_transition_rows():
    """(T2) The printed slot-2..4 values read as the rows S_1(These,.), S_2(keys,.),
    S_3(are,.) of the corrected grid, every other row set lower: the walk follows the
    stated corrected path."""
    grid, words, stated = load_worked_example()
    vals = grid[None].copy()
    S = np.full((1, 3, 3, 3), -10.0)
    path = [words[i].index(stated["corrected"][i]) for i in range(4)]
    for p in range(3):
        S[0, p, path[p], :] = grid[p + 1]
    k, _ = oracle.select(S, vals, np.zeros((1, 4, 3), dtype=np.int64))
    assert list(k[0]) == path


def test_worked_example_uncorrected_reading_needs_other_logits():
    """(T3, builder-invented) A drafter grid whose per-slot argmax reads "These key is
    missing" -- the pages do not print one; this grid swaps the printed values of
    key/keys and is/are -- stays uncorrected when the correction is zero, and a
    correction that favours (These, keys) and (keys, are) turns it into the stated
    corrected path."""
    grid, words, stated = load_worked_example()
    g = grid.copy()
    g[1, [0, 1]] = g[1, [1, 0]]
    g[2, [0, 1]] = g[2, [1, 0]]
    vals = g[None]
    S0 = np.broadcast_to(vals[:, 1:, None, :], (1, 3, 3, 3)).copy()
    k, _ = oracle.select(S0, vals, np.zeros((1, 4, 3), dtype=np.int64))
    assert [words[i][k[0, i]] for i in range(4)] == stated["uncorrected"]
    S = S0.copy()
    S[0, 0, 0, 1] += 3.0       # These -> keys
    S[0, 1, 1, 1] += 3.0       # keys -> are
    k, _ = oracle.select(S, vals, np.zeros((1, 4, 3), dtype=np.int64))
    assert [words[i][k[0, i]] for i in range(4)] == stated["corrected"]


# ---------------------------------------------------------------------------
# Verification
# ---------------------------------------------------------------------------


def test_greedy_verify_closed_form():
    draft = np.array([[5, 6, 7, 8], [5, 6, 7, 8], [5, 6, 7, 8], [1, 1, 1, 1]])
    t = np.array([[5, 6, 7, 8, 9], [4, 6, 7, 8, 9], [5, 6, 0, 8, 9], [1, 1, 1, 2, 3]])
    out = oracle.verify_greedy(draft, t)
    assert list(out["accept_len"]) == [4, 0, 2, 3]
    assert list(out["n_commit"]) == [5, 1, 3, 4]
    np.testing.assert_array_equal(out["committed"], [[5, 6, 7, 8, 9], [4, -1, -1, -1, -1],
                                                     [5, 6, 0, -1, -1], [1, 1, 1, 2, -1]])


def test_greedy_verify_random_against_prefix_definition():
    rng = np.random.default_rng(4)
    draft = rng.integers(0, 3, (200, 6))
    t = rng.integers(0, 3, (200, 7))
    out = oracle.verify_greedy(draft, t)
    for n in range(200):
        A = next((j for j in range(6) if draft[n, j] != t[n, j]), 6)
        assert out["accept_len"][n] == A
        assert list(out["committed"][n, :A + 1]) == list(draft[n, :A]) + [t[n, A]]


def test_stochastic_verify_hand_cases():
    q = np.array([[[0.1, 0.2, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25]]])   # B=1, V=4
    draft = np.array([[2]])
    # accept iff u0 < q(y) = 0.3 (strict); then the bonus comes from q_2 with u[1,1]
    u = np.array([[[0.29, 0.0], [0.0, 0.6]]])
    out = oracle.verify_stochastic(draft, q, u)
    assert out["accept_len"][0] == 1 and list(out["committed"][0]) == [2, 2]
    # reject (u0 == q(y)); residual [0.1, 0.2, 0, 0.4] / 0.7; u1 = 0.5 -> target 0.35 -> token 3
    u = np.array([[[0.3, 0.5], [0.0, 0.0]]])
    out = oracle.verify_stochastic(draft, q, u)
    assert out["accept_len"][0] == 0 and list(out["committed"][0]) == [3, -1]
    # u1 = 0.2 -> target 0.14 -> token 1;  u1 = 0 -> token 0
    u = np.array([[[0.9, 0.2], [0.0, 0.0]]])
    assert oracle.verify_stochastic(draft, q, u)["committed"][0, 0] == 1
    u = np.array([[[0.9, 0.0], [0.0, 0.0]]])
    assert oracle.verify_stochastic(draft, q, u)["committed"][0, 0] == 0


def test_stochastic_verify_preserves_verifier_distribution():
    """Point-mass proposals keep the committed tokens distributed as the verifier's q
    (slot 1 unconditionally; slot 2 given that slot 1 committed the draft token)."""
    from scipy.stats import chi2
    V, T = 6, 60000
    q1 = np.array([0.05, 0.3, 0.1, 0.25, 0.2, 0.1])
    q2 = np.array([0.4, 0.1, 0.1, 0.1, 0.2, 0.1])
    q = np.broadcast_to(np.stack([q1, q2, q1]), (T, 3, V))
    draft = np.broadcast_to(np.array([3, 0]), (T, 2))
    u = np.random.default_rng(2024).random((T, 3, 2))
    out = oracle.verify_stochastic(draft, q, u)
    c = out["committed"]
    for obs, p in ((c[:, 0], q1), (c[(c[:, 0] == 3), 1], q2)):
        counts = np.bincount(obs, minlength=V)
        exp = p * len(obs)
        stat = ((counts - exp) ** 2 / exp).sum()
        assert chi2.sf(stat, V - 1) > 1e-4, (counts, exp)
    # acceptance rate at slot 1 equals q1(y1)
    assert abs((out["accept_len"] > 0).mean() - q1[3]) < 4 * math.sqrt(0.25 / T)


# ---------------------------------------------------------------------------
# Speculative sampling with a general draft distribution
# ---------------------------------------------------------------------------


def _softmax_rows(x):
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def test_speculative_hand_cases():
    p = np.array([[[0.5, 0.5, 0.0, 0.0]]])            # B = 1, V = 4
    q = np.array([[[0.25, 0.25, 0.25, 0.25], [0.1, 0.2, 0.3, 0.4]]])
    draft = np.array([[0]])
    # accept iff u0 * p(y) < q(y): 0.4 * 0.5 = 0.2 < 0.25; then the bonus from q_2 with u[1,1]
    out = oracle.verify_speculative(draft, p, q, np.array([[[0.4, 0.0], [0.0, 0.75]]]))
    assert out["accept_len"][0] == 1 and list(out["committed"][0]) == [0, 3]
    # 0.5 * 0.5 = 0.25 is not below 0.25: reject; residual max(0, q - p) = [0, 0, .25, .25]
    out = oracle.verify_speculative(draft, p, q, np.array([[[0.5, 0.5], [0.0, 0.0]]]))
    assert out["accept_len"][0] == 0 and list(out["committed"][0]) == [3, -1]
    out = oracle.verify_speculative(draft, p, q, np.array([[[0.9, 0.4], [0.0, 0.0]]]))
    assert list(out["committed"][0]) == [2, -1]


def test_speculative_point_mass_is_the_stochastic_rule():
    rng = np.random.default_rng(31)
    N, B, V = 40, 6, 50
    q = _softmax_rows(rng.normal(0, 2, (N, B + 1, V)))
    draft = rng.integers(0, V, (N, B))
    u = rng.random((N, B + 1, 2))
    p = np.zeros((N, B, V))
    np.put_along_axis(p, draft[:, :, None], 1.0, axis=2)
    a = oracle.verify_speculative(draft, p, q, u)
    b = oracle.verify_stochastic(draft, q, u)
    for k in ("accept_len", "committed", "n_commit"):
        np.testing.assert_array_equal(a[k], b[k])


def test_speculative_equal_distributions_accept_everything():
    rng = np.random.default_rng(32)
    N, B, V = 30, 5, 40
    q = _softmax_rows(rng.normal(0, 1, (N, B + 1, V)))
    draft = np.array([[rng.choice(V, p=q[n, j]) for j in range(B)] for n in range(N)])
    out = oracle.verify_speculative(draft, q[:, :B], q, rng.random((N, B + 1, 2)))
    assert (out["accept_len"] == B).all()


def test_speculative_preserves_target_distribution():
    """Drafts drawn from p, verified against q: the committed first token is distributed as q."""
    from scipy.stats import chi2
    V, T = 6, 60000
    p1 = np.array([0.3, 0.05, 0.25, 0.1, 0.2, 0.1])
    q1 = np.array([0.05, 0.3, 0.1, 0.25, 0.2, 0.1])
    rng = np.random.default_rng(2025)
    draft = rng.choice(V, size=(T, 1), p=p1)
    p = np.broadcast_to(p1, (T, 1, V))
    q = np.broadcast_to(np.stack([q1, q1]), (T, 2, V))
    out = oracle.verify_speculative(draft, p, q, rng.random((T, 2, 2)))
    counts = np.bincount(out["committed"][:, 0], minlength=V)
    exp = q1 * T
    assert chi2.sf(((counts - exp) ** 2 / exp).sum(), V - 1) > 1e-4, (counts, exp)
    # the acceptance rate is sum_v min(p(v), q(v))
    rate = np.minimum(p1, q1).sum()
    assert abs((out["accept_len"] > 0).mean() - rate) < 4 * math.sqrt(0.25 / T)


# ---------------------------------------------------------------------------
# Synthetic verifier statistic
# ---------------------------------------------------------------------------


def test_synthetic_verifier_mean_accept_length():
    cfg = wl.HEADLINE.replace(N=3000, V=1000)
    rng = np.random.default_rng(0)
    draft = rng.integers(0, cfg.V, (cfg.N, cfg.B))
    t = wl.verifier_tokens(cfg, draft)
    A = oracle.verify_greedy(draft, t)["accept_len"]
    p = [wl.match_probability(j) for j in range(1, cfg.B + 1)]
    want = sum(np.prod(p[:j + 1]) for j in range(cfg.B))
    assert abs(A.mean() - want) < 4 * A.std() / math.sqrt(cfg.N)
