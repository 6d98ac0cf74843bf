"""Float64 CPU oracle of the DCOCO per-cycle hot path.

TEST INFRASTRUCTURE ONLY.  This is a plain, slow, obviously-correct restatement of
what the method computes, used to check the CUDA library.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it; the library never calls it and has no fallback to it.  It shares no code with
the CUDA path.

Sources (the method has no published code; these pages describe it in prose):
  [Blog]   Two Delta, "Two Delta makes NVIDIA Nemotron 3.5 Super even faster with
           DCOCO", sections "Keep the leading candidates", "Score neighboring
           candidates in parallel", "Select using the realized token identities",
           "How we train the corrector".
  [Review] jaehun.me review of arXiv 2610.12570, "Contextual Correction of Parallel
           Drafts for Speculative Decoding": §3.1 (verification, accept length),
           §3.2 (learned corrector on the block grid: candidate representation,
           pair state, shared two-layer MLP, zero-initialised output layer),
           §3.3 (prefix-first greedy selection), App. D (point-mass proposal under
           stochastic verification), and the worked B=4, K=3 example (Fig. 2).

The display formulas on both pages were lost in extraction.  The functional form
used here is the one the pages describe in words:
    b_ik = LN(W_e Emb[c_ik]),  g_i = LN(W_h h_i)           (LN: no affine, eps 1e-5)
    z_ik = SiLU(W_f [b_ik; g_i]),  s_p = W_pair [h_p; h_{p+1}]
    S_p(a, b) = l_{p+1}(b) + w2 . SiLU(U z_{p,a} + V z_{p+1,b} + W s_p
                                       + u_a l_p(a) + u_b l_{p+1}(b) + b1) + b2
Every array here is float64; inputs arrive as exact float64 widenings of the
bf16/f32 data.  Indices are 0-based: slot i in 0..B-1, transition p in 0..B-2
scores slot p -> slot p+1.

Parity pins (what fixes each function independently of this file) are listed in
each docstring; functions whose internals no page example fixes say
"parity unpinned by the pages" and are pinned by closed-form special cases.
"""
from __future__ import annotations

from typing import Dict, Tuple

import numpy as np

LN_EPS = 1e-5


def canonical(x: np.ndarray) -> np.ndarray:
    """Ordering view of logits: NaN ranks as -inf and -0 equals +0.

    The pages never mention NaN; treating it as the lowest value keeps the order total.
    """
    y = np.where(np.isnan(x), -np.inf, x)
    return y + 0.0  # -0.0 + 0.0 == +0.0


def topk(logits: np.ndarray, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """Keep the K largest logits of each row ([Blog] "Keep the leading candidates";
    [Review] §3.2: the drafter leaves top-K candidates c_ik with logits l_i(k)).

    Order: value descending, equal values by ascending token id.  Done as a full
    stable sort of each row on the negated value, which keeps ids in ascending order
    among equal values.  Returns (vals [..., K] float64, ids [..., K] int64).
    Pinned by brute-force selection in the tests.
    """
    x = canonical(np.asarray(logits, dtype=np.float64))
    order = np.argsort(-x, axis=-1, kind="stable")[..., :K]
    return np.take_along_axis(x, order, axis=-1), order.astype(np.int64)


def lm_logits(h: np.ndarray, W_lm: np.ndarray) -> np.ndarray:
    """The drafter's output projection: l[..., v] = sum_k h[..., k] W_lm[v, k].

    [Blog] "Score neighboring candidates in parallel": the corrector reuses what the
    drafter's own pass produced, and the logits l_i(k) it keeps are that pass's vocabulary
    projection of the drafter's final hidden state at slot i.  W_lm is stored [V, d]
    (one row per token).  Pinned by per-logit loops and one-hot rows in the tests.
    """
    h = np.asarray(h, dtype=np.float64)
    W_lm = np.asarray(W_lm, dtype=np.float64)
    return h @ W_lm.T


def lm_head_topk(h: np.ndarray, W_lm: np.ndarray, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-K of the drafter's logits computed from its hidden state: topk(lm_logits(h, W_lm)).

    The plain definition of the fused LM-head/top-K kernel: the logits exist here in full,
    in float64; the GPU never stores them.
    """
    return topk(lm_logits(h, W_lm), K)


def layer_norm(x: np.ndarray, eps: float = LN_EPS) -> np.ndarray:
    """Non-affine layer normalisation over the last axis ([Review] §3.2: the embedding
    and hidden-state projections are normalised without affine parameters because
    their scales differ by orders of magnitude).  Biased variance; eps = 1e-5 (the
    pages give no eps)."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x)."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def candidate_repr(ids: np.ndarray, emb: np.ndarray, h: np.ndarray, w: Dict[str, np.ndarray]
                   ) -> Dict[str, np.ndarray]:
    """Candidate representations z_ik ([Blog] "Score neighboring candidates in parallel";
    [Review] §3.2, candidate representation).

    b_ik = LN(W_e Emb[c_ik])        -- identity of the candidate token (frozen embedding)
    g_i  = LN(W_h h_i)              -- context of the slot
    z_ik = SiLU(W_f [b_ik; g_i])    -- fused, concatenation order [b; g]

    ids [N,B,K] int, emb [V,E], h [N,B,d]; returns b, g [N,B,r], z [N,B,K,r].
    Parity unpinned by the pages (no numeric example); pinned by closed-form cases
    with structured weights in the tests.
    """
    b = layer_norm(emb[ids] @ w["W_e"].T)
    g = layer_norm(h @ w["W_h"].T)
    gk = np.broadcast_to(g[:, :, None, :], b.shape)
    z = silu(np.concatenate([b, gk], axis=-1) @ w["W_f"].T)
    return {"b": b, "g": g, "z": z}


def pair_state(h: np.ndarray, w: Dict[str, np.ndarray]) -> np.ndarray:
    """Pair state s_p = W_pair [h_p; h_{p+1}] for p = 0..B-2 ([Blog], the shared context of
    neighbouring positions; [Review] §3.2, pair state).  h [N,B,d] -> s [N,B-1,r]."""
    hh = np.concatenate([h[:, :-1, :], h[:, 1:, :]], axis=-1)
    return hh @ w["W_pair"].T


def transition_scores(z: np.ndarray, s: np.ndarray, vals: np.ndarray, w: Dict[str, np.ndarray]
                      ) -> np.ndarray:
    """All (B-1)K^2 transition scores ([Blog] "Score neighboring candidates in parallel";
    [Review] §3.2):

        S_p(a,b) = l_{p+1}(b) + w2 . SiLU(U z_{p,a} + V z_{p+1,b} + W s_p
                                          + u_a l_p(a) + u_b l_{p+1}(b) + b1) + b2

    The first layer of the shared MLP acts on [z_{p,a}; z_{p+1,b}; s_p; l_p(a); l_{p+1}(b)];
    by linearity it is the sum of the five blocks written above, each evaluated with a
    matrix product and summed in that order.  Scores are not normalised at inference
    ([Review] §3.2: the softmax exists only in training).

    z [N,B,K,r], s [N,B-1,r], vals [N,B,K] -> S [N,B-1,K,K] (predecessor a, successor b).
    Pinned by the zero-output-layer identity S = l_{p+1}(b) and closed-form cases.
    """
    N, B, K, _ = z.shape
    UZ = z @ w["U"].T                  # [N,B,K,H]: U z for each candidate
    VZ = z @ w["V"].T
    WS = s @ w["W"].T                  # [N,B-1,H]
    S = np.empty((N, B - 1, K, K))
    for n in range(N):
        pre = (UZ[n, :-1, :, None, :]
               + VZ[n, 1:, None, :, :]
               + WS[n, :, None, None, :]
               + w["u_a"] * vals[n, :-1, :, None, None]
               + w["u_b"] * vals[n, 1:, None, :, None]
               + w["b1"])
        S[n] = vals[n, 1:, None, :] + silu(pre) @ w["w2"] + w["b2"][0]
    return S


def _argmax_first(x: np.ndarray) -> int:
    """Index of the largest entry; ties go to the lowest index; NaN ranks lowest."""
    return int(np.argmax(canonical(x)))


def select(S: np.ndarray, vals: np.ndarray, ids: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Prefix-first greedy walk ([Blog] "Select using the realized token identities";
    [Review] §3.3).

    k_1 keeps the drafter's first choice (argmax of l_1); every later slot takes the
    candidate with the highest score given the candidate actually chosen before it:
    k_{p+1} = argmax_b S_p(k_p, b).  Ties go to the lower candidate index.
    Returns k [N,B] and the draft tokens c_{i,k_i} [N,B].
    Pinned by brute force over all K^B paths and by the zero-correction identity.
    """
    N, B, K = vals.shape
    k = np.empty((N, B), dtype=np.int64)
    for n in range(N):
        k[n, 0] = _argmax_first(vals[n, 0])
        for p in range(B - 1):
            k[n, p + 1] = _argmax_first(S[n, p, k[n, p]])
    tokens = np.take_along_axis(ids, k[:, :, None], axis=2)[:, :, 0]
    return k, tokens


def select_discounted(S: np.ndarray, vals: np.ndarray, ids: np.ndarray, lam: float
                      ) -> Tuple[np.ndarray, np.ndarray]:
    """Whole-path selection rules on the same score grid ([Review] "path choice and ablation",
    Tab. 3): Global-Sum maximises the path's total score, the geometric discount weights later
    slots down by lambda (0.75 on the page).  Both formulas were lost in extraction; the reading
    taken here unifies them (lambda = 1 is Global-Sum):

        maximise  l_0(k_0) + sum_{p=0}^{B-2} lambda^(p+1) S_p(k_p, k_{p+1})   over all K^B paths,

    the weight lambda^i of slot i standing for the chance that its prefix survives.  Computed by
    the max-sum recursion (Viterbi): V_0(a) = l_0(a), V_{p+1}(b) = max_a V_p(a) + lambda^(p+1)
    S_p(a, b), each maximum taken by the lowest index among equal values, then backtracked from
    the lowest maximiser of V_{B-1}.  Returns k [N,B] and the draft tokens [N,B].
    Pinned by brute force over all paths, the zero-correction identity (per-slot argmax for any
    lambda) and the small-lambda limit (the prefix-first greedy walk).
    """
    N, B, K = vals.shape
    k = np.empty((N, B), dtype=np.int64)
    for n in range(N):
        V = canonical(vals[n, 0])
        back = np.zeros((B, K), dtype=np.int64)
        w = 1.0
        for p in range(B - 1):
            w *= lam
            cand = V[:, None] + w * canonical(S[n, p])        # [a, b]
            back[p + 1] = np.argmax(cand, axis=0)              # lowest a among equal values
            V = cand[back[p + 1], np.arange(K)]
        k[n, B - 1] = _argmax_first(V)
        for p in range(B - 1, 0, -1):
            k[n, p - 1] = back[p, k[n, p]]
    tokens = np.take_along_axis(ids, k[:, :, None], axis=2)[:, :, 0]
    return k, tokens


def verify_greedy(draft: np.ndarray, t: np.ndarray) -> Dict[str, np.ndarray]:
    """Greedy verification ([Review] §3.1): slots are judged left to right, slot j is
    accepted while the draft equals the verifier's greedy token; the accept length A
    is the number of accepted slots before the first rejection; the round commits the
    accepted prefix plus the verifier's own token at the first rejected slot (or the
    bonus position B+1 when all B are accepted), A+1 tokens in all.

    draft [N,B], t [N,B+1] -> accept_len [N], committed [N,B+1] (-1 padded), n_commit [N].
    """
    N, B = draft.shape
    acc = np.zeros(N, dtype=np.int64)
    com = np.full((N, B + 1), -1, dtype=np.int64)
    for n in range(N):
        A = 0
        while A < B and draft[n, A] == t[n, A]:
            com[n, A] = draft[n, A]
            A += 1
        com[n, A] = t[n, A]
        acc[n] = A
    return {"accept_len": acc, "committed": com, "n_commit": acc + 1}


def _inverse_cdf(r: np.ndarray, u: float, fallback: int) -> Tuple[int, bool]:
    """The smallest v (vocabulary order) whose running sum of the residual mass r exceeds u * R,
    R = sum(r), and whether u * R lies within 1e-9 R of a step of that running sum (a draw that
    another summation order may resolve differently).  R <= 0 returns `fallback`."""
    cum = np.cumsum(r)
    R = cum[-1]
    if not R > 0.0:
        return fallback, True
    target = float(u) * R
    v = int(np.searchsorted(cum, target, side="right"))
    if v >= len(r):  # only reachable through rounding of u * R
        v = int(np.flatnonzero(r > 0)[-1])
    near = abs(cum[v] - target) <= 1e-9 * R or (v > 0 and abs(cum[v - 1] - target) <= 1e-9 * R)
    return v, bool(near)


def residual_draw(q: np.ndarray, u: float, exclude: int) -> Tuple[int, bool]:
    """Inverse-CDF draw from r(v) = q(v) 1[v != exclude] / R with R = sum_{v != exclude} q(v)
    ([Review] App. D; exclude = -1 draws from q itself).

    Returns the smallest v (in vocabulary order, v != exclude) whose running sum of the
    residual mass exceeds u * R, and whether u * R lies within 1e-9 R of a step of
    that running sum (a draw that another summation order may resolve differently).
    Degenerate R <= 0 returns `exclude` (no residual mass).
    """
    r = np.asarray(q, dtype=np.float64).copy()
    if exclude >= 0:
        r[exclude] = 0.0
    return _inverse_cdf(r, u, exclude)


def verify_stochastic(draft: np.ndarray, q: np.ndarray, u: np.ndarray) -> Dict[str, np.ndarray]:
    """Speculative sampling with a point-mass proposal ([Review] App. D and §3.1).

    The corrected draft is deterministic, so slot j's proposal is p_j = 1[v = y_j].  The
    standard rule min{1, q_j(y_j)/p_j(y_j)} then accepts with probability q_j(y_j): here
    slot j is accepted iff u[j,0] < q_j(y_j).  At the first rejection the verifier token
    is drawn from the residual q_j(v) 1[v != y_j] / (1 - q_j(y_j)) with u[j,1]; if all B
    slots are accepted, the bonus token is drawn from q_{B+1} with u[B,1].

    draft [N,B], q [N,B+1,V], u [N,B+1,2] -> accept_len, committed, n_commit, near_tie [N].
    """
    N, B = draft.shape
    acc = np.zeros(N, dtype=np.int64)
    com = np.full((N, B + 1), -1, dtype=np.int64)
    near = np.zeros(N, dtype=bool)
    for n in range(N):
        A = 0
        while A < B and float(u[n, A, 0]) < float(q[n, A, draft[n, A]]):
            com[n, A] = draft[n, A]
            A += 1
        if A < B:
            v, nt = residual_draw(q[n, A], u[n, A, 1], int(draft[n, A]))
        else:
            v, nt = residual_draw(q[n, B], u[n, B, 1], -1)
        com[n, A] = v
        acc[n] = A
        near[n] = nt
    return {"accept_len": acc, "committed": com, "n_commit": acc + 1, "near_tie": near}


def verify_speculative(draft: np.ndarray, p: np.ndarray, q: np.ndarray, u: np.ndarray) -> Dict[str, np.ndarray]:
    """Speculative sampling with a general draft distribution ([Review] §3.1, the standard rule
    that App. D specialises to a point mass): the draft token y_j was drawn from p_j; slot j is
    accepted with probability min{1, q_j(y_j) / p_j(y_j)}, here iff u[j,0] p_j(y_j) < q_j(y_j)
    (the product of two float32 values, exact in float64); at the first rejection the committed
    token is drawn from the residual max(0, q_j - p_j) / R, R its total, by inverse CDF in
    vocabulary order with u[j,1] (R <= 0 keeps the draft token); if all B slots are accepted the
    bonus token is drawn from q_{B+1}.  A one-hot p_j at y_j gives exactly verify_stochastic.

    draft [N,B], p [N,B,V], q [N,B+1,V], u [N,B+1,2] -> accept_len, committed, n_commit, near_tie.
    """
    N, B = draft.shape
    acc = np.zeros(N, dtype=np.int64)
    com = np.full((N, B + 1), -1, dtype=np.int64)
    near = np.zeros(N, dtype=bool)
    for n in range(N):
        A = 0
        while A < B:
            y = int(draft[n, A])
            if not float(u[n, A, 0]) * float(p[n, A, y]) < float(q[n, A, y]):
                break
            com[n, A] = y
            A += 1
        if A < B:
            r = np.maximum(0.0, np.asarray(q[n, A], dtype=np.float64) - np.asarray(p[n, A], dtype=np.float64))
            v, nt = _inverse_cdf(r, u[n, A, 1], int(draft[n, A]))
        else:
            v, nt = residual_draw(q[n, B], u[n, B, 1], -1)
        com[n, A] = v
        acc[n] = A
        near[n] = nt
    return {"accept_len": acc, "committed": com, "n_commit": acc + 1, "near_tie": near}


def cycle(logits: np.ndarray, emb: np.ndarray, h: np.ndarray, w: Dict[str, np.ndarray], K: int
          ) -> Dict[str, np.ndarray]:
    """One correction pass: top-K, representations, pair states, scores, walk."""
    vals, ids = topk(logits, K)
    rep = candidate_repr(ids, emb, h, w)
    s = pair_state(h, w)
    S = transition_scores(rep["z"], s, vals, w)
    k, tokens = select(S, vals, ids)
    return {"vals": vals, "ids": ids, "s": s, "S": S, "k": k, "tokens": tokens, **rep}


def cycle_lm(h: np.ndarray, W_lm: np.ndarray, emb: np.ndarray, w: Dict[str, np.ndarray], K: int
             ) -> Dict[str, np.ndarray]:
    """One correction pass starting from the drafter's hidden state: its logits are
    lm_logits(h, W_lm), then the same pass as ``cycle``.  The one hidden state h feeds both
    the output projection and the corrector (g and the pair states)."""
    return cycle(lm_logits(h, W_lm), emb, h, w, K)
