"""Per-step parity of the CUDA library against the float64 oracle (needs a GB300).

Every call goes through the C ABI (ctypes binding); inputs come from the seeded
generators and are handed to both sides bit-identically.
"""
import numpy as np
import pytest
import torch

import draft_correction_gb300 as dc
import oracle
import workloads as wl
from helpers import (assert_intermediate_close, assert_scores_close, case, compare_walk, f64, w64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from draft_correction_gb300 import build
    build.build()
    dc.lib()
    yield
    assert dc.device_status() == 0, "a kernel reported a timeout or a bad index"


def _bf16_rows(x32):
    return wl.f32_to_bf16(np.asarray(x32, dtype=np.float32))


def run_topk(x, dtype, K):
    t = dc.to_device(x, dtype)
    vals, ids = dc.topk(t, K)
    torch.cuda.synchronize()
    return vals.cpu().numpy(), ids.cpu().numpy()


def check_topk(x, dtype, K):
    vals, ids = run_topk(x, dtype, K)
    rv, ri = oracle.topk(wl.to_f64(x, dtype), K)
    np.testing.assert_array_equal(ids, ri)
    np.testing.assert_array_equal(vals.astype(np.float64), rv)
    assert not np.signbit(vals[vals == 0]).any()


# ---------------------------------------------------------------- a1 top-K


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V,K", [(1024, 3), (1001, 7), (4099, 16), (64, 64), (40, 40), (20000, 1), (151936, 16),
                                 (9, 1), (300007, 64), (131, 33)])
def test_topk_random(dtype, V, K):
    rng = np.random.default_rng(V * 131 + K)
    x = rng.normal(0, 3, (3, 5, V)).astype(np.float32)
    check_topk(_bf16_rows(x) if dtype == "bf16" else x, dtype, K)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_adversarial(dtype):
    V = 5003
    rows = []
    rows.append(np.full(V, 1.5, np.float32))                               # all equal: lowest K ids
    r = np.zeros(V, np.float32); r[1::2] = -0.0; rows.append(r)            # +-0 ties
    r = np.full(V, -np.inf, np.float32); r[[7, 4000, 5002]] = np.inf; r[[5, 6]] = np.nan; rows.append(r)
    r = np.full(V, np.nan, np.float32); r[100] = -np.inf; rows.append(r)  # NaN ranks as -inf
    r = np.arange(V, dtype=np.float32); rows.append(r)                     # ascending: every element inserts
    r = -np.arange(V, dtype=np.float32); rows.append(r)                    # descending
    r = np.random.default_rng(0).normal(0, 1, V).astype(np.float32); r[[0, V - 1]] = 50; rows.append(r)
    r = np.round(np.random.default_rng(1).normal(0, 1, V), 0).astype(np.float32); rows.append(r)  # many ties
    x = np.stack(rows)[None]
    if dtype == "bf16":
        x = _bf16_rows(x)
        x[x == 0x7FC1] = 0x7FC0
    for K in (1, 5, 16, 33, 64):
        check_topk(x, dtype, K)


@pytest.mark.parametrize("split", [1, 2, 3, 5, 8])
def test_topk_independent_of_split(split):
    rng = np.random.default_rng(9)
    x = _bf16_rows(np.round(rng.normal(0, 2, (2, 3, 70001)), 1))
    prev = dc.set_topk_split(split)
    try:
        check_topk(x, "bf16", 16)
    finally:
        dc.set_topk_split(prev)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [wl.QWEN3_8B, wl.HEADLINE], ids=lambda c: c.name)
def test_topk_full_size(cfg):
    check_topk(wl.logits(cfg), cfg.dtype, cfg.K)


# ---------------------------------------------------------------- a5 walk, a6 verify


@pytest.mark.parametrize("N,B,K", [(3, 4, 3), (8, 16, 16), (5, 7, 33), (2, 64, 64), (2, 3, 1), (40, 16, 5)])
def test_select_matches_oracle(N, B, K):
    rng = np.random.default_rng(N * 1000 + B * 10 + K)
    vals = np.round(rng.normal(0, 1, (N, B, K)), 1).astype(np.float32)
    S = np.round(rng.normal(0, 1, (N, B - 1, K, K)), 1).astype(np.float32)
    S[0, 0, :, 0] = np.nan
    ids = rng.integers(0, 10 ** 6, (N, B, K)).astype(np.int32)
    k, tok = dc.select(dc.to_device(S, "f32"), dc.to_device(vals, "f32"), dc.to_device(ids, "i32"))
    rk, rt = oracle.select(S.astype(np.float64), vals.astype(np.float64), ids)
    np.testing.assert_array_equal(k.cpu().numpy(), rk)
    np.testing.assert_array_equal(tok.cpu().numpy(), rt)


def _path_score(S, vals, path, lam):
    return vals[0, path[0]] + sum(lam ** (p + 1) * S[p, path[p], path[p + 1]] for p in range(len(path) - 1))


@pytest.mark.parametrize("lam", [1.0, 0.75, 0.5])
@pytest.mark.parametrize("seed", range(4))
def test_select_path_exact_on_dyadic_grids(seed, lam):
    """Half-integer scores and power-of-two-friendly discounts make every path score exact in
    float32 as well, so the GPU recursion must pick exactly the oracle's path (ties included)."""
    rng = np.random.default_rng(500 + seed)
    N, B, K = 40, int(rng.integers(2, 9)), int(rng.integers(1, 17))
    vals = (rng.integers(-6, 7, (N, B, K)) * 0.5).astype(np.float32)
    S = (rng.integers(-6, 7, (N, B - 1, K, K)) * 0.5).astype(np.float32)
    ids = rng.integers(0, 10 ** 6, (N, B, K)).astype(np.int32)
    rule = "global_sum" if lam == 1.0 else "geometric"
    k, tok = dc.select_path(dc.to_device(S, "f32"), dc.to_device(vals, "f32"), dc.to_device(ids, "i32"), rule, lam)
    rk, rt = oracle.select_discounted(S.astype(np.float64), vals.astype(np.float64), ids, lam)
    np.testing.assert_array_equal(k.cpu().numpy(), rk)
    np.testing.assert_array_equal(tok.cpu().numpy(), rt)


@pytest.mark.parametrize("rule,lam", [("global_sum", 1.0), ("geometric", 0.75)])
@pytest.mark.parametrize("N,B,K", [(32, 16, 16), (5, 64, 64), (3, 9, 33)])
def test_select_path_matches_oracle(rule, lam, N, B, K):
    """Continuous scores: where the float32 recursion picks another path than the float64 one,
    that path must score within the float32 accumulation error of the optimum (with lambda < 1
    the late slots weigh lambda^p, far below that error at B = 64, so many paths tie there)."""
    rng = np.random.default_rng(N + B + K)
    vals = rng.normal(0, 3, (N, B, K)).astype(np.float32)
    S = rng.normal(0, 3, (N, B - 1, K, K)).astype(np.float32)
    ids = rng.integers(0, 10 ** 6, (N, B, K)).astype(np.int32)
    k, tok = dc.select_path(dc.to_device(S, "f32"), dc.to_device(vals, "f32"), dc.to_device(ids, "i32"), rule, lam)
    k = k.cpu().numpy()
    S64, v64 = S.astype(np.float64), vals.astype(np.float64)
    rk, _ = oracle.select_discounted(S64, v64, ids, lam)
    for n in range(N):
        if (k[n] == rk[n]).all():
            continue
        best, got = _path_score(S64[n], v64[n], rk[n], lam), _path_score(S64[n], v64[n], k[n], lam)
        assert got >= best - 1e-5 * (1.0 + abs(best)), (n, got, best)
    np.testing.assert_array_equal(tok.cpu().numpy(), np.take_along_axis(ids, k[:, :, None], axis=2)[:, :, 0])


def test_select_path_greedy_rule_is_the_walk():
    rng = np.random.default_rng(9)
    N, B, K = 20, 12, 8
    vals = dc.to_device(rng.normal(0, 1, (N, B, K)).astype(np.float32), "f32")
    S = dc.to_device(rng.normal(0, 1, (N, B - 1, K, K)).astype(np.float32), "f32")
    ids = dc.to_device(rng.integers(0, 1000, (N, B, K)).astype(np.int32), "i32")
    k1, t1 = dc.select(S, vals, ids)
    k2, t2 = dc.select_path(S, vals, ids, "greedy")
    assert torch.equal(k1, k2) and torch.equal(t1, t2)


@pytest.mark.parametrize("N,B", [(1, 1), (50, 16), (7, 64), (9, 33)])
def test_verify_greedy_matches_oracle(N, B):
    rng = np.random.default_rng(B)
    draft = rng.integers(0, 4, (N, B)).astype(np.int32)
    t = rng.integers(0, 4, (N, B + 1)).astype(np.int32)
    t[0, :B] = draft[0]                          # one fully accepted block
    out = dc.verify(dc.to_device(draft, "i32"), t=dc.to_device(t, "i32"))
    ref = oracle.verify_greedy(draft, t)
    for k in ("accept_len", "committed", "n_commit"):
        np.testing.assert_array_equal(out[k].cpu().numpy(), ref[k])


def _softmax32(x):
    x = x - x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


@pytest.mark.parametrize("N,B,V", [(64, 16, 1000), (8, 8, 151936), (16, 4, 5)])
def test_verify_speculative_matches_oracle(N, B, V):
    rng = np.random.default_rng(V + B)
    p = _softmax32(rng.normal(0, 2, (N, B, V)))
    q = _softmax32(rng.normal(0, 2, (N, B + 1, V)))
    q[:, :B] = 0.5 * q[:, :B] + 0.5 * p        # overlap, so that drafts are often accepted
    cum = np.cumsum(p.astype(np.float64), axis=2)           # drafts drawn from p by inverse CDF
    draft = np.minimum((cum < rng.random((N, B, 1)) * cum[:, :, -1:]).sum(axis=2), V - 1).astype(np.int32)
    u = rng.random((N, B + 1, 2)).astype(np.float32)
    out = dc.verify_speculative(dc.to_device(draft, "i32"), dc.to_device(p, "f32"), dc.to_device(q, "f32"),
                                dc.to_device(u, "f32"))
    ref = oracle.verify_speculative(draft, p, q, u)
    np.testing.assert_array_equal(out["accept_len"].cpu().numpy(), ref["accept_len"])
    np.testing.assert_array_equal(out["n_commit"].cpu().numpy(), ref["n_commit"])
    com, rcom, tie = out["committed"].cpu().numpy(), ref["committed"], ref["near_tie"]
    for n in range(N):
        if not tie[n]:
            np.testing.assert_array_equal(com[n], rcom[n])


def test_verify_speculative_point_mass_equals_stochastic():
    rng = np.random.default_rng(77)
    N, B, V = 32, 8, 3000
    q = _softmax32(rng.normal(0, 2, (N, B + 1, V)))
    draft = rng.integers(0, V, (N, B)).astype(np.int32)
    u = rng.random((N, B + 1, 2)).astype(np.float32)
    p = np.zeros((N, B, V), dtype=np.float32)
    np.put_along_axis(p, draft[:, :, None].astype(np.int64), 1.0, axis=2)
    d_draft, d_q, d_u = dc.to_device(draft, "i32"), dc.to_device(q, "f32"), dc.to_device(u, "f32")
    a = dc.verify_speculative(d_draft, dc.to_device(p, "f32"), d_q, d_u)
    b = dc.verify(d_draft, q=d_q, u=d_u, mode=dc.VERIFY_STOCHASTIC)
    for k in ("accept_len", "committed", "n_commit"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("N,B,V", [(64, 16, 1000), (8, 8, 151936), (16, 4, 5)])
def test_verify_stochastic_matches_oracle(N, B, V):
    cfg = wl.HEADLINE.replace(N=N, B=B, V=V)
    q = wl.verifier_probs(cfg)
    u = wl.uniforms(cfg)
    rng = np.random.default_rng(V)
    draft = rng.integers(0, V, (N, B)).astype(np.int32)
    # make acceptance likely at some slots: put mass on the draft token
    for n in range(0, N, 2):
        q[n, :B][np.arange(B), draft[n]] = 0.9
    out = dc.verify(dc.to_device(draft, "i32"), q=dc.to_device(q, "f32"), u=dc.to_device(u, "f32"),
                    mode=dc.VERIFY_STOCHASTIC)
    ref = oracle.verify_stochastic(draft, q, u)
    np.testing.assert_array_equal(out["accept_len"].cpu().numpy(), ref["accept_len"])
    near = out["near_tie"].cpu().numpy().astype(bool) | ref["near_tie"]
    com = out["committed"].cpu().numpy()
    np.testing.assert_array_equal(com[~near], ref["committed"][~near])
    assert near.sum() <= max(1, N // 20)


# ---------------------------------------------------------------- a2, a3, a4

SMALL_BF16 = wl.scaled(wl.QWEN3_8B, N=2, B=5, K=5, V=3001, d=256, E=192, r=64, H=128)
SMALL_R256 = wl.scaled(wl.HEADLINE, N=3, B=6, K=16, V=5000, d=512, E=512, r=256, H=512)
SMALL_R512 = wl.scaled(wl.LARGE, N=2, B=4, K=8, V=2000, d=1024, E=1024, r=512, H=1024)
SMALL_H320 = wl.scaled(wl.QWEN3_8B, N=2, B=4, K=6, V=2000, d=128, E=128, r=64, H=320)
REPR_CASES = [wl.TINY, SMALL_BF16, SMALL_R256, SMALL_R512, SMALL_H320]


def _device_case(cfg, variant=None):
    c = case(cfg, variant)
    dev = {"logits": dc.to_device(c["logits"], cfg.dtype), "h": dc.to_device(c["h"], cfg.dtype),
           "emb": dc.to_device(c["emb"], cfg.dtype)}
    w = dc.CorrectorWeights.from_numpy(c["w"], cfg.dtype)
    return c, dev, w


@pytest.mark.parametrize("cfg", REPR_CASES, ids=lambda c: c.name)
def test_candidate_repr_and_pair_state(cfg):
    c, dev, w = _device_case(cfg)
    vals, ids = oracle.topk(f64(c["logits"], cfg), cfg.K)
    W = w64(c["w"], cfg)
    rep = oracle.candidate_repr(ids, f64(c["emb"], cfg), f64(c["h"], cfg), W)
    s = oracle.pair_state(f64(c["h"], cfg), W)
    uz, vz = dc.candidate_repr(dc.to_device(ids.astype(np.int32), "i32"), dev["emb"], dev["h"], w)
    wsp = dc.pair_state(dev["h"], w)
    torch.cuda.synchronize()
    assert_intermediate_close(uz.float().cpu().numpy(), rep["z"] @ W["U"].T, "uz")
    assert_intermediate_close(vz.float().cpu().numpy(), rep["z"] @ W["V"].T, "vz")
    assert_intermediate_close(wsp.cpu().numpy(), s @ W["W"].T, "W s")


@pytest.mark.parametrize("cfg", REPR_CASES + [wl.TINY.replace(K=64, V=128), SMALL_BF16.replace(K=3)],
                         ids=lambda c: f"{c.name}_K{c.K}")
@pytest.mark.parametrize("variant", [None, "delta_zero", "amplified"])
def test_score_transitions(cfg, variant):
    c, dev, w = _device_case(cfg, variant)
    W = w64(c["w"], cfg)
    vals, ids = oracle.topk(f64(c["logits"], cfg), cfg.K)
    rep = oracle.candidate_repr(ids, f64(c["emb"], cfg), f64(c["h"], cfg), W)
    s = oracle.pair_state(f64(c["h"], cfg), W)
    S_ref = oracle.transition_scores(rep["z"], s, vals, W)
    act = "bf16" if cfg.dtype == "bf16" else "f32"
    to_act = (lambda a: dc.to_device(wl.f32_to_bf16(a.astype(np.float32)), "bf16")) if act == "bf16" else \
        (lambda a: dc.to_device(a.astype(np.float32), "f32"))
    S = dc.score_transitions(to_act(rep["z"] @ W["U"].T), to_act(rep["z"] @ W["V"].T),
                             dc.to_device((s @ W["W"].T).astype(np.float32), "f32"),
                             dc.to_device(vals.astype(np.float32), "f32"), w)
    S = S.cpu().numpy()
    unary = np.broadcast_to(vals[:, 1:, None, :], S_ref.shape) if variant == "amplified" else None
    assert_scores_close(S, S_ref, unary=unary)
    if variant == "delta_zero":
        np.testing.assert_array_equal(S, np.broadcast_to(vals[:, 1:, None, :], S.shape).astype(np.float32))
