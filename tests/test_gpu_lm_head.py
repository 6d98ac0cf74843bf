"""Fused drafter output projection + top-K (dcoco_lm_head_topk, dcoco_cycle_lm) against the
float64 oracle.

The GPU forms fp32 logits (exact bf16 products, or tf32 operands for f32 inputs, summed in
fp32) and selects exactly on them; the oracle selects on exact float64 logits.  Two tokens
whose exact logits lie within the accumulation error of each other may therefore rank in
either order, so the comparison is:
  - the returned ids are distinct, in range, and ordered by the returned values (equal values
    by ascending id);
  - every returned value is within tol(v) of token v's exact logit;
  - wherever the GPU's token at a rank differs from the oracle's, the two exact logits are
    within tol of each other (a near-tie swap), and such swaps are rare.
tol(v) = rel * sum_k |h_k W_lm[v, k]| + 1e-6 with
  bf16 inputs: rel = 2 d 2^-24 (products are exact in fp32; d additions of relative
               rounding 2^-24 each, doubled for headroom);
  f32 inputs:  rel = 2^-9 + 2 d 2^-24 (tf32 keeps 10 mantissa bits of each operand, 2^-10
               relative per operand when truncated).
"""
import functools

import numpy as np
import pytest
import torch

import draft_correction_gb300 as dc
import oracle
import workloads as wl
from helpers import assert_scores_close, compare_walk, emb_table, f64, w64
from test_gpu_kernels import SMALL_BF16, SMALL_R256

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from draft_correction_gb300 import build
    build.build()
    dc.lib()
    yield
    dc.set_lm_pair(0)
    assert dc.device_status() == 0, "a kernel reported a timeout or a bad index"


def rel_tol(cfg):
    r = 2.0 * cfg.d * 2.0 ** -24
    return r if cfg.dtype == "bf16" else r + 2.0 ** -9


def lm_cfg(dtype, N, B, d, V, K):
    return wl.TINY.replace(name=f"lm_{dtype}_{N}x{B}_d{d}_V{V}_K{K}", N=N, B=B, d=d, E=d, V=V, K=K, dtype=dtype,
                           logit_sigma=3.0, base_seed=5)


@functools.lru_cache(maxsize=4)
def lm_inputs(cfg):
    return wl.hidden(cfg), wl.lm_head(cfg)


def exact_logits(h64, W, cfg, chunk=8192):
    """Exact float64 logits and sum_k |h_k W[v,k]| for a few rows; W (stored dtype) is widened
    one chunk of tokens at a time."""
    L = np.empty((h64.shape[0], W.shape[0]))
    A = np.empty_like(L)
    ah = np.abs(h64)
    for s in range(0, W.shape[0], chunk):
        Wc = f64(W[s:s + chunk], cfg)
        L[:, s:s + chunk] = oracle.lm_logits(h64, Wc)
        A[:, s:s + chunk] = ah @ np.abs(Wc).T
    return L, A


def check_rows(g_vals, g_ids, L, A, K, rel, max_swap_frac=0.02):
    """The comparison rule of this file on rows given by their exact logits L and magnitudes A."""
    vals_ref, ids_ref = oracle.topk(L, K)
    swaps = 0
    for i in range(L.shape[0]):
        gi = g_ids[i].astype(np.int64)
        gv = g_vals[i].astype(np.float64)
        assert len(set(gi.tolist())) == K and gi.min() >= 0 and gi.max() < L.shape[1], f"row {i}: ids {gi}"
        for j in range(K - 1):
            assert gv[j] > gv[j + 1] or (gv[j] == gv[j + 1] and gi[j] < gi[j + 1]), f"row {i}: order at {j}"
        tol = rel * A[i] + 1e-6
        err = np.abs(gv - L[i, gi])
        assert np.all(err <= tol[gi]), f"row {i}: value error {err.max():.3e} > tol {tol[gi][err.argmax()]:.3e}"
        for j in range(K):
            a, b = gi[j], ids_ref[i, j]
            if a != b:
                assert abs(L[i, a] - L[i, b]) <= tol[a] + tol[b], (
                    f"row {i} rank {j}: gpu token {a} ({L[i, a]:.6f}) vs oracle {b} ({L[i, b]:.6f})")
                swaps += 1
    assert swaps <= max(2, max_swap_frac * L.shape[0] * K), f"{swaps} near-tie swaps"
    return swaps


LM_CASES = [
    ("f32", 1, 4, 64, 1024, 3),       # the tiny configuration's shapes, tf32 path
    ("bf16", 1, 1, 64, 300, 1),       # one row, one partial vocabulary tile
    ("bf16", 2, 16, 200, 4097, 16),   # ragged k-block (200 = 3 x 64 + 8) and vocabulary tail
    ("bf16", 3, 43, 520, 2500, 33),   # two row tiles, K above 32
    ("bf16", 2, 150, 136, 5000, 64),  # three row tiles, K = 64 (two pipeline stages)
    ("bf16", 1, 520, 64, 777, 8),     # five row tiles: the last pair half empty
    ("f32", 2, 7, 100, 3333, 10),     # f32 with a ragged k-block
]


@pytest.mark.parametrize("dtype,N,B,d,V,K", LM_CASES, ids=[f"{c[0]}-{c[1]}x{c[2]}-d{c[3]}-V{c[4]}-K{c[5]}"
                                                           for c in LM_CASES])
def test_lm_head_topk_matches_oracle(dtype, N, B, d, V, K):
    cfg = lm_cfg(dtype, N, B, d, V, K)
    h, W = lm_inputs(cfg)
    vals, ids = dc.lm_head_topk(dc.to_device(h, dtype), dc.to_device(W, dtype), K)
    torch.cuda.synchronize()
    h64 = f64(h, cfg).reshape(N * B, d)
    L, A = exact_logits(h64, W, cfg)
    check_rows(vals.cpu().numpy().reshape(N * B, K), ids.cpu().numpy().reshape(N * B, K), L, A, K, rel_tol(cfg))


@pytest.mark.parametrize("shape", [(3, 43, 520, 2500, 16), (4, 32, 128, 3000, 16)], ids=["3-row-tiles", "4-row-tiles"])
def test_lm_head_topk_pairs_and_single_ctas_bit_identical(shape):
    """Each CTA accumulates its whole 128 x 256 tile in the same order (k ascending, 16 per MMA)
    whether it issues 128-row MMAs alone or 256-row MMAs with its pair, so the logits and the
    selection are bit-identical."""
    N, B, d, V, K = shape
    cfg = lm_cfg("bf16", N, B, d, V, K)
    h, W = lm_inputs(cfg)
    hd, Wd = dc.to_device(h, "bf16"), dc.to_device(W, "bf16")
    res = []
    try:
        for mode in (-1, 1):
            dc.set_lm_pair(mode)
            v, i = dc.lm_head_topk(hd, Wd, K)
            torch.cuda.synchronize()
            res.append((v.cpu().numpy(), i.cpu().numpy()))
    finally:
        dc.set_lm_pair(0)
    np.testing.assert_array_equal(res[1][1], res[0][1])
    np.testing.assert_array_equal(res[1][0], res[0][0])


PAIR_CASES = [
    (1, 1, 64, 300, 1),      # one row: the odd CTA of the pair holds only zero-filled rows
    (2, 16, 200, 4097, 16),  # one row tile, ragged k-block and vocabulary tail
    (3, 43, 520, 2500, 33),  # two row tiles: one full pair
    (1, 520, 64, 777, 8),    # five row tiles: three pairs, the last one half empty
    (2, 150, 136, 5000, 64), # three row tiles, K = 64
]


@pytest.mark.parametrize("mode", [1, -1], ids=["pairs", "one-cta"])
@pytest.mark.parametrize("N,B,d,V,K", PAIR_CASES, ids=[f"{c[0]}x{c[1]}-d{c[2]}-V{c[3]}-K{c[4]}" for c in PAIR_CASES])
def test_lm_head_topk_cta_pairs_and_single_ctas(N, B, d, V, K, mode):
    """CTA-pair MMAs (one 256-row MMA over two CTAs' shared memory) forced on, and forced off,
    against exact float64 logits under the rule of this file."""
    cfg = lm_cfg("bf16", N, B, d, V, K)
    h, W = lm_inputs(cfg)
    prev = dc.set_lm_pair(mode)
    try:
        vals, ids = dc.lm_head_topk(dc.to_device(h, "bf16"), dc.to_device(W, "bf16"), K)
        torch.cuda.synchronize()
    finally:
        dc.set_lm_pair(prev)
    h64 = f64(h, cfg).reshape(N * B, d)
    L, A = exact_logits(h64, W, cfg)
    check_rows(vals.cpu().numpy().reshape(N * B, K), ids.cpu().numpy().reshape(N * B, K), L, A, K, rel_tol(cfg))


def test_lm_head_topk_duplicate_rows_tie_to_lower_id():
    """Tokens with identical W_lm rows get bit-identical logits; the lower id ranks first."""
    cfg = lm_cfg("bf16", 1, 8, 128, 1500, 12)
    h, W = lm_inputs(cfg)
    W = W.copy()
    W[1000:1500] = W[0:500]   # token 1000 + j repeats token j
    vals, ids = dc.lm_head_topk(dc.to_device(h, "bf16"), dc.to_device(W, "bf16"), cfg.K)
    torch.cuda.synchronize()
    v, i = vals.cpu().numpy()[0], ids.cpu().numpy()[0]
    for r in range(cfg.B):
        for j in range(cfg.K):
            if i[r, j] < 500 and j + 1 < cfg.K:  # its twin has the same logit and comes right after it
                assert i[r, j + 1] == i[r, j] + 1000 and v[r, j + 1] == v[r, j], (r, j, i[r], v[r])


@functools.lru_cache(maxsize=1)
def headline_inputs():
    cfg = wl.HEADLINE
    return wl.hidden(cfg), wl.lm_head(cfg)


@pytest.mark.parametrize("mode", [0, -1], ids=["automatic", "one-cta"])
def test_lm_head_topk_headline_size(mode):
    """512 rows x V = 151936 x d = 4096 in the launch configuration the benchmark times (the
    automatic plan: CTA pairs), and with one-CTA MMAs: all rows for order and distinctness,
    sampled rows against exact float64 logits."""
    cfg = wl.HEADLINE
    h, W = headline_inputs()
    prev = dc.set_lm_pair(mode)
    try:
        vals, ids = dc.lm_head_topk(dc.to_device(h, "bf16"), dc.to_device(W, "bf16"), cfg.K)
        torch.cuda.synchronize()
    finally:
        dc.set_lm_pair(prev)
    g_v = vals.cpu().numpy().reshape(-1, cfg.K).astype(np.float64)
    g_i = ids.cpu().numpy().reshape(-1, cfg.K)
    assert np.all(np.diff(g_v, axis=1) <= 0)
    assert all(len(set(r.tolist())) == cfg.K for r in g_i)
    rows = [0, 1, 127, 128, 255, 300, 383, 511]
    h64 = f64(h, cfg).reshape(-1, cfg.d)[rows]
    L, A = exact_logits(h64, W, cfg)
    check_rows(g_v[rows], g_i[rows], L, A, cfg.K, rel_tol(cfg))


LM_CYCLES = [wl.TINY, SMALL_BF16, SMALL_R256]


@pytest.mark.parametrize("cfg", LM_CYCLES, ids=[c.name for c in LM_CYCLES])
def test_cycle_lm_matches_oracle(cfg):
    """dcoco_cycle_lm against oracle.cycle_lm (exact float64 logits).  Streams whose top-K ids
    equal the oracle's are compared in full like dcoco_cycle; a stream with a near-tie swap in
    its candidates is checked for that swap only."""
    h = wl.hidden(cfg)
    W_lm = wl.lm_head(cfg)
    emb = emb_table(cfg)
    w = wl.weights(cfg)
    W = w64(w, cfg)
    h64 = f64(h, cfg)
    ref = oracle.cycle_lm(h64, f64(W_lm, cfg), f64(emb, cfg), W, cfg.K)
    t = wl.verifier_tokens(cfg, ref["tokens"])
    ver = oracle.verify_greedy(ref["tokens"], t)

    cw = dc.CorrectorWeights.from_numpy(w, cfg.dtype)
    cyc = dc.Cycle(cw, cfg.N, cfg.B, cfg.K, cfg.V)
    out = cyc.run(None, dc.to_device(emb, cfg.dtype), dc.to_device(h, cfg.dtype), t=dc.to_device(t, "i32"),
                  W_lm=dc.to_device(W_lm, cfg.dtype))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items()}

    L, A = exact_logits(h64.reshape(-1, cfg.d), W_lm, cfg)
    check_rows(g["vals"].reshape(-1, cfg.K), g["ids"].reshape(-1, cfg.K), L, A, cfg.K, rel_tol(cfg))
    same = [n for n in range(cfg.N) if np.array_equal(g["ids"][n], ref["ids"][n])]
    assert len(same) >= cfg.N - max(1, cfg.N // 10)
    for n in same:
        assert_scores_close(g["S"][n][None], ref["S"][n][None])
        near = compare_walk(g["k_sel"][n][None], ref["k"][n][None], ref["S"][n][None], ref["vals"][n][None])
        if near == 0:
            np.testing.assert_array_equal(g["tokens"][n], ref["tokens"][n])
            assert g["accept_len"][n] == ver["accept_len"][n]
            np.testing.assert_array_equal(g["committed"][n], ver["committed"][n])


@pytest.mark.slow
def test_cycle_lm_headline_size():
    """dcoco_cycle_lm at the headline shapes (512 rows, V = 151936, d = 4096, CTA-pair MMAs):
    three sampled streams through the whole cycle against the oracle, whose top-K comes from
    exact float64 logits of those streams' rows.  A stream with a near-tie swap among its
    candidates is checked for that swap only (the rule of this file)."""
    cfg = wl.HEADLINE
    h, W_lm = headline_inputs()
    emb = emb_table(cfg)
    w = wl.weights(cfg)
    W = w64(w, cfg)
    sam = [0, cfg.N // 2, cfg.N - 1]
    h64 = f64(h[sam], cfg)
    L, A = exact_logits(h64.reshape(-1, cfg.d), W_lm, cfg)
    vals_r, ids_r = oracle.topk(L, cfg.K)
    vals_r = vals_r.reshape(len(sam), cfg.B, cfg.K)
    ids_r = ids_r.reshape(len(sam), cfg.B, cfg.K)
    uniq, inv = np.unique(ids_r, return_inverse=True)
    rep = oracle.candidate_repr(inv.reshape(ids_r.shape), f64(emb[uniq], cfg), h64, W)
    S_ref = oracle.transition_scores(rep["z"], oracle.pair_state(h64, W), vals_r, W)
    k_ref, tok_ref = oracle.select(S_ref, vals_r, ids_r)
    draft = np.zeros((cfg.N, cfg.B), dtype=np.int64)  # streams the oracle does not walk: any draft
    draft[sam] = tok_ref
    t = wl.verifier_tokens(cfg, draft)
    ver = oracle.verify_greedy(tok_ref, t[sam])

    cw = dc.CorrectorWeights.from_numpy(w, cfg.dtype)
    cyc = dc.Cycle(cw, cfg.N, cfg.B, cfg.K, cfg.V)
    out = cyc.run(None, dc.to_device(emb, cfg.dtype), dc.to_device(h, cfg.dtype), t=dc.to_device(t, "i32"),
                  W_lm=dc.to_device(W_lm, cfg.dtype))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy()[sam] for k, v in out.items()}

    check_rows(g["vals"].reshape(-1, cfg.K), g["ids"].reshape(-1, cfg.K), L, A, cfg.K, rel_tol(cfg))
    full = 0
    for i in range(len(sam)):
        if not np.array_equal(g["ids"][i], ids_r[i]):
            continue
        assert_scores_close(g["S"][i][None], S_ref[i][None])
        if compare_walk(g["k_sel"][i][None], k_ref[i][None], S_ref[i][None], vals_r[i][None]) == 0:
            np.testing.assert_array_equal(g["tokens"][i], tok_ref[i])
            assert g["accept_len"][i] == ver["accept_len"][i]
            np.testing.assert_array_equal(g["committed"][i], ver["committed"][i])
            full += 1
    assert full >= 2, f"only {full} of {len(sam)} sampled streams compared in full"
