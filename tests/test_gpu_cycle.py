"""Whole-cycle parity (a1..a6 through dcoco_cycle) against the float64 oracle.

Small configurations are compared in full.  At the full workload sizes (the launch
configuration the benchmark times) top-K is compared on every row of every stream and the
rest on a sample of streams that the oracle recomputes end to end.  Every point of the
streams x B x K sweep is compared, with greedy and with stochastic verification.
"""
import functools
import os

import numpy as np
import pytest
import torch

import draft_correction_gb300 as dc
import oracle
import workloads as wl
from conftest import GOLDEN
from helpers import assert_scores_close, case, compare_walk, emb_table, f64, oracle_topk_rows, w64
from test_gpu_kernels import SMALL_BF16, SMALL_R256, SMALL_R512

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from draft_correction_gb300 import build
    build.build()
    dc.lib()
    yield
    assert dc.device_status() == 0, "a kernel reported a timeout or a bad index"


def sample_streams(N):
    return list(range(N)) if N <= 4 else sorted({0, N // 2, N - 1})


def run_cycle_and_compare(cfg, variant=None, logits=None, mode=dc.VERIFY_GREEDY, use_table=False, inputs=None):
    """inputs, when given, holds this configuration's host tensors (logits, h, emb, w; q and u
    for stochastic verification; optionally "topk", the oracle's top-K of every row for some
    K' >= K, whose first K columns are the top-K)."""
    c = case(cfg, variant) if inputs is None else inputs
    logits = c["logits"] if logits is None else logits
    W = w64(c["w"], cfg)
    sam = sample_streams(cfg.N)
    # top-K parity on every row of every stream
    if c.get("topk") is not None and logits is c["logits"]:
        vals_r, ids_r = c["topk"][0][..., :cfg.K], c["topk"][1][..., :cfg.K]
    else:
        vals_r, ids_r = oracle_topk_rows(logits, cfg, cfg.K)
    vals, ids = vals_r[sam], ids_r[sam]
    h64 = f64(c["h"][sam], cfg)
    # the oracle sees exactly the embedding rows it gathers (never the whole table in float64)
    uniq, inv = np.unique(ids, return_inverse=True)
    rep = oracle.candidate_repr(inv.reshape(ids.shape), f64(c["emb"][uniq], cfg), h64, W)
    s = oracle.pair_state(h64, W)
    S_ref = oracle.transition_scores(rep["z"], s, vals, W)
    k_ref, tok_ref = oracle.select(S_ref, vals, ids)
    # the drafter's top-1 stands in as the draft of streams the oracle does not walk
    draft = np.stack([np.argmax(f64(logits[n], cfg), axis=1) for n in range(cfg.N)]).astype(np.int64)
    draft[sam] = tok_ref
    if mode == dc.VERIFY_GREEDY:
        t = wl.verifier_tokens(cfg, draft)
        ver_ref = oracle.verify_greedy(tok_ref, t[sam])
        extra = {"t": dc.to_device(t, "i32")}
    else:
        q = c["q"] if "q" in c else wl.verifier_probs(cfg)
        u = c["u"] if "u" in c else wl.uniforms(cfg)
        ver_ref = oracle.verify_stochastic(tok_ref, q[sam], u[sam])
        extra = {"q": dc.to_device(q, "f32"), "u": dc.to_device(u, "f32")}

    w = dc.CorrectorWeights.from_numpy(c["w"], cfg.dtype)
    cyc = dc.Cycle(w, cfg.N, cfg.B, cfg.K, cfg.V)
    emb = dc.to_device(c["emb"], cfg.dtype)
    table = dc.embedding_table(emb, w) if use_table else None
    out = cyc.run(dc.to_device(logits, cfg.dtype), emb, dc.to_device(c["h"], cfg.dtype), mode=mode, table=table,
                  **extra)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items()}

    np.testing.assert_array_equal(g["ids"], ids_r)
    np.testing.assert_array_equal(g["vals"].astype(np.float64), vals_r)
    unary = np.broadcast_to(vals[:, 1:, None, :], S_ref.shape) if variant == "amplified" else None
    assert_scores_close(g["S"][sam], S_ref, unary=unary)
    near = compare_walk(g["k_sel"][sam], k_ref, S_ref, vals)
    exact = [i for i, n in enumerate(sam) if np.array_equal(g["k_sel"][n], k_ref[i])]
    assert len(exact) >= len(sam) - near
    for i in exact:
        n = sam[i]
        np.testing.assert_array_equal(g["tokens"][n], tok_ref[i])
        if mode == dc.VERIFY_STOCHASTIC and (ver_ref["near_tie"][i] or g["near_tie"][n]):
            continue
        assert g["accept_len"][n] == ver_ref["accept_len"][i]
        assert g["n_commit"][n] == ver_ref["n_commit"][i]
        np.testing.assert_array_equal(g["committed"][n], ver_ref["committed"][i])
    return g, {"k": k_ref, "tokens": tok_ref, "S": S_ref}


@pytest.mark.parametrize("variant", [None, "delta_zero", "amplified"])
def test_cycle_tiny(variant):
    run_cycle_and_compare(wl.TINY, variant)


def test_cycle_tiny_zero_correction_is_drafter_argmax():
    g, _ = run_cycle_and_compare(wl.TINY, "delta_zero")
    np.testing.assert_array_equal(g["k_sel"], np.zeros_like(g["k_sel"]))  # sorted grid: argmax is candidate 0


def _worked_grid():
    rows = []
    for line in open(os.path.join(GOLDEN, "worked_example.txt")):
        p = line.split()
        if p and p[0] == "slot":
            rows.append([float(v) for v in p[3::2]])
    return rows


def test_cycle_worked_example_printed_logits():
    """The pages' B=4, K=3 grid as drafter logits with the output layer zeroed: the walk
    returns the per-slot argmax (These, keys, are, missing -> ids 0, 4, 7, 9)."""
    grid = _worked_grid()
    cfg = wl.TINY
    g, ref = run_cycle_and_compare(cfg, "delta_zero", logits=wl.grid_logits(grid, V=cfg.V))
    assert list(g["tokens"][0]) == [0, 4, 7, 9]


@pytest.mark.parametrize("cfg", [SMALL_BF16, SMALL_R256, SMALL_R512, SMALL_BF16.replace(K=1),
                                 SMALL_BF16.replace(name="small_h64", H=64),
                                 # 515 candidate rows, one slot each: five 128-row tiles, the
                                 # last one with 3 live rows whose slot lookups start at 512
                                 SMALL_BF16.replace(name="small_ragged", N=103, K=1),
                                 # the degenerate block of two slots (one transition per stream)
                                 # and the largest candidate count
                                 SMALL_BF16.replace(name="small_b2", B=2),
                                 SMALL_BF16.replace(name="small_k64", K=64)],
                         ids=lambda c: f"{c.name}_K{c.K}")
@pytest.mark.parametrize("variant", [None, "amplified"])
def test_cycle_small(cfg, variant):
    run_cycle_and_compare(cfg, variant)


@pytest.mark.parametrize("cfg", [SMALL_R256.replace(N=5), SMALL_BF16], ids=lambda c: c.name)
def test_cycle_small_stochastic(cfg):
    run_cycle_and_compare(cfg, None, mode=dc.VERIFY_STOCHASTIC)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [wl.QWEN3_8B, wl.HEADLINE], ids=lambda c: c.name)
def test_cycle_full_size(cfg):
    run_cycle_and_compare(cfg)


@functools.lru_cache(maxsize=1)
def sweep_inputs(n, b):
    """Host inputs of the sweep's (streams, B) point, shared by its three K and two verify modes:
    the oracle's top-16 of every row gives the top-4 and top-8 as its first columns."""
    cfg = wl.HEADLINE.replace(name=f"sweep_n{n}_b{b}", N=n, B=b)
    lg = wl.logits(cfg)
    return {"logits": lg, "h": wl.hidden(cfg), "emb": emb_table(cfg), "w": wl.weights(cfg),
            "q": wl.verifier_probs(cfg), "u": wl.uniforms(cfg), "topk": oracle_topk_rows(lg, cfg, max(wl.SWEEP_K))}


SWEEP_POINTS = [(n, b, k, mode) for n in wl.SWEEP_STREAMS for b in wl.SWEEP_B for k in wl.SWEEP_K
                for mode in (dc.VERIFY_GREEDY, dc.VERIFY_STOCHASTIC)]


@pytest.mark.slow
@pytest.mark.parametrize("n,b,k,mode", SWEEP_POINTS,
                         ids=[f"n{n}-b{b}-k{k}-{'greedy' if m == dc.VERIFY_GREEDY else 'stochastic'}"
                              for n, b, k, m in SWEEP_POINTS])
def test_cycle_sweep_points(n, b, k, mode):
    """All 42 (streams, B, K) points of the draft-correct-verify sweep, each with greedy and with
    stochastic verification, in the launch configuration the sweep benchmark times."""
    cfg = wl.HEADLINE.replace(name=f"sweep_n{n}_b{b}_k{k}", N=n, B=b, K=k)
    run_cycle_and_compare(cfg, mode=mode, inputs=sweep_inputs(n, b))


@pytest.mark.slow
def test_cycle_large():
    run_cycle_and_compare(wl.LARGE)


# ---------------------------------------------------------------------------
# The per-vocabulary table variant (LN(W_e Emb) precomputed once)
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("cfg", [wl.TINY, SMALL_BF16, SMALL_R256, SMALL_R512], ids=lambda c: c.name)
def test_embedding_table_rows(cfg):
    from helpers import assert_intermediate_close
    c = case(cfg)
    W = w64(c["w"], cfg)
    w = dc.CorrectorWeights.from_numpy(c["w"], cfg.dtype)
    table = dc.embedding_table(dc.to_device(c["emb"], cfg.dtype), w).float().cpu().numpy()
    rows = np.unique(np.random.default_rng(0).integers(0, cfg.V, 300))
    ref = oracle.layer_norm(f64(c["emb"][rows], cfg) @ W["W_e"].T)
    assert_intermediate_close(table[rows], ref, "LN(W_e Emb) table")


@pytest.mark.parametrize("cfg", [wl.TINY, SMALL_BF16, SMALL_R256, SMALL_R512], ids=lambda c: c.name)
@pytest.mark.parametrize("variant", [None, "amplified"])
def test_cycle_with_table(cfg, variant):
    run_cycle_and_compare(cfg, variant, use_table=True)


def test_cycle_with_table_headline():
    run_cycle_and_compare(wl.HEADLINE, use_table=True)


def test_cycle_on_caller_helper_streams_from_two_host_threads():
    """Two host threads, each with its own stream and its own pair of helper streams, enqueue
    cycles at the same time; each result equals the cycle run alone on the library's streams."""
    import threading
    cfg = SMALL_BF16
    c = case(cfg)
    w = dc.CorrectorWeights.from_numpy(c["w"], cfg.dtype)
    emb, lg, h = dc.to_device(c["emb"], cfg.dtype), dc.to_device(c["logits"], cfg.dtype), dc.to_device(c["h"], cfg.dtype)
    t = dc.to_device(wl.verifier_tokens(cfg, np.zeros((cfg.N, cfg.B), dtype=np.int64)), "i32")
    want = {k: v.cpu().numpy() for k, v in dc.Cycle(w, cfg.N, cfg.B, cfg.K, cfg.V).run(lg, emb, h, t=t).items()}
    torch.cuda.synchronize()
    got, errors = [None, None], []

    def worker(i):
        try:
            torch.cuda.set_device(lg.device)
            s, ha, hb = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
            dc.set_helper_streams(ha, hb)
            with torch.cuda.stream(s):
                cyc = dc.Cycle(w, cfg.N, cfg.B, cfg.K, cfg.V)
                for _ in range(5):
                    out = cyc.run(lg, emb, h, t=t)
                s.synchronize()
                got[i] = {k: v.cpu().numpy() for k, v in out.items()}
        except Exception as exc:  # reported below
            errors.append(exc)
        finally:
            dc.set_helper_streams(None, None)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for g in got:
        for k, v in want.items():
            np.testing.assert_array_equal(g[k], v, err_msg=k)
