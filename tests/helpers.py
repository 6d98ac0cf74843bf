"""Shared test plumbing: seeded cases, uploads, and the comparison rules.

Tolerances (floating point):
  transition scores   |gpu - ref| <= 2e-2 + 1e-2 |ref|   (the stated bar for bf16 inputs
                      with fp32 accumulation; applied to the fp32/tf32 tiny case as well)
  intermediates       |gpu - ref| <= 0.03 rms(ref) + 0.02 |ref|  (uz, vz, W s): bf16 storage
                      of b, z and the outputs each contribute ~2^-9 relative error, tf32
                      operands ~2^-11; the bound leaves ~5x headroom over that budget
Selections must equal the oracle's except after a step whose oracle top-2 margin is at
most 5e-2; ids, candidate indices, accept lengths and committed tokens are bit-exact.
"""
from __future__ import annotations

import concurrent.futures
import functools
import os

import numpy as np

import oracle
import workloads as wl

SCORE_ATOL, SCORE_RTOL = 2e-2, 1e-2
MARGIN = 5e-2


def assert_scores_close(gpu, ref, what="S", unary=None):
    """Stated bound |gpu - ref| <= 2e-2 + 1e-2 |ref|.

    With `unary` (l_{p+1}(b) broadcast to S's shape) the relative part applies to the
    magnitudes of the two summands, |l| + |Delta|.  Used only for the stress variant whose
    output layer is scaled by 100: there Delta reaches ~17 and the bf16 storage of the
    per-candidate first-layer blocks (2^-9 relative) alone moves S by ~1e-3 |Delta|.
    """
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    scale = np.abs(ref) if unary is None else np.abs(unary) + np.abs(ref - unary)
    bound = SCORE_ATOL + SCORE_RTOL * scale
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")


def assert_intermediate_close(gpu, ref, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(gpu - ref)
    bound = 0.03 * rms + 0.02 * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst err {err.max():.3e}, "
                           f"rms(ref) {rms:.3e}")


def compare_walk(k_gpu, k_ref, S_ref, vals_ref):
    """Walk parity with the margin rule.  Returns the number of streams that diverged at a
    near-tie (allowed); raises on any other disagreement."""
    N, B = k_ref.shape
    near = 0
    for n in range(N):
        for i in range(B):
            if k_gpu[n, i] == k_ref[n, i]:
                continue
            row = vals_ref[n, 0] if i == 0 else S_ref[n, i - 1, k_ref[n, i - 1]]
            srt = np.sort(oracle.canonical(row))[::-1]
            margin = srt[0] - srt[1] if len(srt) > 1 else np.inf
            assert margin <= MARGIN, f"stream {n} slot {i}: gpu {k_gpu[n, i]} vs oracle {k_ref[n, i]}, margin {margin}"
            # the gpu's choice must also be a maximiser within the margin
            assert oracle.canonical(row)[k_gpu[n, i]] >= srt[0] - MARGIN
            near += 1
            break
    return near


@functools.lru_cache(maxsize=2)
def _emb_table(V, E, dtype, seed, sigma):
    return wl.embedding(wl.TINY.replace(V=V, E=E, dtype=dtype, base_seed=seed, emb_sigma=sigma))


def emb_table(cfg: wl.Config):
    """The embedding table depends only on (V, E, dtype, seed, sigma): shared across configs."""
    return _emb_table(cfg.V, cfg.E, cfg.dtype, cfg.base_seed, cfg.emb_sigma)


@functools.lru_cache(maxsize=6)
def case(cfg: wl.Config, variant=None):
    """Host inputs of one configuration (cached per test session)."""
    return {"logits": wl.logits(cfg), "h": wl.hidden(cfg), "emb": emb_table(cfg), "w": wl.weights(cfg, variant)}


def f64(arr, cfg):
    return wl.to_f64(arr, cfg.dtype)


def w64(w, cfg):
    return {k: f64(v, cfg) for k, v in w.items()}


def oracle_topk_rows(logits, cfg: wl.Config, K: int):
    """oracle.topk over every row of [N, B, V] logits, rows split over host threads (each
    thread runs the oracle itself on its own rows; numpy's sort releases the GIL)."""
    x = np.asarray(logits).reshape(-1, logits.shape[-1])
    n = x.shape[0]
    starts = list(range(0, n, 32))  # 32 rows per call bounds the float64 copies in flight

    def part(s0):
        return oracle.topk(f64(x[s0:s0 + 32], cfg), K)

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        parts = list(ex.map(part, starts))
    vals = np.concatenate([p[0] for p in parts]).reshape(logits.shape[:-1] + (K,))
    ids = np.concatenate([p[1] for p in parts]).reshape(logits.shape[:-1] + (K,))
    return vals, ids
