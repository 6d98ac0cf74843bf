"""Seeded synthetic inputs for the DCOCO per-cycle hot path.

This module is the one place both sides of every parity check get their inputs
from: the float64 oracle and the CUDA library see the same bits.  It holds no
part of the method's arithmetic (no top-K, projection, normalisation, scoring,
selection or verification); only random draws, bf16 rounding of those draws, and
the shapes of the workloads.

The pages measure DCOCO on public benchmark suites with trained drafters and
target models, none of which is available here.  These configurations stand in
for them with the shapes the pages use (block B=16, top-K up to 16, Qwen3-8B
sized drafter d=4096 / vocabulary 151936, 1..128 concurrent streams) and simple
value distributions.  Every tensor is a pure function of (config, seed, tag).

bf16 tensors are carried as ``uint16`` bit patterns (numpy has no bf16 type);
``bf16_to_f64`` widens them exactly.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
from typing import Dict, Iterator, Optional

import numpy as np

# ----------------------------------------------------------------------------
# bf16 bit helpers (data conversion only)
# ----------------------------------------------------------------------------


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits.

    Inputs here are finite draws, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 view of a generated tensor ('bf16' bits or 'f32' values)."""
    if dtype == "bf16":
        return bf16_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Configurations
# ----------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    N: int            # concurrent streams (independent draft blocks)
    B: int            # draft slots per block
    K: int            # candidates kept per slot
    V: int            # vocabulary
    d: int            # drafter hidden size
    E: int            # token-embedding width
    r: int            # corrector width
    H: int            # transition-MLP hidden width
    dtype: str        # 'f32' or 'bf16' for every input tensor
    logit_sigma: float
    zipf_boost: bool  # add the +8 * rank^-1.1 boost on 32 random ids per slot
    base_seed: int
    weight_sigma: float = 0.02
    emb_sigma: float = 0.02

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)

    @property
    def rows(self) -> int:
        return self.N * self.B


TINY = Config("tiny", N=1, B=4, K=3, V=1024, d=64, E=64, r=32, H=64, dtype="f32",
              logit_sigma=2.0, zipf_boost=False, base_seed=0)
QWEN3_8B = Config("qwen3_8b_1stream", N=1, B=16, K=8, V=151936, d=4096, E=4096, r=256, H=512,
                  dtype="bf16", logit_sigma=3.0, zipf_boost=True, base_seed=1)
HEADLINE = QWEN3_8B.replace(name="headline_k16_32streams", K=16, N=32)
LARGE = Config("large_64streams", N=64, B=16, K=16, V=262144, d=8192, E=8192, r=512, H=1024,
               dtype="bf16", logit_sigma=3.0, zipf_boost=True, base_seed=1)

CONFIGS: Dict[str, Config] = {c.name: c for c in (TINY, QWEN3_8B, HEADLINE, LARGE)}

SWEEP_STREAMS = (1, 4, 8, 16, 32, 64, 128)
SWEEP_B = (8, 16)
SWEEP_K = (4, 8, 16)


def sweep_configs() -> Iterator[Config]:
    """The 42-point draft-correct-verify sweep on the headline shapes."""
    for n in SWEEP_STREAMS:
        for b in SWEEP_B:
            for k in SWEEP_K:
                yield HEADLINE.replace(name=f"sweep_n{n}_b{b}_k{k}", N=n, B=b, K=k)


def scaled(cfg: Config, **kw) -> Config:
    """A smaller case with the same distributions (for tests that must run in seconds)."""
    return cfg.replace(name=cfg.name + "_scaled", **kw)


# ----------------------------------------------------------------------------
# Seeded draws
# ----------------------------------------------------------------------------

TAG_LOGITS, TAG_HIDDEN, TAG_EMB, TAG_WEIGHTS, TAG_VERIFIER, TAG_PROBS, TAG_LM_HEAD = 1, 2, 3, 4, 5, 6, 7
_CHUNK = 1 << 24


def _rng(seed: int, tag: int, *sub: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(entropy=seed, spawn_key=(tag,) + sub)))


def _normal(seed: int, tag: int, sub: int, shape, sigma: float, dtype: str) -> np.ndarray:
    """sigma * N(0,1) draws stored in ``dtype`` (bf16 bits or float32).

    The flat tensor is cut into fixed blocks of 2^24 values; block b draws from its own
    generator (seed, tag, sub, b), so the result does not depend on how many threads fill it.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def fill(b):
        s = b * _CHUNK
        m = min(_CHUNK, n - s)
        buf = _rng(seed, tag, sub, b).standard_normal(m, dtype=np.float32)
        buf *= np.float32(sigma)
        out[s:s + m] = f32_to_bf16(buf) if dtype == "bf16" else buf

    blocks = range((n + _CHUNK - 1) // _CHUNK)
    if n > _CHUNK:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, blocks))
    else:
        for b in blocks:
            fill(b)
    return out.reshape(shape)


def stream_logits(cfg: Config, n: int) -> np.ndarray:
    """Drafter logits of stream n, shape [B, V]."""
    rng = _rng(cfg.base_seed + n, TAG_LOGITS)
    x = rng.standard_normal((cfg.B, cfg.V), dtype=np.float32) * np.float32(cfg.logit_sigma)
    if cfg.zipf_boost:
        # 32 distinct uniformly drawn ids per slot; the r-th gets +8 * r^-1.1.
        boost = (8.0 * np.arange(1, 33, dtype=np.float64) ** -1.1).astype(np.float32)
        for i in range(cfg.B):
            ids = rng.choice(cfg.V, size=32, replace=False)
            x[i, ids] += boost
    return f32_to_bf16(x) if cfg.dtype == "bf16" else x


def logits(cfg: Config) -> np.ndarray:
    """All streams' drafter logits, shape [N, B, V]."""
    out = np.empty((cfg.N, cfg.B, cfg.V), dtype=np.uint16 if cfg.dtype == "bf16" else np.float32)
    for n in range(cfg.N):
        out[n] = stream_logits(cfg, n)
    return out


def hidden(cfg: Config) -> np.ndarray:
    """Drafter hidden states h, shape [N, B, d], ~N(0,1)."""
    out = np.empty((cfg.N, cfg.B, cfg.d), dtype=np.uint16 if cfg.dtype == "bf16" else np.float32)
    for n in range(cfg.N):
        out[n] = _normal(cfg.base_seed + n, TAG_HIDDEN, 0, (cfg.B, cfg.d), 1.0, cfg.dtype)
    return out


def embedding(cfg: Config) -> np.ndarray:
    """Frozen token-embedding table, shape [V, E], ~N(0, emb_sigma^2)."""
    return _normal(cfg.base_seed, TAG_EMB, 0, (cfg.V, cfg.E), cfg.emb_sigma, cfg.dtype)


def lm_head(cfg: Config) -> np.ndarray:
    """Drafter output projection W_lm, shape [V, d], ~N(0, (logit_sigma / sqrt(d))^2).

    With h ~ N(0, 1) this gives logits h . W_lm[v] ~ N(0, logit_sigma^2), the spread of the
    stored-logit workloads (without their Zipf boost).
    """
    return _normal(cfg.base_seed, TAG_LM_HEAD, 0, (cfg.V, cfg.d), cfg.logit_sigma / np.sqrt(cfg.d), cfg.dtype)


WEIGHT_NAMES = ("W_e", "W_h", "W_f", "W_pair", "U", "V", "W", "u_a", "u_b", "b1", "w2", "b2")


def weight_shapes(cfg: Config) -> Dict[str, tuple]:
    r, H = cfg.r, cfg.H
    return {"W_e": (r, cfg.E), "W_h": (r, cfg.d), "W_f": (r, 2 * r), "W_pair": (r, 2 * cfg.d),
            "U": (H, r), "V": (H, r), "W": (H, r),
            "u_a": (H,), "u_b": (H,), "b1": (H,), "w2": (H,), "b2": (1,)}


def weights(cfg: Config, variant: Optional[str] = None) -> Dict[str, np.ndarray]:
    """Corrector weights, every entry ~N(0, weight_sigma^2).

    variant:
      None         -- as drawn
      'delta_zero' -- output layer zeroed (w2 = b2 = 0), so the correction vanishes
      'amplified'  -- w2 and b2 scaled by 100 so corrections move selections
    """
    w = {k: _normal(cfg.base_seed, TAG_WEIGHTS, i, s, cfg.weight_sigma, cfg.dtype)
         for i, (k, s) in enumerate(weight_shapes(cfg).items())}
    if variant == "delta_zero":
        for k in ("w2", "b2"):
            w[k] = np.zeros_like(w[k])
    elif variant == "amplified":
        for k in ("w2", "b2"):
            f = to_f64(w[k], cfg.dtype) * 100.0
            w[k] = f32_to_bf16(f.astype(np.float32)) if cfg.dtype == "bf16" else f.astype(np.float32)
    elif variant is not None:
        raise ValueError(f"unknown weight variant {variant!r}")
    return w


# ----------------------------------------------------------------------------
# Verifier-side inputs
# ----------------------------------------------------------------------------


def match_probability(j: int) -> float:
    """Probability that the synthetic verifier agrees with the draft at 1-based slot j."""
    return 0.8 * 0.93 ** (j - 1)


def verifier_tokens(cfg: Config, draft: np.ndarray) -> np.ndarray:
    """Synthetic greedy-verifier tokens t, shape [N, B+1] int32.

    Slot j (1-based) agrees with draft[:, j-1] with probability 0.8 * 0.93^(j-1); on a
    disagreement t_j is uniform over the other V-1 tokens.  t_{B+1} is uniform.
    """
    N, B = draft.shape
    t = np.empty((N, B + 1), dtype=np.int32)
    for n in range(N):
        rng = _rng(cfg.base_seed + n, TAG_VERIFIER)
        m = rng.random(B) < np.array([match_probability(j) for j in range(1, B + 1)])
        other = rng.integers(0, cfg.V - 1, size=B)
        for j in range(B):
            y = int(draft[n, j])
            t[n, j] = y if m[j] else (other[j] if other[j] < y else other[j] + 1)
        t[n, B] = rng.integers(0, cfg.V)
    return t


def verifier_probs(cfg: Config, sigma: float = 2.0) -> np.ndarray:
    """Synthetic verifier distributions q = softmax(N(0, sigma^2) logits), [N, B+1, V] float32.

    The softmax is evaluated in float64 and rounded to float32 once.
    """
    q = np.empty((cfg.N, cfg.B + 1, cfg.V), dtype=np.float32)
    for n in range(cfg.N):
        rng = _rng(cfg.base_seed + n, TAG_PROBS)
        x = rng.standard_normal((cfg.B + 1, cfg.V)) * sigma
        x -= x.max(axis=1, keepdims=True)
        e = np.exp(x)
        q[n] = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return q


def uniforms(cfg: Config, seed: int = 7) -> np.ndarray:
    """Accept/resample uniforms u in [0,1), [N, B+1, 2] float32, from Philox(seed).

    u[n, j, 0] decides acceptance at position j, u[n, j, 1] drives the residual
    (or, at position B, the bonus) draw.
    """
    rng = np.random.Generator(np.random.Philox(seed))
    return rng.random((cfg.N, cfg.B + 1, 2), dtype=np.float32)


# ----------------------------------------------------------------------------
# Hand-set candidate grids
# ----------------------------------------------------------------------------


def grid_logits(values, V: int = 1024, rest: float = -100.0) -> np.ndarray:
    """[1, B, V] float32 logits holding a hand-set B x K grid.

    Slot i's k-th value goes to token id i*K + k; every other id gets ``rest``, so a
    top-K over each slot returns exactly the grid.
    """
    B, K = len(values), len(values[0])
    x = np.full((1, B, V), rest, dtype=np.float32)
    for i, row in enumerate(values):
        for k, v in enumerate(row):
            x[0, i, i * K + k] = v
    return x
