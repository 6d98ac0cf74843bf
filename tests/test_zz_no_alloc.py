"""The allocation-free pair-state entry point.

dcoco_pair_state_noalloc serves callers that cannot allocate device memory (their own
allocator owns it all), so its scratch is a fixed 8 MiB array inside the library.  Its
results must match dcoco_pair_state's, call after call, through the C ABI, and the float64
oracle's W s_p.  This file is collected last so that a failure here comes after every other
test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import draft_correction_gb300 as dc
import oracle
import workloads as wl
from helpers import assert_intermediate_close, f64, w64

FIRST = wl.scaled(wl.HEADLINE, N=4, B=16, K=16, V=1000, d=4096, E=64, r=256, H=512)
SECOND = wl.scaled(wl.QWEN3_8B, N=3, B=7, K=8, V=1000, d=512, E=64, r=128, H=192)


def _run_both(cfg):
    w_h = wl.weights(cfg)
    h_h = wl.hidden(cfg)
    w = dc.CorrectorWeights.from_numpy(w_h, cfg.dtype)
    h = dc.to_device(h_h, cfg.dtype)
    want = dc.pair_state(h, w)
    out = torch.full((cfg.N, cfg.B - 1, cfg.H), float("nan"), dtype=torch.float32, device=h.device)
    got = dc.pair_state_noalloc(h, w, out=out)
    torch.cuda.synchronize()
    W = w64(w_h, cfg)
    ref = oracle.pair_state(f64(h_h, cfg), W) @ W["W"].T   # W s_p in float64
    return got.cpu().numpy(), want.cpu().numpy(), ref


@pytest.mark.gpu
def test_noalloc_pair_state_matches_workspace_version_twice_in_a_row():
    from draft_correction_gb300 import build
    build.build()
    for cfg in (FIRST, SECOND):
        got, want, ref = _run_both(cfg)
        assert np.isfinite(got).all()
        assert_intermediate_close(got, want.astype(np.float64), f"pair state without allocation ({cfg.name})")
        assert_intermediate_close(got, ref, f"pair state without allocation vs the oracle ({cfg.name})")
    assert dc.device_status() == 0


def test_noalloc_rejects_shapes_beyond_the_builtin_scratch():
    from draft_correction_gb300 import build
    build.build()
    L = dc.lib()
    fake = ctypes.c_void_p(0x10000)
    w = dc._Weights(dc.DCOCO_BF16, 4096, 4096, 512, 1024, *([0x20000] * len(dc.WEIGHT_FIELDS)))
    need = L.dcoco_pair_state_workspace_size(ctypes.byref(w), 256, 16)
    assert need > (8 << 20)
    rc = L.dcoco_pair_state_noalloc(fake, ctypes.byref(w), 256, 16, fake, None)
    assert rc == 3
    assert b"built-in" in L.dcoco_last_error()
