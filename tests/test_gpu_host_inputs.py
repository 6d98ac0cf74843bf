"""Logits in page-locked host memory: top-K (alone and inside the cycle) reads them over the host
link through their mapped device address and must give exactly what it gives on a device copy;
pageable host memory is rejected before any launch."""
import numpy as np
import pytest
import torch

import draft_correction_gb300 as dc
import oracle
import workloads as wl
from helpers import case, f64
from test_gpu_kernels import SMALL_BF16, SMALL_R256

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from draft_correction_gb300 import build
    build.build()
    dc.lib()
    yield
    assert dc.device_status() == 0, "a kernel reported a timeout or a bad index"


def pinned(arr, dtype):
    t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16) if dtype == "bf16" \
        else torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    return t.pin_memory()


@pytest.mark.parametrize("cfg", [wl.TINY, SMALL_BF16, wl.HEADLINE], ids=lambda c: c.name)
def test_topk_from_pinned_host_logits(cfg):
    lg = case(cfg)["logits"] if cfg is not wl.HEADLINE else wl.logits(cfg)
    host = pinned(lg, cfg.dtype)
    dev = dc.to_device(lg, cfg.dtype)
    shape = (cfg.N, cfg.B, cfg.K)
    v_h = torch.empty(shape, dtype=torch.float32, device="cuda")
    i_h = torch.empty(shape, dtype=torch.int32, device="cuda")
    dc.topk(host, cfg.K, vals=v_h, ids=i_h)
    v_d, i_d = dc.topk(dev, cfg.K)
    torch.cuda.synchronize()
    assert torch.equal(i_h, i_d) and torch.equal(v_h, v_d)
    if cfg is not wl.HEADLINE:
        vals, ids = oracle.topk(f64(lg, cfg), cfg.K)
        np.testing.assert_array_equal(i_h.cpu().numpy(), ids)


def test_cycle_from_pinned_host_logits():
    cfg = SMALL_R256
    c = case(cfg)
    w = dc.CorrectorWeights.from_numpy(c["w"], cfg.dtype)
    emb = dc.to_device(c["emb"], cfg.dtype)
    h = dc.to_device(c["h"], cfg.dtype)
    t = torch.zeros((cfg.N, cfg.B + 1), dtype=torch.int32, device="cuda")
    a = dc.Cycle(w, cfg.N, cfg.B, cfg.K, cfg.V).run(dc.to_device(c["logits"], cfg.dtype), emb, h, t=t)
    a = {k: v.clone() for k, v in a.items()}
    b = dc.Cycle(w, cfg.N, cfg.B, cfg.K, cfg.V).run(pinned(c["logits"], cfg.dtype), emb, h, t=t)
    torch.cuda.synchronize()
    for k in ("ids", "vals", "S", "tokens", "committed"):
        assert torch.equal(a[k], b[k]), k


def test_pageable_host_logits_are_rejected_unless_mapped():
    """Pageable host memory is refused unless the driver reports a device mapping for it (as it
    may where the GPU reads host page tables directly); when accepted, the result is exact."""
    cfg = SMALL_BF16
    lg = torch.from_numpy(np.ascontiguousarray(case(cfg)["logits"]).view(np.int16)).view(torch.bfloat16)
    assert not lg.is_pinned()
    v = torch.empty((cfg.N, cfg.B, cfg.K), dtype=torch.float32, device="cuda")
    i = torch.empty((cfg.N, cfg.B, cfg.K), dtype=torch.int32, device="cuda")
    try:
        dc.topk(lg, cfg.K, vals=v, ids=i)
    except dc.DcocoError as e:
        assert "page-locked" in str(e)
        return
    torch.cuda.synchronize()
    _, ids = oracle.topk(f64(case(cfg)["logits"], cfg), cfg.K)
    np.testing.assert_array_equal(i.cpu().numpy(), ids)
