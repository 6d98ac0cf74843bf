"""The device-side failure path, taken without faulting anything (needs a GB300).

A bounded wait that gives up must leave a timeout bit in the status word and a usable
context; a token id outside [0, V) reaching the embedding gather must be reported and replaced
by row 0.  Neither case traps, hangs or touches memory out of bounds.
"""
import ctypes

import numpy as np
import pytest
import torch

import draft_correction_gb300 as dc
import oracle
import workloads as wl
from helpers import case, f64
from test_gpu_kernels import SMALL_BF16

pytestmark = pytest.mark.gpu

DEV_TIMEOUT_TMA, DEV_BAD_INDEX = 1, 8


@pytest.fixture(scope="module", autouse=True)
def built():
    from draft_correction_gb300 import build
    build.build()
    dc.lib()
    assert dc.device_status() == 0
    yield
    assert dc.device_status() == 0, "a status bit was left set"


def _status():
    bits = ctypes.c_uint32(0)
    rc = dc.lib().dcoco_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(bits))
    return rc, int(bits.value)


def test_bounded_wait_gives_up_and_reports_a_timeout():
    dc.selftest_timeout(64)
    rc, bits = _status()
    assert rc == 5, "DCOCO_ERR_TIMEOUT expected"
    assert bits == DEV_TIMEOUT_TMA
    assert b"bounded wait" in dc.lib().dcoco_last_error()
    # the word was cleared by the read, and the context still runs kernels correctly
    assert _status() == (0, 0)
    x = wl.f32_to_bf16(np.random.default_rng(5).normal(0, 3, (1, 4, 3000)).astype(np.float32))
    vals, ids = dc.topk(dc.to_device(x, "bf16"), 8)
    torch.cuda.synchronize()
    rv, ri = oracle.topk(wl.to_f64(x, "bf16"), 8)
    np.testing.assert_array_equal(ids.cpu().numpy(), ri)
    np.testing.assert_array_equal(vals.cpu().numpy().astype(np.float64), rv)
    assert _status() == (0, 0)


def test_out_of_range_token_id_is_reported_and_replaced_by_row_0():
    cfg = SMALL_BF16
    c = case(cfg)
    _, ids = oracle.topk(f64(c["logits"], cfg), cfg.K)
    ids = ids.astype(np.int32)
    bad = ids.copy()
    bad[0, 0, 0] = cfg.V + 5
    bad[-1, 1, cfg.K - 1] = -1
    fixed = bad.copy()
    fixed[0, 0, 0] = 0
    fixed[-1, 1, cfg.K - 1] = 0
    w = dc.CorrectorWeights.from_numpy(c["w"], cfg.dtype)
    emb = dc.to_device(c["emb"], cfg.dtype)
    h = dc.to_device(c["h"], cfg.dtype)
    uz_bad, vz_bad = dc.candidate_repr(dc.to_device(bad, "i32"), emb, h, w)
    rc, bits = _status()
    assert rc == 0, "an out-of-range id is not a timeout"
    assert bits == DEV_BAD_INDEX
    uz_ok, vz_ok = dc.candidate_repr(dc.to_device(fixed, "i32"), emb, h, w)
    torch.cuda.synchronize()
    assert _status() == (0, 0)
    # the projection is deterministic: the substituted rows give bit-identical results
    assert torch.equal(uz_bad, uz_ok) and torch.equal(vz_bad, vz_ok)
