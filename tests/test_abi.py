"""The C ABI library loads, exports every declared entry point, and rejects bad arguments
on the host before touching the GPU (runs without a GPU)."""
import ctypes
import os
import re

import pytest

import draft_correction_gb300 as dc
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "dcoco.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dcoco_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from draft_correction_gb300 import build
    build.build()
    return dc.lib()


def test_header_declares_the_hot_path():
    names = declared_functions()
    for want in ("dcoco_topk", "dcoco_candidate_repr", "dcoco_pair_state", "dcoco_score_transitions",
                 "dcoco_select", "dcoco_verify", "dcoco_cycle"):
        assert want in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(declared_functions()) == set(dc._SIGNATURES), "binding signatures out of sync with the header"


def test_version_and_error_string(L):
    assert L.dcoco_version() >= 100
    assert isinstance(L.dcoco_last_error(), bytes)


FAKE = ctypes.c_void_p(0x10000)        # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x10008)


def _weights(dtype=dc.DCOCO_BF16, d=64, E=64, r=32, H=64, ptr=0x20000):
    return dc._Weights(dtype, d, E, r, H, *([ptr] * len(dc.WEIGHT_FIELDS)))


def test_topk_argument_errors(L):
    assert L.dcoco_topk(None, 1, 1, 4, 100, 3, FAKE, FAKE, None) == 1
    assert "logits" in L.dcoco_last_error().decode()
    assert L.dcoco_topk(FAKE, 7, 1, 4, 100, 3, FAKE, FAKE, None) == 2     # dtype
    assert L.dcoco_topk(FAKE, 1, 1, 4, 100, 65, FAKE, FAKE, None) == 1    # K > 64
    assert L.dcoco_topk(FAKE, 1, 1, 4, 10, 11, FAKE, FAKE, None) == 1     # K > V
    assert L.dcoco_topk(MISALIGNED, 1, 1, 4, 100, 3, FAKE, FAKE, None) == 1
    assert L.dcoco_topk(FAKE, 1, 300, 300, 100, 3, FAKE, FAKE, None) == 2  # too many rows


def test_weight_and_shape_errors(L):
    w = _weights(r=48)
    assert L.dcoco_candidate_repr(FAKE, FAKE, 100, FAKE, ctypes.byref(w), 1, 4, 3, FAKE, FAKE, FAKE, 1 << 30,
                                  None) == 2
    w = _weights(H=96)
    assert L.dcoco_pair_state(FAKE, ctypes.byref(w), 1, 4, FAKE, FAKE, 1 << 30, None) == 2
    w = _weights()
    w.U = None
    assert L.dcoco_score_transitions(FAKE, FAKE, FAKE, FAKE, ctypes.byref(w), 1, 4, 3, FAKE, None) == 1
    w = _weights()
    assert L.dcoco_score_transitions(FAKE, FAKE, FAKE, FAKE, ctypes.byref(w), 1, 1, 3, FAKE, None) == 1  # B < 2
    assert L.dcoco_select(FAKE, FAKE, FAKE, 1, 4, 0, FAKE, FAKE, None) == 1                             # K = 0


def test_workspace_errors(L):
    w = _weights()
    need = L.dcoco_candidate_repr_workspace_size(ctypes.byref(w), 2, 4, 3)
    assert need > 0
    assert L.dcoco_candidate_repr(FAKE, FAKE, 100, FAKE, ctypes.byref(w), 2, 4, 3, FAKE, FAKE, FAKE, need - 1,
                                  None) == 3
    assert L.dcoco_candidate_repr(FAKE, FAKE, 100, FAKE, ctypes.byref(w), 2, 4, 3, FAKE, FAKE, None, need,
                                  None) == 3
    need = L.dcoco_pair_state_workspace_size(ctypes.byref(w), 2, 4)
    assert L.dcoco_pair_state(FAKE, ctypes.byref(w), 2, 4, FAKE, FAKE, need - 1, None) == 3
    need = L.dcoco_cycle_workspace_size(ctypes.byref(w), 2, 4, 3)
    assert need >= L.dcoco_candidate_repr_workspace_size(ctypes.byref(w), 2, 4, 3)
    args = [FAKE, 100, FAKE, FAKE, ctypes.byref(w), 2, 4, 3, 0, FAKE, None, None] + [None] * 4 + [FAKE] * 4 + [None]
    assert L.dcoco_cycle(*args, FAKE, need - 1, None) == 3


def test_cycle_shape_errors(L):
    """The cycle's block shape is checked before anything is enqueued: 2 <= B <= 64,
    1 <= K <= 64, N >= 1 (DCOCO_ERR_INVALID_ARG)."""
    w = _weights()
    for N, B, K in [(0, 4, 3), (1, 1, 3), (1, 65, 3), (1, 4, 0), (1, 4, 65)]:
        args = [FAKE, 100, FAKE, FAKE, ctypes.byref(w), N, B, K, 0, FAKE, None, None] + [None] * 4 + [FAKE] * 4 + [None]
        assert L.dcoco_cycle(*args, FAKE, 1 << 30, None) == 1, (N, B, K)


def test_verify_errors(L):
    assert L.dcoco_verify(3, FAKE, FAKE, None, None, 1, 4, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert L.dcoco_verify(0, FAKE, None, None, None, 1, 4, 0, FAKE, FAKE, FAKE, None, None) == 1   # greedy, no t
    assert L.dcoco_verify(1, FAKE, None, FAKE, None, 1, 4, 10, FAKE, FAKE, FAKE, None, None) == 1  # no u
    assert L.dcoco_verify(0, FAKE, FAKE, None, None, 1, 65, 0, FAKE, FAKE, FAKE, None, None) == 1  # B > 64


def test_topk_split_knob(L):
    prev = L.dcoco_set_topk_split(3)
    assert L.dcoco_set_topk_split(prev) == 3


def test_select_path_argument_errors(L):
    fake = ctypes.c_void_p(0x10000)
    rc = L.dcoco_select_path(fake, fake, fake, 1, 4, 3, 7, ctypes.c_float(1.0), fake, fake, None)
    assert rc == 1 and b"path rule" in L.dcoco_last_error()
    for lam in (0.0, -0.5, 1.5, float("nan")):
        rc = L.dcoco_select_path(fake, fake, fake, 1, 4, 3, 1, ctypes.c_float(lam), fake, fake, None)
        assert rc == 1 and b"lambda" in L.dcoco_last_error()


def test_verify_speculative_argument_errors(L):
    fake = ctypes.c_void_p(0x10000)
    rc = L.dcoco_verify_speculative(fake, None, fake, fake, 2, 4, 10, fake, fake, fake, None, None)
    assert rc == 1 and b"p is NULL" in L.dcoco_last_error()
    rc = L.dcoco_verify_speculative(fake, fake, fake, fake, 2, 65, 10, fake, fake, fake, None, None)
    assert rc == 1


def test_table_argument_errors(L):
    fake = ctypes.c_void_p(0x10000)
    w = dc._Weights(dc.DCOCO_BF16, 4096, 4096, 256, 512, *([0x20000] * len(dc.WEIGHT_FIELDS)))
    assert L.dcoco_embedding_table_bytes(ctypes.byref(w), 151936) == 151936 * 256 * 2
    assert L.dcoco_embedding_table(None, 10, ctypes.byref(w), fake, None) == 1
    assert L.dcoco_embedding_table(fake, 10, ctypes.byref(w), None, None) == 1


def test_lm_head_topk_argument_errors(L):
    # h, W_lm, dtype, N, B, d, V, K, vals, ids, ws, ws_bytes, stream
    ok = dict(h=FAKE, W=FAKE, dt=dc.DCOCO_BF16, N=1, B=4, d=64, V=1000, K=8)

    def call(**kw):
        a = {**ok, **kw}
        return L.dcoco_lm_head_topk(a["h"], a["W"], a["dt"], a["N"], a["B"], a["d"], a["V"], a["K"], FAKE, FAKE,
                                    FAKE, 1 << 20, None)

    assert call(dt=7) == 2
    assert call(K=65) == 1 and call(K=0) == 1 and call(V=7) == 1
    assert call(d=12) == 1 and b"16 bytes" in L.dcoco_last_error()        # 24-byte bf16 rows
    assert call(dt=dc.DCOCO_F32, d=6) == 1                                  # 24-byte f32 rows
    assert call(h=None) == 1 and b"h is NULL" in L.dcoco_last_error()
    assert call(W=MISALIGNED) == 1 and b"W_lm" in L.dcoco_last_error()
    assert call(N=4096, B=17) == 2                                          # rows > 65535
    assert L.dcoco_lm_head_topk_workspace_size(7, 1, 4, 1000, 8) == 0
    assert L.dcoco_lm_head_topk_workspace_size(dc.DCOCO_BF16, 1, 4, 1000, 65) == 0


def test_lm_pair_knob(L):
    prev = L.dcoco_set_lm_pair(5)                # any positive value: always
    assert L.dcoco_set_lm_pair(-3) == 1          # any negative value: never
    assert L.dcoco_set_lm_pair(prev) == -1


def test_cycle_lm_argument_errors(L):
    w = _weights()
    args = [1000, FAKE, FAKE, ctypes.byref(w), 1, 4, 3, 0, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
            FAKE, FAKE, None, FAKE, 1 << 30, None]
    assert L.dcoco_cycle_lm(None, *args) == 1 and b"W_lm is NULL" in L.dcoco_last_error()
    assert L.dcoco_cycle_lm(MISALIGNED, *args) == 1 and b"W_lm" in L.dcoco_last_error()
    assert L.dcoco_cycle_lm_workspace_size(None, 1, 4, 3, 1000) == 0


def test_selftest_timeout_argument_errors(L):
    assert L.dcoco_selftest_timeout(0, None) == 1 and b"polls" in L.dcoco_last_error()
    assert L.dcoco_selftest_timeout(65537, None) == 1


def test_helper_streams_argument_errors(L):
    assert L.dcoco_set_helper_streams(FAKE, None) == 1 and b"two" in L.dcoco_last_error()
    assert L.dcoco_set_helper_streams(None, FAKE) == 1
    assert L.dcoco_set_helper_streams(FAKE, FAKE) == 1 and b"differ" in L.dcoco_last_error()
    assert L.dcoco_set_helper_streams(None, None) == 0
