"""DCOCO per-cycle correction hot path on one GB300: Python binding of libdcoco.so.

Argument marshalling only.  Every step of the path runs in the library's CUDA kernels;
PyTorch supplies device memory and the current stream.  There is no CPU fallback: if
the library is not built, importing the binding works but every call raises.

Python names mirror the C ABI in include/dcoco.h without the ``dcoco_`` prefix.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdcoco.so")

DCOCO_F32, DCOCO_BF16 = 0, 1
VERIFY_GREEDY, VERIFY_STOCHASTIC = 0, 1
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA", 5: "TIMEOUT"}

WEIGHT_FIELDS = ("W_e", "W_h", "W_f", "W_pair", "U", "V", "W", "u_a", "u_b", "b1", "w2", "b2")


class DcocoError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dcoco: {STATUS.get(code, code)}: {msg}")
        self.code = code


class _Weights(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("d", ctypes.c_int), ("E", ctypes.c_int), ("r", ctypes.c_int),
                ("H", ctypes.c_int)] + [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_WP = ctypes.POINTER(_Weights)
_SIGNATURES = {
    "dcoco_version": ([], _I),
    "dcoco_last_error": ([], ctypes.c_char_p),
    "dcoco_device_status": ([_P, ctypes.POINTER(ctypes.c_uint32)], _I),
    "dcoco_selftest_timeout": ([ctypes.c_uint32, _P], _I),
    "dcoco_set_helper_streams": ([_P, _P], _I),
    "dcoco_set_topk_split": ([_I], _I),
    "dcoco_topk": ([_P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "dcoco_candidate_repr_workspace_size": ([_WP, _I, _I, _I], _Z),
    "dcoco_candidate_repr": ([_P, _P, _I, _P, _WP, _I, _I, _I, _P, _P, _P, _Z, _P], _I),
    "dcoco_pair_state_workspace_size": ([_WP, _I, _I], _Z),
    "dcoco_pair_state": ([_P, _WP, _I, _I, _P, _P, _Z, _P], _I),
    "dcoco_pair_state_noalloc": ([_P, _WP, _I, _I, _P, _P], _I),
    "dcoco_score_transitions": ([_P, _P, _P, _P, _WP, _I, _I, _I, _P, _P], _I),
    "dcoco_select": ([_P, _P, _P, _I, _I, _I, _P, _P, _P], _I),
    "dcoco_select_path": ([_P, _P, _P, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P], _I),
    "dcoco_verify": ([_I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "dcoco_verify_speculative": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "dcoco_cycle_workspace_size": ([_WP, _I, _I, _I], _Z),
    "dcoco_cycle": ([_P, _I, _P, _P, _WP, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z,
                     _P], _I),
    "dcoco_cycle_table": ([_P, _I, _P, _P, _WP, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                           _Z, _P], _I),
    "dcoco_lm_head_topk_workspace_size": ([_I, _I, _I, _I, _I], _Z),
    "dcoco_lm_head_topk": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _Z, _P], _I),
    "dcoco_set_lm_pair": ([_I], _I),
    "dcoco_cycle_lm_workspace_size": ([_WP, _I, _I, _I, _I], _Z),
    "dcoco_cycle_lm": ([_P, _I, _P, _P, _WP, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z,
                        _P], _I),
    "dcoco_embedding_table_bytes": ([_WP, _I], _Z),
    "dcoco_embedding_table": ([_P, _I, _WP, _P, _P], _I),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with draft_correction_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise DcocoError(rc, lib().dcoco_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("dcoco: tensors must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("dcoco: tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _ptr_logits(t: Optional[torch.Tensor]):
    """Logits may also be a host tensor: page-locked host memory is read by top-K through its
    device mapping; the library refuses pageable memory."""
    if t is None or t.is_cuda:
        return _ptr(t)
    if not t.is_contiguous():
        raise ValueError("dcoco: tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DCOCO_BF16
    if t.dtype == torch.float32:
        return DCOCO_F32
    raise ValueError(f"dcoco: unsupported dtype {t.dtype}")


def _act_dtype(code: int):
    return torch.bfloat16 if code == DCOCO_BF16 else torch.float32


def to_device(arr: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Upload a generated array: 'bf16' arrays are uint16 bit patterns, 'f32' float32."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)
    if dtype == "i32":
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32)).to(device)
    raise ValueError(dtype)


class CorrectorWeights:
    """Device tensors of the corrector plus the C struct that points at them."""

    def __init__(self, tensors: Dict[str, torch.Tensor]):
        self.t = dict(tensors)
        code = _dtype_code(self.t["W_e"])
        for k in WEIGHT_FIELDS:
            if _dtype_code(self.t[k]) != code:
                raise ValueError(f"dcoco: weight {k} has dtype {self.t[k].dtype}")
        self.dtype = code
        self.r, self.E = self.t["W_e"].shape
        self.d = self.t["W_h"].shape[1]
        self.H = self.t["U"].shape[0]
        self.c = _Weights(code, self.d, self.E, self.r, self.H, *[self.t[k].data_ptr() for k in WEIGHT_FIELDS])

    @classmethod
    def from_numpy(cls, w: Dict[str, np.ndarray], dtype: str, device="cuda") -> "CorrectorWeights":
        return cls({k: to_device(w[k], dtype, device) for k in WEIGHT_FIELDS})

    @property
    def ref(self):
        return ctypes.byref(self.c)

    @property
    def act_dtype(self):
        return _act_dtype(self.dtype)


def version() -> int:
    return lib().dcoco_version()


def device_status() -> int:
    """Read and clear the device status word (synchronises the current stream)."""
    bits = ctypes.c_uint32(0)
    rc = lib().dcoco_device_status(_stream(), ctypes.byref(bits))
    if rc not in (0, 5):
        _check(rc)
    return int(bits.value)


def selftest_timeout(polls: int) -> None:
    """Enqueue one bounded wait that gives up after `polls` polls and reports it in the status word."""
    _check(lib().dcoco_selftest_timeout(int(polls), _stream()))


def set_helper_streams(a: Optional[torch.cuda.Stream], b: Optional[torch.cuda.Stream]) -> None:
    """Caller-owned helper streams for the cycles enqueued by this host thread (None, None: the
    library's shared per-device streams)."""
    _check(lib().dcoco_set_helper_streams(ctypes.c_void_p(a.cuda_stream) if a is not None else None,
                                          ctypes.c_void_p(b.cuda_stream) if b is not None else None))


def set_topk_split(ctas_per_row: int) -> int:
    return lib().dcoco_set_topk_split(int(ctas_per_row))


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def topk(logits: torch.Tensor, K: int, vals=None, ids=None):
    """a1: top-K of every row of logits [N, B, V] -> vals [N, B, K] f32, ids [N, B, K] i32.
    logits may be a pinned host tensor (pass vals and ids on the GPU then)."""
    N, B, V = logits.shape
    vals = _empty((N, B, K), torch.float32, logits) if vals is None else vals
    ids = _empty((N, B, K), torch.int32, logits) if ids is None else ids
    _check(lib().dcoco_topk(_ptr_logits(logits), _dtype_code(logits), N, B, V, K, _ptr(vals), _ptr(ids), _stream()))
    return vals, ids


def candidate_repr(ids: torch.Tensor, emb: torch.Tensor, h: torch.Tensor, w: CorrectorWeights):
    """a2: uz = U z, vz = V z for every candidate, [N, B, K, H] in the weights' dtype."""
    N, B, K = ids.shape
    uz = _empty((N, B, K, w.H), w.act_dtype, ids)
    vz = _empty((N, B, K, w.H), w.act_dtype, ids)
    nbytes = lib().dcoco_candidate_repr_workspace_size(w.ref, N, B, K)
    ws = _empty((nbytes,), torch.uint8, ids)
    _check(lib().dcoco_candidate_repr(_ptr(ids), _ptr(emb), emb.shape[0], _ptr(h), w.ref, N, B, K, _ptr(uz), _ptr(vz),
                                      _ptr(ws), nbytes, _stream()))
    return uz, vz


def pair_state(h: torch.Tensor, w: CorrectorWeights):
    """a3: ws_pair[n, p] = W s_p, s_p = W_pair [h_p; h_{p+1}] -> [N, B-1, H] f32."""
    N, B, _ = h.shape
    out = _empty((N, B - 1, w.H), torch.float32, h)
    nbytes = lib().dcoco_pair_state_workspace_size(w.ref, N, B)
    ws = _empty((nbytes,), torch.uint8, h)
    _check(lib().dcoco_pair_state(_ptr(h), w.ref, N, B, _ptr(out), _ptr(ws), nbytes, _stream()))
    return out


def pair_state_noalloc(h: torch.Tensor, w: CorrectorWeights, out: Optional[torch.Tensor] = None):
    """a3 without a workspace: the library's built-in 8 MiB scratch array is used instead.

    For callers that cannot allocate device memory (their allocator owns all of it).  All
    calls share that array: calls that may overlap on the GPU must be ordered.  `out`
    ([N, B-1, H] f32) may be passed in so that the call itself allocates nothing.
    """
    N, B, _ = h.shape
    out = _empty((N, B - 1, w.H), torch.float32, h) if out is None else out
    _check(lib().dcoco_pair_state_noalloc(_ptr(h), w.ref, N, B, _ptr(out), _stream()))
    return out


def score_transitions(uz, vz, ws_pair, vals, w: CorrectorWeights):
    """a4: S [N, B-1, K, K] f32."""
    N, B, K = vals.shape
    S = _empty((N, B - 1, K, K), torch.float32, vals)
    _check(lib().dcoco_score_transitions(_ptr(uz), _ptr(vz), _ptr(ws_pair), _ptr(vals), w.ref, N, B, K, _ptr(S),
                                         _stream()))
    return S


def select(S, vals, ids):
    """a5: prefix-first walk -> k_sel [N, B] i32, tokens [N, B] i32."""
    N, B, K = vals.shape
    k_sel = _empty((N, B), torch.int32, vals)
    tokens = _empty((N, B), torch.int32, vals)
    _check(lib().dcoco_select(_ptr(S), _ptr(vals), _ptr(ids), N, B, K, _ptr(k_sel), _ptr(tokens), _stream()))
    return k_sel, tokens


PATH_GREEDY, PATH_DISCOUNTED = 0, 1


def select_path(S, vals, ids, rule: str = "greedy", lam: float = 0.75):
    """Path rules on the score grid: 'greedy' (the prefix-first walk), 'global_sum' (maximise the
    whole path's score) or 'geometric' (slot i weighted by lam^i) -> k_sel, tokens."""
    code, l = {"greedy": (PATH_GREEDY, 1.0), "global_sum": (PATH_DISCOUNTED, 1.0),
               "geometric": (PATH_DISCOUNTED, lam)}[rule]
    N, B, K = vals.shape
    k_sel = _empty((N, B), torch.int32, vals)
    tokens = _empty((N, B), torch.int32, vals)
    _check(lib().dcoco_select_path(_ptr(S), _ptr(vals), _ptr(ids), N, B, K, code, float(l), _ptr(k_sel),
                                   _ptr(tokens), _stream()))
    return k_sel, tokens


def verify(draft, t=None, q=None, u=None, mode: int = VERIFY_GREEDY):
    """a6: greedy (t [N, B+1]) or stochastic (q [N, B+1, V], u [N, B+1, 2]) verification."""
    N, B = draft.shape
    V = q.shape[2] if q is not None else 0
    out = {"accept_len": _empty((N,), torch.int32, draft), "committed": _empty((N, B + 1), torch.int32, draft),
           "n_commit": _empty((N,), torch.int32, draft), "near_tie": torch.zeros((N,), dtype=torch.int32,
                                                                                 device=draft.device)}
    _check(lib().dcoco_verify(mode, _ptr(draft), _ptr(t), _ptr(q), _ptr(u), N, B, V, _ptr(out["accept_len"]),
                              _ptr(out["committed"]), _ptr(out["n_commit"]), _ptr(out["near_tie"]), _stream()))
    return out


def verify_speculative(draft, p, q, u):
    """Speculative sampling with a draft distribution p [N, B, V]: q [N, B+1, V], u [N, B+1, 2]."""
    N, B = draft.shape
    V = q.shape[2]
    out = {"accept_len": _empty((N,), torch.int32, draft), "committed": _empty((N, B + 1), torch.int32, draft),
           "n_commit": _empty((N,), torch.int32, draft), "near_tie": torch.zeros((N,), dtype=torch.int32,
                                                                                 device=draft.device)}
    _check(lib().dcoco_verify_speculative(_ptr(draft), _ptr(p), _ptr(q), _ptr(u), N, B, V, _ptr(out["accept_len"]),
                                          _ptr(out["committed"]), _ptr(out["n_commit"]), _ptr(out["near_tie"]),
                                          _stream()))
    return out


def set_lm_pair(mode: int) -> int:
    return lib().dcoco_set_lm_pair(int(mode))


def lm_head_topk(h: torch.Tensor, W_lm: torch.Tensor, K: int, vals=None, ids=None, ws=None):
    """Fused drafter output projection + top-K: h [N, B, d], W_lm [V, d] (same dtype) ->
    vals [N, B, K] f32 (the fp32 logits), ids [N, B, K] i32; the logits are never stored."""
    N, B, d = h.shape
    V = W_lm.shape[0]
    code = _dtype_code(h)
    vals = _empty((N, B, K), torch.float32, h) if vals is None else vals
    ids = _empty((N, B, K), torch.int32, h) if ids is None else ids
    nbytes = lib().dcoco_lm_head_topk_workspace_size(code, N, B, V, K)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=h.device)
    _check(lib().dcoco_lm_head_topk(_ptr(h), _ptr(W_lm), code, N, B, d, V, K, _ptr(vals), _ptr(ids), _ptr(ws),
                                    ws.numel(), _stream()))
    return vals, ids


def embedding_table(emb, w):
    """b(v) = LN(W_e Emb[v]) for every token v: [V, r] in the activation dtype."""
    V = emb.shape[0]
    table = torch.empty((V, w.r), dtype=w.act_dtype, device=emb.device)
    _check(lib().dcoco_embedding_table(_ptr(emb), V, w.ref, _ptr(table), _stream()))
    return table


class Cycle:
    """Preallocated outputs and workspace for repeated whole cycles (a1..a6) of one shape."""

    def __init__(self, w: CorrectorWeights, N: int, B: int, K: int, V: int, device="cuda", keep_intermediates=True):
        self.w, self.N, self.B, self.K, self.V = w, N, B, K, V
        dev = torch.device(device)
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
        self.out = {"tokens": e((N, B), torch.int32), "accept_len": e((N,), torch.int32),
                    "committed": e((N, B + 1), torch.int32), "n_commit": e((N,), torch.int32),
                    "near_tie": torch.zeros((N,), dtype=torch.int32, device=dev)}
        if keep_intermediates:
            self.out.update({"vals": e((N, B, K), torch.float32), "ids": e((N, B, K), torch.int32),
                             "S": e((N, B - 1, K, K), torch.float32), "k_sel": e((N, B), torch.int32)})
        self.ws_bytes = lib().dcoco_cycle_workspace_size(w.ref, N, B, K)
        self.ws = e((self.ws_bytes,), torch.uint8)
        self.ws_lm = None

    def run(self, logits, emb, h, mode=VERIFY_GREEDY, t=None, q=None, u=None, table=None, W_lm=None):
        """One cycle.  With `table` (from embedding_table) the candidate rows come from it and
        `emb` is not read.  With `W_lm` [V, d] the logits are not an input: top-K is the fused
        output projection of `h` (dcoco_cycle_lm) and `logits` is not read."""
        o = self.out
        if W_lm is not None:
            # the size depends on the LM-head knobs (set_lm_pair): grow if needed
            nbytes = lib().dcoco_cycle_lm_workspace_size(self.w.ref, self.N, self.B, self.K, self.V)
            if self.ws_lm is None or self.ws_lm.numel() < nbytes:
                self.ws_lm = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=self.ws.device)
            ws = self.ws_lm
            _check(lib().dcoco_cycle_lm(_ptr(W_lm), self.V, _ptr(emb), _ptr(h), self.w.ref, self.N, self.B, self.K,
                                        mode, _ptr(t), _ptr(q), _ptr(u), _ptr(o.get("vals")), _ptr(o.get("ids")),
                                        _ptr(o.get("S")), _ptr(o.get("k_sel")), _ptr(o["tokens"]),
                                        _ptr(o["accept_len"]), _ptr(o["committed"]), _ptr(o["n_commit"]),
                                        _ptr(o["near_tie"]), _ptr(ws), ws.numel(), _stream()))
            return o
        fn = lib().dcoco_cycle_table if table is not None else lib().dcoco_cycle
        src = table if table is not None else emb
        _check(fn(_ptr_logits(logits), self.V, _ptr(src), _ptr(h), self.w.ref, self.N, self.B, self.K, mode,
                                 _ptr(t), _ptr(q), _ptr(u), _ptr(o.get("vals")), _ptr(o.get("ids")),
                                 _ptr(o.get("S")), _ptr(o.get("k_sel")), _ptr(o["tokens"]), _ptr(o["accept_len"]),
                                 _ptr(o["committed"]), _ptr(o["n_commit"]), _ptr(o["near_tie"]), _ptr(self.ws),
                                 self.ws_bytes, _stream()))
        return o


def cycle(logits, emb, h, w: CorrectorWeights, K: int, mode=VERIFY_GREEDY, t=None, q=None, u=None):
    """One whole correction cycle; returns a dict of output tensors."""
    N, B, V = logits.shape
    c = Cycle(w, N, B, K, V, device=logits.device)
    return c.run(logits, emb, h, mode, t, q, u)
