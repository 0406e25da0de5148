"""Python binding of libstill.so (the C ABI declared in include/still.h).

Argument marshalling only: tensors are checked for dtype, shape, device and
contiguity, and their device pointers are handed to the library; every step of
the layer runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as ct
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libstill.so")

# still_metric (include/still.h): routing metrics of the chunk selection
METRICS = {"self_saliency": 0, "diagonal": 1, "qk": 2, "key_norm": 3, "uniform": 4, "random": 5}

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "CUDA error",
          4: "device wait timed out", 5: "index out of bounds", 6: "workspace too small"}


class StillError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({code})")
        self.code = code


class Shape(ct.Structure):
    _fields_ = [("B", ct.c_int), ("Hq", ct.c_int), ("Hkv", ct.c_int), ("N", ct.c_int),
                ("d", ct.c_int), ("d_f", ct.c_int)]


class DecodeStateC(ct.Structure):
    _fields_ = [(n, ct.c_void_p) for n in
                ("K", "V", "slot_pos", "slot_cnt", "slot_score", "S", "z", "score_ring", "t", "status")]


class KernelTime(ct.Structure):
    _fields_ = [("name", ct.c_char * 48), ("launches", ct.c_int), ("ms", ct.c_double)]


_lib = None

# The exported functions and their C signatures (include/still.h).
SIGNATURES = {
    "still_status_string": (ct.c_char_p, [ct.c_int]),
    "still_lambda": (ct.c_int, [ct.c_int, ct.c_int, ct.c_int]),
    "still_score": (ct.c_int, [ct.POINTER(Shape), ct.c_void_p, ct.c_void_p, ct.c_int, ct.c_void_p,
                               ct.c_void_p]),
    "still_select": (ct.c_int, [ct.POINTER(Shape), ct.c_void_p, ct.c_int, ct.c_int, ct.c_int, ct.c_int,
                                ct.c_void_p, ct.c_void_p]),
    "still_score_metric": (ct.c_int, [ct.POINTER(Shape), ct.c_void_p, ct.c_void_p, ct.c_int, ct.c_int, ct.c_int,
                                      ct.c_int, ct.c_int, ct.c_uint64, ct.c_void_p, ct.c_void_p]),
    "still_npmap": (ct.c_int, [ct.c_void_p, ct.c_longlong, ct.c_int, ct.c_void_p, ct.c_int, ct.c_void_p,
                               ct.c_void_p]),
    "still_prefill_workspace_size": (ct.c_size_t, [ct.POINTER(Shape), ct.c_int, ct.c_int, ct.c_int,
                                                   ct.c_int]),
    "still_prefill": (ct.c_int, [ct.POINTER(Shape), ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_void_p,
                                 ct.c_int, ct.c_int, ct.c_int, ct.c_int, ct.c_void_p, ct.c_void_p,
                                 ct.c_void_p, ct.c_size_t, ct.POINTER(DecodeStateC), ct.c_void_p]),
    "still_prefill_routed": (ct.c_int, [ct.POINTER(Shape), ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_void_p,
                                        ct.c_int, ct.c_int, ct.c_int, ct.c_int, ct.c_int, ct.c_uint64,
                                        ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_size_t, ct.c_void_p]),
    "still_prefill_gated": (ct.c_int, [ct.POINTER(Shape), ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_void_p,
                                       ct.c_void_p, ct.c_int, ct.c_int, ct.c_int, ct.c_int, ct.c_void_p,
                                       ct.c_void_p, ct.c_void_p, ct.c_size_t, ct.POINTER(DecodeStateC), ct.c_void_p]),
    "still_decode_step_gated": (ct.c_int, [ct.POINTER(Shape), ct.POINTER(DecodeStateC), ct.c_void_p, ct.c_void_p,
                                           ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_int, ct.c_int, ct.c_int,
                                           ct.c_int, ct.c_void_p, ct.c_void_p]),
    "still_backward_workspace_size": (ct.c_size_t, [ct.POINTER(Shape), ct.c_int, ct.c_int, ct.c_int, ct.c_int]),
    "still_backward": (ct.c_int, [ct.POINTER(Shape), ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_void_p,
                                  ct.c_int, ct.c_int, ct.c_int, ct.c_int, ct.c_void_p, ct.c_void_p,
                                  ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_void_p,
                                  ct.c_void_p, ct.c_size_t, ct.c_void_p]),
    "still_prefill_noalloc_max_bytes": (ct.c_size_t, []),
    "still_prefill_noalloc": (ct.c_int, [ct.POINTER(Shape), ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_void_p,
                                         ct.c_int, ct.c_int, ct.c_int, ct.c_int, ct.c_void_p, ct.c_void_p,
                                         ct.POINTER(DecodeStateC), ct.c_void_p]),
    "still_decode_state_init": (ct.c_int, [ct.POINTER(Shape), ct.POINTER(DecodeStateC), ct.c_int, ct.c_int,
                                           ct.c_int, ct.c_int, ct.c_void_p]),
    "still_decode_step": (ct.c_int, [ct.POINTER(Shape), ct.POINTER(DecodeStateC), ct.c_void_p, ct.c_void_p,
                                     ct.c_void_p, ct.c_void_p, ct.c_int, ct.c_int, ct.c_int, ct.c_int,
                                     ct.c_void_p, ct.c_void_p]),
    "still_read_status": (ct.c_int, [ct.c_void_p, ct.c_void_p, ct.POINTER(ct.c_int32)]),
    "still_debug_set_wait_limit": (None, [ct.c_longlong]),
    "still_timing_enable": (None, [ct.c_int]),
    "still_timing_read": (ct.c_int, [ct.POINTER(KernelTime), ct.c_int]),
}


def lib():
    """Load libstill.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libstill.so not built ({LIB_PATH}); run "
                              "python -m linear_attention_linearization_gb300.build")
        L = ct.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(code, what):
    if code != 0:
        raise StillError(code, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ct.c_void_p(stream.cuda_stream)


def _ptr(t, dtype, what):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return ct.c_void_p(t.data_ptr())


def lam_of(W, m, T_max):
    return lib().still_lambda(W, m, T_max)


def shape_of(q, k, Wf):
    B, Hq, N, d = q.shape
    return Shape(B, Hq, k.shape[1], N, d, Wf.shape[1])


def score(q, k, W, scores=None, stream=None):
    """Self-Saliency scores [B, Hkv, N] (fp32) of bf16 q [B,Hq,N,d], k [B,Hkv,N,d]."""
    B, Hq, N, d = q.shape
    sh = Shape(B, Hq, k.shape[1], N, d, d)
    if scores is None:
        scores = torch.empty((B, k.shape[1], N), dtype=torch.float32, device=q.device)
    _check(lib().still_score(ct.byref(sh), _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), W,
                             _ptr(scores, torch.float32, "scores"), _stream(stream)), "still_score")
    return scores


def select(scores, Hq, d, W, C, m, T_max, sel_idx=None, stream=None):
    """Top-lambda of each completed chunk: int32 [B, Hkv, T_max, lambda]."""
    B, Hkv, N = scores.shape
    lam = lam_of(W, m, T_max)
    sh = Shape(B, Hq, Hkv, N, d, d)
    if sel_idx is None:
        sel_idx = torch.empty((B, Hkv, T_max, max(lam, 0)), dtype=torch.int32, device=scores.device)
    _check(lib().still_select(ct.byref(sh), _ptr(scores, torch.float32, "scores"), W, C, m, T_max,
                              _ptr(sel_idx, torch.int32, "sel_idx"), _stream(stream)), "still_select")
    return sel_idx


def score_metric(q, k, W, C, m, T_max, metric, seed=0, B=None, Hq=None, Hkv=None, N=None, d=None,
                 scores=None, stream=None):
    """Scores [B, Hkv, N] (fp32) of one routing metric (a name of METRICS).  q and
    k are bf16 [B,Hq,N,d] / [B,Hkv,N,d]; either may be None for the metrics that do
    not read it, and the sizes are then taken from the keyword arguments."""
    mid = METRICS[metric]
    if q is not None:
        B, Hq, N, d = q.shape
    if k is not None:
        B, Hkv, N, d = k.shape
    sh = Shape(B, Hq, Hkv, N, d, d)
    dev = q.device if q is not None else (k.device if k is not None else torch.device("cuda"))
    if scores is None:
        scores = torch.empty((B, Hkv, N), dtype=torch.float32, device=dev)
    _check(lib().still_score_metric(ct.byref(sh), _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), W, C,
                                    m, T_max, mid, ct.c_uint64(seed), _ptr(scores, torch.float32, "scores"),
                                    _stream(stream)), "still_score_metric")
    return scores


def npmap(x, Wf, stream=None):
    """NP-Map of the rows of bf16 x [..., d] with fp32 Wf [d, d_f] -> fp32 [..., d_f]."""
    d, df = Wf.shape
    rows = x.numel() // d
    phi = torch.empty(x.shape[:-1] + (df,), dtype=torch.float32, device=x.device)
    _check(lib().still_npmap(_ptr(x, torch.bfloat16, "x"), rows, d, _ptr(Wf, torch.float32, "Wf"), df,
                             _ptr(phi, torch.float32, "phi"), _stream(stream)), "still_npmap")
    return phi


def workspace_size(q, k, Wf, W, C, m, T_max):
    sh = shape_of(q, k, Wf)
    return lib().still_prefill_workspace_size(ct.byref(sh), W, C, m, T_max)


class DecodeState:
    """Caller-owned decode state of B sequences (device tensors), see still.h."""

    def __init__(self, B, Hkv, d, df, C, m, device="cuda"):
        dev = torch.device(device)
        self.B, self.Hkv, self.d, self.df, self.C, self.m = B, Hkv, d, df, C, m
        self.K = torch.zeros((B, Hkv, m, d), dtype=torch.bfloat16, device=dev)
        self.V = torch.zeros((B, Hkv, m, d), dtype=torch.bfloat16, device=dev)
        self.slot_pos = torch.full((B, Hkv, m), -1, dtype=torch.int32, device=dev)
        self.slot_cnt = torch.zeros((B, Hkv, m), dtype=torch.int32, device=dev)
        self.slot_score = torch.zeros((B, Hkv, m), dtype=torch.float32, device=dev)
        self.S = torch.zeros((B, Hkv, df, d), dtype=torch.float32, device=dev)
        self.z = torch.zeros((B, Hkv, df), dtype=torch.float32, device=dev)
        self.score_ring = torch.zeros((B, Hkv, C), dtype=torch.float32, device=dev)
        self.t = torch.zeros((B, Hkv), dtype=torch.int64, device=dev)
        self.status = torch.zeros((4,), dtype=torch.int32, device=dev)

    def c_struct(self):
        return DecodeStateC(*(t.data_ptr() for t in (self.K, self.V, self.slot_pos, self.slot_cnt,
                                                       self.slot_score, self.S, self.z, self.score_ring,
                                                       self.t, self.status)))

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in (self.K, self.V, self.slot_pos, self.slot_cnt,
                                                          self.slot_score, self.S, self.z, self.score_ring,
                                                          self.t))

    def read_status(self, stream=None):
        v = ct.c_int32(0)
        _check(lib().still_read_status(ct.c_void_p(self.status.data_ptr()), _stream(stream), ct.byref(v)),
               "still_read_status")
        return v.value


def prefill(q, k, v, Wf, W, C, m, T_max, out=None, sel_idx=None, workspace=None, export_state=None,
            stream=None):
    """Chunk-parallel prefill of one layer.  Returns (out [B,Hq,N,d] bf16, sel_idx)."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    lam = lam_of(W, m, T_max)
    sh = shape_of(q, k, Wf)
    if out is None:
        out = torch.empty_like(q)
    if sel_idx is None:
        sel_idx = torch.empty((B, Hkv, T_max, max(lam, 0)), dtype=torch.int32, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, torch.uint8, "workspace"), workspace.numel()
    st = ct.byref(export_state.c_struct()) if export_state is not None else None
    _check(lib().still_prefill(ct.byref(sh), _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"),
                               _ptr(v, torch.bfloat16, "v"), _ptr(Wf, torch.float32, "Wf"), W, C, m, T_max,
                               _ptr(out, torch.bfloat16, "out"),
                               _ptr(sel_idx, torch.int32, "sel_idx") if sel_idx.numel() else None,
                               ws_ptr, ws_bytes, st, _stream(stream)), "still_prefill")
    return out, sel_idx


def prefill_routed(q, k, v, Wf, W, C, m, T_max, metric, seed=0, out=None, sel_idx=None, workspace=None,
                   stream=None):
    """The prefill with the chunk selection ranked by a routing metric (a name of
    METRICS).  Returns (out [B,Hq,N,d] bf16, sel_idx)."""
    B, Hq, N, d = q.shape
    lam = lam_of(W, m, T_max)
    sh = shape_of(q, k, Wf)
    if out is None:
        out = torch.empty_like(q)
    if sel_idx is None:
        sel_idx = torch.empty((B, k.shape[1], T_max, max(lam, 0)), dtype=torch.int32, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, torch.uint8, "workspace"), workspace.numel()
    _check(lib().still_prefill_routed(ct.byref(sh), _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"),
                                      _ptr(v, torch.bfloat16, "v"), _ptr(Wf, torch.float32, "Wf"), W, C, m, T_max,
                                      METRICS[metric], ct.c_uint64(seed), _ptr(out, torch.bfloat16, "out"),
                                      _ptr(sel_idx, torch.int32, "sel_idx") if sel_idx.numel() else None,
                                      ws_ptr, ws_bytes, _stream(stream)), "still_prefill_routed")
    return out, sel_idx


def prefill_gated(q, k, v, gate, Wf, W, C, m, T_max, out=None, sel_idx=None, workspace=None, export_state=None,
                  stream=None):
    """The layer with a per-channel sigmoid gate on the linear branch's numerator:
    gate [B,Hq,N,d] bf16 holds the pre-activations (see still_prefill_gated).
    export_state (optional DecodeState) receives the state still_decode_step_gated
    continues from."""
    B, Hq, N, d = q.shape
    if tuple(gate.shape) != tuple(q.shape):
        raise ValueError("gate must have the shape of q")
    lam = lam_of(W, m, T_max)
    sh = shape_of(q, k, Wf)
    if out is None:
        out = torch.empty_like(q)
    if sel_idx is None:
        sel_idx = torch.empty((B, k.shape[1], T_max, max(lam, 0)), dtype=torch.int32, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, torch.uint8, "workspace"), workspace.numel()
    _check(lib().still_prefill_gated(ct.byref(sh), _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"),
                                     _ptr(v, torch.bfloat16, "v"), _ptr(gate, torch.bfloat16, "gate"),
                                     _ptr(Wf, torch.float32, "Wf"), W, C, m, T_max, _ptr(out, torch.bfloat16, "out"),
                                     _ptr(sel_idx, torch.int32, "sel_idx") if sel_idx.numel() else None,
                                     ws_ptr, ws_bytes,
                                     ct.byref(export_state.c_struct()) if export_state is not None else None,
                                     _stream(stream)), "still_prefill_gated")
    return out, sel_idx


def backward_workspace_size(q, k, Wf, W, C, m, T_max):
    sh = shape_of(q, k, Wf)
    return lib().still_backward_workspace_size(ct.byref(sh), W, C, m, T_max)


def backward(q, k, v, Wf, W, C, m, T_max, sel_idx, dout, grads=None, cmax_idx=None, workspace=None, stream=None):
    """Gradients of sum(dout * y) for the layer still_prefill computed with the
    selection sel_idx held fixed (see still_backward).  grads (optional) is a
    tuple (dq, dk, dv, dWf) of fp32 tensors to write; cmax_idx (optional) an
    int32 [B,Hq,N] tensor that receives the row-max key positions.
    Returns (dq, dk, dv, dWf)."""
    sh = shape_of(q, k, Wf)
    if grads is None:
        grads = (torch.empty(q.shape, dtype=torch.float32, device=q.device),
                 torch.empty(k.shape, dtype=torch.float32, device=q.device),
                 torch.empty(v.shape, dtype=torch.float32, device=q.device),
                 torch.empty(Wf.shape, dtype=torch.float32, device=q.device))
    dq, dk, dv, dWf = grads
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, torch.uint8, "workspace"), workspace.numel()
    _check(lib().still_backward(ct.byref(sh), _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"),
                                _ptr(v, torch.bfloat16, "v"), _ptr(Wf, torch.float32, "Wf"), W, C, m, T_max,
                                _ptr(sel_idx, torch.int32, "sel_idx") if sel_idx.numel() else None,
                                _ptr(dout, torch.bfloat16, "dout"), _ptr(dq, torch.float32, "dq"),
                                _ptr(dk, torch.float32, "dk"), _ptr(dv, torch.float32, "dv"),
                                _ptr(dWf, torch.float32, "dWf"),
                                _ptr(cmax_idx, torch.int32, "cmax_idx") if cmax_idx is not None else None,
                                ws_ptr, ws_bytes, _stream(stream)), "still_backward")
    return dq, dk, dv, dWf


def prefill_noalloc(q, k, v, Wf, W, C, m, T_max, out=None, sel_idx=None, export_state=None, stream=None):
    """still_prefill with the library's fixed scratch array instead of a workspace
    (for callers that may not allocate device memory); raises StillError when the
    size needs more scratch than the array holds."""
    B, Hq, N, d = q.shape
    lam = lam_of(W, m, T_max)
    sh = shape_of(q, k, Wf)
    if out is None:
        out = torch.empty_like(q)
    if sel_idx is None:
        sel_idx = torch.empty((B, k.shape[1], T_max, max(lam, 0)), dtype=torch.int32, device=q.device)
    st = ct.byref(export_state.c_struct()) if export_state is not None else None
    _check(lib().still_prefill_noalloc(ct.byref(sh), _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"),
                                       _ptr(v, torch.bfloat16, "v"), _ptr(Wf, torch.float32, "Wf"), W, C, m, T_max,
                                       _ptr(out, torch.bfloat16, "out"),
                                       _ptr(sel_idx, torch.int32, "sel_idx") if sel_idx.numel() else None,
                                       st, _stream(stream)), "still_prefill_noalloc")
    return out, sel_idx


def workspace_status(workspace, stream=None):
    """The device status word of a prefill (the first int32 of its workspace),
    read after synchronising `stream`: 0, or the still_status a kernel found."""
    val = ct.c_int32(0)
    _check(lib().still_read_status(_ptr(workspace, torch.uint8, "workspace"), _stream(stream), ct.byref(val)),
           "still_read_status")
    return int(val.value)


def debug_set_wait_limit(cycles):
    """Wait limit (clock cycles) of the prefill kernels' row-side waits; 0 restores
    the default.  For tests of the timeout path only."""
    lib().still_debug_set_wait_limit(int(cycles))


def decode_state_init(state: DecodeState, Hq, W, C, m, T_max, stream=None):
    sh = Shape(state.B, Hq, state.Hkv, 0, state.d, state.df)
    _check(lib().still_decode_state_init(ct.byref(sh), ct.byref(state.c_struct()), W, C, m, T_max,
                                         _stream(stream)), "still_decode_state_init")


def decode_step(state: DecodeState, q_t, k_t, v_t, Wf, W, C, m, T_max, out_t=None, stream=None):
    """One token per sequence: q_t [B,Hq,d], k_t, v_t [B,Hkv,d] (bf16) -> out_t [B,Hq,d]."""
    B, Hq, d = q_t.shape
    sh = Shape(B, Hq, k_t.shape[1], 0, d, Wf.shape[1])
    if out_t is None:
        out_t = torch.empty_like(q_t)
    _check(lib().still_decode_step(ct.byref(sh), ct.byref(state.c_struct()), _ptr(q_t, torch.bfloat16, "q_t"),
                                   _ptr(k_t, torch.bfloat16, "k_t"), _ptr(v_t, torch.bfloat16, "v_t"),
                                   _ptr(Wf, torch.float32, "Wf"), W, C, m, T_max,
                                   _ptr(out_t, torch.bfloat16, "out_t"), _stream(stream)), "still_decode_step")
    return out_t


def decode_step_gated(state: DecodeState, q_t, k_t, v_t, gate_t, Wf, W, C, m, T_max, out_t=None, stream=None):
    """One token per sequence of the gated layer: gate_t [B,Hq,d] bf16 holds this
    step's gate pre-activations (see still_decode_step_gated)."""
    B, Hq, d = q_t.shape
    if tuple(gate_t.shape) != tuple(q_t.shape):
        raise ValueError("gate_t must have the shape of q_t")
    sh = Shape(B, Hq, k_t.shape[1], 0, d, Wf.shape[1])
    if out_t is None:
        out_t = torch.empty_like(q_t)
    _check(lib().still_decode_step_gated(ct.byref(sh), ct.byref(state.c_struct()), _ptr(q_t, torch.bfloat16, "q_t"),
                                         _ptr(k_t, torch.bfloat16, "k_t"), _ptr(v_t, torch.bfloat16, "v_t"),
                                         _ptr(gate_t, torch.bfloat16, "gate_t"), _ptr(Wf, torch.float32, "Wf"),
                                         W, C, m, T_max, _ptr(out_t, torch.bfloat16, "out_t"), _stream(stream)),
           "still_decode_step_gated")
    return out_t


def timing_enable(on=True):
    lib().still_timing_enable(1 if on else 0)


def timing_read():
    """{kernel name: (launches, total ms)} since the last read."""
    buf = (KernelTime * 64)()
    n = lib().still_timing_read(buf, 64)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].ms) for i in range(min(n, 64))}


class HybridAttention(torch.autograd.Function):
    """The layer as a differentiable PyTorch op: forward = still_prefill, backward =
    still_backward with the forward's selection held fixed (the selection is a
    discrete choice and carries no gradient).  Inputs: q [B,Hq,N,d], k, v
    [B,Hkv,N,d] bf16, Wf [d,d_f] fp32; returns (y bf16, sel_idx int32).
    Gradients come back in the inputs' dtypes (bf16 for q, k, v; fp32 for Wf)."""

    @staticmethod
    def forward(ctx, q, k, v, Wf, W, C, m, T_max):
        y, sel = prefill(q, k, v, Wf, W, C, m, T_max)
        ctx.save_for_backward(q, k, v, Wf, sel)
        ctx.routing = (W, C, m, T_max)
        ctx.mark_non_differentiable(sel)
        return y, sel

    @staticmethod
    def backward(ctx, dy, _dsel):
        q, k, v, Wf, sel = ctx.saved_tensors
        W, C, m, T_max = ctx.routing
        dq, dk, dv, dWf = backward(q, k, v, Wf, W, C, m, T_max, sel, dy.to(torch.bfloat16).contiguous())
        return dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype), dWf, None, None, None, None


def hybrid_attention(q, k, v, Wf, W, C, m, T_max):
    """y of the layer with autograd support (see HybridAttention)."""
    y, _ = HybridAttention.apply(q, k, v, Wf, W, C, m, T_max)
    return y
