"""ctypes wrapper of the C streaming oracle (``still_ref.c``).

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  The shared library
is built with gcc on first use (or by ``build()``); it links nothing from the
CUDA library.  All arrays are float64 / int32, C-contiguous.
"""
from __future__ import annotations

import ctypes as ct
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "still_ref.c")
_LIB = os.path.join(_HERE, "libstill_ref.so")
_lock = threading.Lock()
_lib = None

_D = ct.POINTER(ct.c_double)
_I32 = ct.POINTER(ct.c_int32)
_I64 = ct.POINTER(ct.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc if the library is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC,
                        "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ct.CDLL(_LIB)
            L.oref_lambda.restype = ct.c_int
            L.oref_lambda.argtypes = [ct.c_int] * 3
            L.oref_npmap.restype = None
            L.oref_npmap.argtypes = [_D, ct.c_long, ct.c_int, _D, ct.c_int, _D]
            L.oref_scores.restype = None
            L.oref_scores.argtypes = [_D, _D] + [ct.c_int] * 5 + [_D, _D]
            L.oref_metric_scores.restype = None
            L.oref_metric_scores.argtypes = [_D, _D] + [ct.c_int] * 8 + [ct.c_uint64, ct.c_long, _D]
            L.oref_select.restype = None
            L.oref_select.argtypes = [_D] + [ct.c_int] * 5 + [_I32]
            L.oref_state_init.restype = None
            L.oref_state_init.argtypes = [ct.c_int] * 6 + [_D, _D, _I32, _I32, _D, _D, _D, _D]
            L.oref_prefill.restype = ct.c_int
            L.oref_prefill.argtypes = ([ct.c_int] * 10 + [_D, _D, _D, _D, _I32, _D, _D, _D]
                                       + [_D, _D, _I32, _I32, _D, _D, _D, _D, ct.c_int])
            L.oref_decode_step.restype = ct.c_int
            L.oref_decode_step.argtypes = ([ct.c_int] * 9 + [_I64, _D, _D, _D, _D, _D, _D]
                                           + [_D, _D, _I32, _I32, _D, _D, _D, _D, ct.c_int])
            L.oref_max_threads.restype = ct.c_int
            _lib = L
    return _lib


def _d(a):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_D)


def _i32(a):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(_I32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def lam_of(m, W, T_max):
    return lib().oref_lambda(m, W, T_max)


def max_threads():
    return lib().oref_max_threads()


def npmap(x, Wf):
    x = _f64(x)
    Wf = _f64(Wf)
    d, df = Wf.shape
    rows = x.size // d
    phi = np.empty(x.shape[:-1] + (df,))
    lib().oref_npmap(_d(x), rows, d, _d(Wf), df, _d(phi))
    return phi


def scores(q, k, W):
    """q [Hq,N,d], k [Hkv,N,d] (one sequence) -> (head scores [Hq,N], kv scores [Hkv,N])."""
    q, k = _f64(q), _f64(k)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    hs = np.empty((Hq, N))
    s = np.empty((Hkv, N))
    lib().oref_scores(_d(q), _d(k), Hq, Hkv, N, d, W, _d(hs), _d(s))
    return hs, s


# routing metrics of the ablation (the ids of still_metric in include/still.h are
# the library's; these are the oracle's own, written out here)
METRICS = {"self_saliency": 0, "diagonal": 1, "qk": 2, "key_norm": 3, "uniform": 4, "random": 5}


def metric_scores(q, k, W, C, lam, metric, seed=0, unit0=0):
    """Routing-metric scores of one sequence: q [Hq,N,d], k [Hkv,N,d] -> [Hkv,N].
    unit0 = b * Hkv places the sequence in the random metric's counter."""
    if metric == "self_saliency":
        return scores(q, k, W)[1]
    q, k = _f64(q), _f64(k)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    out = np.empty((Hkv, N))
    lib().oref_metric_scores(_d(q), _d(k), Hq, Hkv, N, d, W, C, lam, METRICS[metric], ct.c_uint64(seed),
                             int(unit0), _d(out))
    return out


def prefill_routed(q, k, v, Wf, W, C, m, T_max, metric, seed=0, sel=None, threads=0):
    """The layer with its chunks ranked by a routing metric: the metric's scores,
    the top-lambda of every completed chunk, then the prefill with that
    selection.  sel (optional [B,Hkv,T_max,lam]) replaces the selection.
    Returns (y [B,Hq,N,d], metric scores [B,Hkv,N], selection)."""
    q, k = _f64(q), _f64(k)
    B, Hkv = q.shape[0], k.shape[1]
    lam = lam_of(m, W, T_max)
    sc = np.stack([metric_scores(q[b], k[b], W, C, lam, metric, seed, b * Hkv) for b in range(B)])
    if sel is None:
        sel = np.stack([select(sc[b], C, lam, T_max) for b in range(B)])
    y, _, _ = prefill(q, k, v, Wf, W, C, m, T_max, sel_override=sel if lam > 0 else None, threads=threads)
    return y, sc, sel


def select(scores_kv, C, lam, T_max):
    s = _f64(scores_kv)
    Hkv, N = s.shape
    sel = np.empty((Hkv, T_max, max(lam, 0)), dtype=np.int32)
    if lam > 0:
        lib().oref_select(_d(s), Hkv, N, C, lam, T_max, _i32(sel))
    return sel


class State:
    """Streaming state of B sequences (float64 mirror of the decode cache)."""

    def __init__(self, B, Hkv, d, df, C, m):
        self.K = np.zeros((B, Hkv, m, d))
        self.V = np.zeros((B, Hkv, m, d))
        self.pos = np.full((B, Hkv, m), -1, dtype=np.int32)
        self.cnt = np.zeros((B, Hkv, m), dtype=np.int32)
        self.ssc = np.zeros((B, Hkv, m))
        self.S = np.zeros((B, Hkv, df, d))
        self.z = np.zeros((B, Hkv, df))
        self.ring = np.zeros((B, Hkv, C))
        self.t = np.zeros(B, dtype=np.int64)

    def ptrs(self):
        return [_d(self.K), _d(self.V), _i32(self.pos), _i32(self.cnt), _d(self.ssc),
                _d(self.S), _d(self.z), _d(self.ring)]

    def copy(self):
        o = object.__new__(State)
        for key, val in self.__dict__.items():
            setattr(o, key, val.copy())
        return o


def prefill(q, k, v, Wf, W, C, m, T_max, sel_override=None, threads=0, gate=None):
    """q [B,Hq,N,d], k,v [B,Hkv,N,d] -> (y [B,Hq,N,d], scores [B,Hkv,N], State).
    gate (optional [B,Hq,N,d]): pre-activations of the linear branch's gate."""
    q, k, v, Wf = _f64(q), _f64(k), _f64(v), _f64(Wf)
    gt = _f64(gate) if gate is not None else None
    if gt is not None:
        assert gt.shape == q.shape
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    df = Wf.shape[1]
    lam = lam_of(m, W, T_max)
    if lam < 0:
        raise ValueError("invalid budget")
    st = State(B, Hkv, d, df, C, m)
    y = np.empty_like(q)
    sc = np.empty((B, Hkv, N))
    ovr = None
    if sel_override is not None and lam > 0:
        ovr = np.ascontiguousarray(sel_override, dtype=np.int32)
        assert ovr.shape == (B, Hkv, T_max, lam)
    rc = lib().oref_prefill(B, Hq, Hkv, N, d, df, W, C, m, T_max, _d(q), _d(k), _d(v), _d(Wf),
                            _i32(ovr) if ovr is not None else None, _d(gt) if gt is not None else None,
                            _d(y), _d(sc),
                            *st.ptrs(), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle prefill failed ({rc})")
    st.t[:] = N
    return y, sc, st


def decode_step(st: State, q_t, k_t, v_t, Wf, W, C, m, T_max, threads=0, gate_t=None):
    """One token for every sequence; updates `st` in place and returns y [B,Hq,d].
    gate_t (optional [B,Hq,d]): pre-activations of the linear branch's gate."""
    q_t, k_t, v_t, Wf = _f64(q_t), _f64(k_t), _f64(v_t), _f64(Wf)
    gt = _f64(gate_t) if gate_t is not None else None
    B, Hq, d = q_t.shape
    Hkv = k_t.shape[1]
    df = Wf.shape[1]
    y = np.empty_like(q_t)
    rc = lib().oref_decode_step(B, Hq, Hkv, d, df, W, C, m, T_max, st.t.ctypes.data_as(_I64),
                                _d(q_t), _d(k_t), _d(v_t), _d(Wf), _d(gt) if gt is not None else None, _d(y),
                                *st.ptrs(), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle decode step failed ({rc})")
    st.t += 1
    return y
