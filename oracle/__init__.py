"""fp64 CPU oracle for the Gated DeltaNet recurrence that CPR evaluates.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path never imports this package,
and this package imports nothing from the product.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, token by token); this module
builds it with gcc and marshals numpy arrays through ctypes.  See the C file's header for
the operator, the conventions and the citations.

Pins (what ties the oracle to something other than itself) live in
``tests/test_oracle_pins.py``: closed forms for beta=0, the delta-rule projection for
g=0/beta=1/unit k, hand-worked tiny cases under ``tests/golden/``, the scalar recurrence,
the chunk (WY/UT) form against the token recurrence, grouped heads against repeated heads,
linearity in (v, state_in), and central finite differences for the backward.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into libgdn_oracle.so next to it (gcc, -O2, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_fwd.argtypes = [I, P, I, I, I, I, P, P, P, P, P, P, P, P, I, P, I]
            lib.oracle_fwd.restype = I
            lib.oracle_bwd.argtypes = [I, P, I, I, I, I] + [P] * 14 + [I]
            lib.oracle_bwd.restype = I
            lib.oracle_chunk_states.argtypes = [I, P, I, I, I, I, P, P, P, P, P, I, P, P, I]
            lib.oracle_chunk_states.restype = I
            lib.oracle_num_chunks.argtypes = [I, P, I]
            lib.oracle_num_chunks.restype = ctypes.c_longlong
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def num_chunks(cu_seqlens, chunk: int) -> int:
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    return int(_load().oracle_num_chunks(len(cu) - 1, _ptr(cu), chunk))


def fwd(q, k, v, g, beta, cu_seqlens, state_in=None, chunk: int = 0, n_threads: int | None = None):
    """Token-by-token forward.  Shapes: q,k [T,Hqk,dk]; v [T,Hv,dv]; g,beta [T,Hv];
    state_in [N,Hv,dv,dk] or None.  Returns (o [T,Hv,dv], state_out [N,Hv,dv,dk], bnd)
    where bnd [sum ceil(L/C), Hv, dv, dk] holds the state before every chunk (None if
    chunk == 0)."""
    lib = _load()
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    state_in = _f64(state_in)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, hqk, dk = k.shape
    hv, dv = v.shape[1], v.shape[2]
    n = len(cu) - 1
    o = np.zeros((T, hv, dv))
    st = np.zeros((n, hv, dv, dk))
    bnd = None
    if chunk > 0:
        bnd = np.zeros((num_chunks(cu, chunk), hv, dv, dk))
    rc = lib.oracle_fwd(n, _ptr(cu), hqk, hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                        _ptr(beta), _ptr(state_in), _ptr(o), _ptr(st), chunk, _ptr(bnd),
                        n_threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_fwd rejected its arguments (rc={rc})")
    return o, st, bnd


def bwd(q, k, v, g, beta, cu_seqlens, dout, state_in=None, dstate_out=None,
        n_threads: int | None = None):
    """Reverse-mode gradient of fwd.  Returns dict with dq, dk [T,Hqk,dk], dv [T,Hv,dv],
    dg, dbeta [T,Hv], dstate_in [N,Hv,dv,dk]."""
    lib = _load()
    q, k, v, g, beta, dout = map(_f64, (q, k, v, g, beta, dout))
    state_in, dstate_out = _f64(state_in), _f64(dstate_out)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, hqk, dk = k.shape
    hv, dv = v.shape[1], v.shape[2]
    n = len(cu) - 1
    out = dict(dq=np.zeros((T, hqk, dk)), dk=np.zeros((T, hqk, dk)), dv=np.zeros((T, hv, dv)),
               dg=np.zeros((T, hv)), dbeta=np.zeros((T, hv)), dstate_in=np.zeros((n, hv, dv, dk)))
    rc = lib.oracle_bwd(n, _ptr(cu), hqk, hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                        _ptr(beta), _ptr(state_in), _ptr(dout), _ptr(dstate_out),
                        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                        _ptr(out["dbeta"]), _ptr(out["dstate_in"]),
                        n_threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_bwd rejected its arguments (rc={rc})")
    return out


def chunk_states(k, v, g, beta, cu_seqlens, chunk: int, state_in=None,
                 n_threads: int | None = None):
    """Chunk (WY/UT) form: returns (bnd [sum ceil(L/C),Hv,dv,dk], state_out [N,Hv,dv,dk])."""
    lib = _load()
    k, v, g, beta = map(_f64, (k, v, g, beta))
    state_in = _f64(state_in)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, hqk, dk = k.shape
    hv, dv = v.shape[1], v.shape[2]
    n = len(cu) - 1
    bnd = np.zeros((num_chunks(cu, chunk), hv, dv, dk))
    st = np.zeros((n, hv, dv, dk))
    rc = lib.oracle_chunk_states(n, _ptr(cu), hqk, hv, dk, dv, _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta), _ptr(state_in), chunk, _ptr(bnd), _ptr(st),
                                 n_threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_chunk_states rejected its arguments (rc={rc})")
    return bnd, st
