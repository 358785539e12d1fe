"""Float64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. The CUDA library never calls it
and shares no code with it.

``forward`` runs the plain serial token-by-token recurrence written in
``dplr_oracle.c`` (see that file for what each mode computes and the passages
it follows); ``backward`` runs its reverse mode (the gradients of
sum(do * o) + sum(dST * S_T) with respect to every input); ``hla`` runs HLA's
query-gated composition of chunk transitions on the Gated DeltaNet update; ``gdp``
runs Gated DeltaProduct-style stacked Householders. Inputs of any float dtype are
upcast to float64 exactly.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dplr_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_handle = None

MODES = {"gdn": 1, "hdla": 2, "generic": 3}


def build(force: bool = False) -> str:
    """Compile dplr_oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_forward.restype = ctypes.c_int
            lib.oracle_forward.argtypes = [ctypes.c_int] * 8 + [dp] * 12 + [ctypes.c_int]
            lib.oracle_backward.restype = ctypes.c_int
            lib.oracle_backward.argtypes = [ctypes.c_int] * 8 + [dp] * 22 + [ctypes.c_int]
            lib.oracle_hla.restype = ctypes.c_int
            lib.oracle_hla.argtypes = [ctypes.c_int] * 6 + [ctypes.c_double] + [dp] * 7 + [ctypes.c_int]
            lib.oracle_gdp.restype = ctypes.c_int
            lib.oracle_gdp.argtypes = [ctypes.c_int] * 6 + [dp] * 8 + [ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            _handle = lib
    return _handle


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def forward(mode: str, q, k=None, v=None, decay=None, beta=None, A=None, Bm=None,
            K=None, V=None, S0=None, threads: Optional[int] = None):
    """Serial float64 recurrence. Returns (o [B,H,T,dv], S_T [B,H,dk,dv]).

    Shapes follow the library layout: q [B,H,T,dk]; structured modes take
    k [B,H,T,dk], v [B,H,T,dv], decay ([B,H,T] for GDN, [B,H,T,dk] for HDLA),
    beta [B,H,T]; generic mode takes decay [B,H,T,dk], A/Bm [B,H,T,r,dk],
    K [B,H,T,p,dk], V [B,H,T,p,dv]. S0 [B,H,dk,dv] or None (zero).
    """
    m = MODES[mode]
    q = _f64(q)
    B, H, T, dk = q.shape
    k, v, decay, beta = _f64(k), _f64(v), _f64(decay), _f64(beta)
    A, Bm, K, V, S0 = _f64(A), _f64(Bm), _f64(K), _f64(V), _f64(S0)
    if m == 3:
        r = 0 if A is None else A.shape[3]
        p = 0 if K is None else K.shape[3]
        dv = V.shape[4] if V is not None else (S0.shape[3] if S0 is not None else None)
        if dv is None:
            raise ValueError("generic mode needs V or S0 to fix dv")
    else:
        r, p = (1, 1) if m == 1 else (2, 1)
        dv = v.shape[3]
    o = np.zeros((B, H, T, dv), dtype=np.float64)
    ST = np.zeros((B, H, dk, dv), dtype=np.float64)
    rc = _lib().oracle_forward(m, B, H, T, dk, dv, r, p, _ptr(q), _ptr(k), _ptr(v), _ptr(decay),
                               _ptr(beta), _ptr(A), _ptr(Bm), _ptr(K), _ptr(V), _ptr(S0),
                               _ptr(o), _ptr(ST), int(threads or 0))
    if rc != 0:
        raise ValueError(f"oracle_forward rejected its arguments (code {rc})")
    return o, ST


def forward_inputs(inp: dict, threads: Optional[int] = None):
    """``forward`` on a dict produced by ``workloads.generate``."""
    w = inp["workload"]
    return forward(w.mode, inp["q"], inp["k"], inp["v"], inp["decay"], inp["beta"], inp["A"],
                   inp["Bm"], inp["K"], inp["V"], inp["S0"], threads=threads)


def backward(mode: str, q, k=None, v=None, decay=None, beta=None, A=None, Bm=None, K=None, V=None,
             S0=None, do=None, dST=None, threads: Optional[int] = None) -> dict:
    """Reverse mode of ``forward``: the gradients of sum(do * o) + sum(dST * S_T) with respect to every
    input, in float64. ``do`` [B,H,T,dv] is required, ``dST`` [B,H,dk,dv] may be None (zero). Returns a
    dict with the inputs' names (q, k, v, decay, beta for the structured modes; q, decay, A, Bm, K, V for
    the generic mode) and S0, each shaped like its input."""
    m = MODES[mode]
    q = _f64(q)
    B, H, T, dk = q.shape
    k, v, decay, beta = _f64(k), _f64(v), _f64(decay), _f64(beta)
    A, Bm, K, V, S0 = _f64(A), _f64(Bm), _f64(K), _f64(V), _f64(S0)
    do, dST = _f64(do), _f64(dST)
    dv = do.shape[3]
    if m == 3:
        r = 0 if A is None else A.shape[3]
        p = 0 if K is None else K.shape[3]
    else:
        r, p = 1, 0
    z = lambda shape: np.zeros(shape, dtype=np.float64)
    g = {"q": z(q.shape), "S0": z((B, H, dk, dv)), "decay": z(decay.shape)}
    if m == 3:
        g.update(A=z(A.shape) if A is not None else None, Bm=z(Bm.shape) if Bm is not None else None,
                 K=z(K.shape) if K is not None else None, V=z(V.shape) if V is not None else None)
    else:
        g.update(k=z(k.shape), v=z(v.shape), beta=z(beta.shape))
    rc = _lib().oracle_backward(m, B, H, T, dk, dv, r, p, _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta),
                                _ptr(A), _ptr(Bm), _ptr(K), _ptr(V), _ptr(S0), _ptr(do), _ptr(dST),
                                _ptr(g["q"]), _ptr(g.get("k")), _ptr(g.get("v")), _ptr(g["decay"]),
                                _ptr(g.get("beta")), _ptr(g.get("A")), _ptr(g.get("Bm")), _ptr(g.get("K")),
                                _ptr(g.get("V")), _ptr(g["S0"]), int(threads or 0))
    if rc != 0:
        raise ValueError(f"oracle_backward rejected its arguments (code {rc})")
    return g


def backward_inputs(inp: dict, do, dST=None, threads: Optional[int] = None) -> dict:
    """``backward`` on a dict produced by ``workloads.generate``."""
    w = inp["workload"]
    return backward(w.mode, inp["q"], inp["k"], inp["v"], inp["decay"], inp["beta"], inp["A"], inp["Bm"],
                    inp["K"], inp["V"], inp["S0"], do, dST, threads=threads)


def hla(q, k, v, g, beta, W, L: int, theta: float = 0.0, threads: Optional[int] = None):
    """HLA's query-gated composition of chunk transitions on the Gated DeltaNet update (see dplr_oracle.c):
    q, k [B,H,T,dk]; v [B,H,T,dv]; g, beta [B,H,T]; gates W [B,H,T,N] with N = ceil(T / L) (only the entries of
    earlier chunks are used; those below theta count as zero). Returns o [B,H,T,dv] in float64."""
    q, k, v, g, beta, W = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta), _f64(W)
    B, H, T, dk = q.shape
    dv = v.shape[3]
    N = (T + int(L) - 1) // int(L)
    if W.shape != (B, H, T, N):
        raise ValueError(f"gates W must be [B, H, T, ceil(T / L)] = {(B, H, T, N)}, got {W.shape}")
    o = np.zeros((B, H, T, dv), dtype=np.float64)
    rc = _lib().oracle_hla(B, H, T, dk, dv, int(L), float(theta), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(W), _ptr(o), int(threads or 0))
    if rc != 0:
        raise ValueError(f"oracle_hla rejected its arguments (code {rc})")
    return o


def gdp(q, k, v, g, beta, S0=None, threads: Optional[int] = None):
    """Gated DeltaProduct-style stacked Householders (see dplr_oracle.c): per token the gate, then n_h delta-rule
    steps. q [B,H,T,dk]; k [B,H,T,nh,dk]; v [B,H,T,nh,dv]; g [B,H,T]; beta [B,H,T,nh]; S0 [B,H,dk,dv] or None.
    Returns (o [B,H,T,dv], S_T [B,H,dk,dv]) in float64."""
    q, k, v, g, beta, S0 = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta), _f64(S0)
    B, H, T, dk = q.shape
    nh, dv = k.shape[3], v.shape[4]
    o = np.zeros((B, H, T, dv), dtype=np.float64)
    ST = np.zeros((B, H, dk, dv), dtype=np.float64)
    rc = _lib().oracle_gdp(B, H, T, dk, dv, nh, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(o),
                           _ptr(ST), int(threads or 0))
    if rc != 0:
        raise ValueError(f"oracle_gdp rejected its arguments (code {rc})")
    return o, ST
