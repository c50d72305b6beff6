"""CPU oracle for the KDA chunked prefill -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg import this package.  The product path (``libkda.so`` and
``kda_gated_delta_chunk_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``kda_oracle.c``: a plain token-by-token fp64
recurrence (the definition of the operation; see that file's header for the
passages it follows).  This module only compiles it with gcc and marshals
numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")

# l2norm epsilon inside the square root (a reading: the pages do not state it)
L2NORM_EPS = 1e-6

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O3, OpenMP, IEEE semantics; no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.kda_oracle_fwd.restype = ctypes.c_int
            lib.kda_oracle_fwd.argtypes = [
                ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                P, P, P, P, P, P, P,
                ctypes.c_double, ctypes.c_double, ctypes.c_double,
                P, P, P, P, ctypes.c_int]
            lib.kda_oracle_max_threads.restype = ctypes.c_int
            lib.kda_oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle's OpenMP runtime uses by default."""
    return int(_load().kda_oracle_max_threads())


def _f64(x, shape):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def kda_oracle_fwd(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                   initial_state, cu_seqlens, eps: float = L2NORM_EPS,
                   num_threads: int = 0):
    """Token-by-token fp64 KDA recurrence.

    q, k, v, g: [T, H, D]; beta: raw logits [T, H]; A_log: [H];
    dt_bias: [H, D]; initial_state: [N, H, D, D] (key-channel major) or None;
    cu_seqlens: [N+1] ints.  Returns (out [T, H, D], final_state [N, H, D, D])
    as float64 arrays.  Rows of ``out`` for tokens past cu_seqlens[N] are 0.
    """
    q = np.asarray(q)
    T, H, D = q.shape
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    q = _f64(q, (T, H, D))
    k = _f64(k, (T, H, D))
    v = _f64(v, (T, H, D))
    g = _f64(g, (T, H, D))
    beta = _f64(beta, (T, H))
    A_log = _f64(A_log, (H,))
    dt_bias = _f64(dt_bias, (H, D))
    s0 = None if initial_state is None else _f64(initial_state, (N, H, D, D))
    out = np.zeros((T, H, D), dtype=np.float64)
    fin = np.zeros((N, H, D, D), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = _load().kda_oracle_fwd(
        T, N, H, D, ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(A_log),
        ptr(dt_bias), float(lower_bound), float(scale), float(eps), ptr(s0),
        ptr(cu), ptr(out), ptr(fin), int(num_threads))
    if rc != 0:
        raise ValueError("kda_oracle_fwd rejected its arguments")
    return out, fin
