"""CPU oracle for the low-M projections (kda_skinny_proj) -- test infrastructure only.

The two GEMMs of the Kimi-K3 low-M KDA projection overlap in the vLLM PR report
"[Bugfix] Fix Kimi-K3 KDA projection overlap compile on Hopper" (its skinny-GEMM test
listing): the first projects the hidden states, the second takes the first r columns of
the first's output, as stored in bf16, and projects them again:

    y = x w_ab^T                   (fp64 here; the device rounds it to bf16)
    z = bf16(y)[:, :r] w_b^T

Each product is numpy's fp64 matrix product of the exact bf16 input values.  The one
decision taken in floating point -- rounding y to bf16 before the second product -- is
made here in fp64 with round-to-nearest-even, by bit manipulation of the value's float32
image after an exact float64 -> float32 step when the value is representable, else by
rounding the float64 directly.
"""
from __future__ import annotations

import numpy as np


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits: the nearest multiple of 2^(e - 7) for a value in
    [2^e, 2^(e+1)).  Computed from the exponent with frexp, so no float32 step is involved
    (which would double-round)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    nz = a != 0
    mant, exp = np.frexp(a[nz])            # a = mant * 2^exp, 0.5 <= |mant| < 1
    scale = np.ldexp(1.0, (exp - 8).astype(np.int64))   # ulp of an 8-significant-bit value
    q = a[nz] / scale                      # exact: a power-of-two division
    out[nz] = np.round(q) * scale          # numpy rounds halves to even
    return out


def skinny_proj(x: np.ndarray, w_ab: np.ndarray, w_b: np.ndarray, r: int):
    """x [m, k], w_ab [n_ab, k], w_b [n_b, r] (the bf16 values, as float64).
    Returns (y, z): y = x w_ab^T in fp64, z = bf16(y)[:, :r] w_b^T in fp64."""
    x = np.asarray(x, dtype=np.float64)
    w_ab = np.asarray(w_ab, dtype=np.float64)
    w_b = np.asarray(w_b, dtype=np.float64)
    y = x @ w_ab.T
    z = bf16_round(y)[:, :r] @ w_b.T
    return y, z
