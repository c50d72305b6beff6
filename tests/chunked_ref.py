"""The chunked (WY/UT) form of the KDA recurrence, in numpy -- a test aid.

This is not the oracle (``oracle/`` holds the token-by-token definition) and
not the CUDA path (which shares no code with anything here).  It restates,
in plain numpy, the chunk algebra the CUDA kernels are designed on, so that
the algebra -- and the exponent anchoring that keeps it inside the fp32/bf16
range -- can be checked against the oracle on the CPU, and so that the
rounding of bf16 tensor-core operands can be emulated to predict the
kernels' error before they run.

Chunk algebra (per sequence n, head h; chunk of L <= C tokens; rows r, s are
tokens of the chunk; Gam_r = inclusive cumsum of the log decay a over the
chunk, per key channel; S is the state entering the chunk):

  A[r,s]  = b_r * sum_d kh_r kh_s exp(Gam_r - Gam_s),   s < r   (else 0)
  QK[r,s] =       sum_d qh_r kh_s exp(Gam_r - Gam_s),   s <= r  (else 0)
  T       = (I + A)^-1                     (unit lower triangular)
  W       = T diag(b) (kh * exp(Gam))      U' = T diag(b) V
  U       = U' - W S
  O       = (qh * exp(Gam)) S + QK U
  S_next  = diag(exp(Gam_last)) S + (kh * exp(Gam_last - Gam))^T U

Anchoring ("anchored" mode).  The chunk is cut into sub-blocks of ``sub``
tokens (32 for C = 64).  Inside sub-block j the cumsum is taken from the
sub-block start (c_r) and anchored at its middle row m_j (alpha_j = c_m):
E_r = exp(c_r - alpha_j) and Ei_r = exp(alpha_j - c_r) stay within
exp(+-|lb| sub/2) -- inside fp32 for |lb| <= 5.5.  Products inside one
sub-block use E (row) and Ei (column).  Between sub-blocks the row operand
is the row block's own E and the column operand carries all the remaining
factors (each <= 1), so the diagonal and off-diagonal products share one row
operand.  The chunk-level factors exp(Gam_r) and exp(Gam_last - Gam_s) are
built from the same per-element E/Ei times per-channel constants.
"""
from __future__ import annotations

import math

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even), back as fp32."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(a), a, out)


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def _factors_anchored(a, sub, dt):
    """Per-element factors for one chunk, in dtype ``dt``; a: [L, D] log decay.

    Returns dict with E, Ei (sub-block anchored), and the chunk-level
    factors g_row = exp(Gam_r), g_end = exp(Gam_last - Gam_r), decay, and
    for every ordered pair of sub-blocks (i > j) the row / column factors.
    """
    L, D = a.shape
    nb = (L + sub - 1) // sub
    E = np.empty((L, D), dt)
    Ei = np.empty((L, D), dt)
    c_loc = np.empty((L, D), dt)
    alpha, btot = [], []
    for j in range(nb):
        r0, r1 = j * sub, min(L, (j + 1) * sub)
        c = np.cumsum(a[r0:r1].astype(dt), axis=0, dtype=dt)
        m = min(sub // 2 - 1, r1 - r0 - 1)
        al = c[m]
        c_loc[r0:r1] = c
        E[r0:r1] = np.exp(c - al)
        Ei[r0:r1] = np.exp(al - c)
        alpha.append(al)
        btot.append(c[-1])
    # chunk-level factors: exp(Gam_r) = exp(c_r) * exp(sum of earlier totals)
    g_row = np.empty((L, D), dt)
    g_end = np.empty((L, D), dt)
    before = np.zeros(D, dt)
    total = np.sum(np.stack(btot), axis=0, dtype=dt)
    for j in range(nb):
        r0, r1 = j * sub, min(L, (j + 1) * sub)
        loc = E[r0:r1] * np.exp(alpha[j])                   # exp(c_r)  (<= 1)
        g_row[r0:r1] = loc * np.exp(before)
        after = total - before - btot[j]                   # totals of later blocks
        tail = Ei[r0:r1] * np.exp(btot[j] - alpha[j])       # exp(B_j - c_r) (<= 1)
        g_end[r0:r1] = tail * np.exp(after)
        before = before + btot[j]
    pair_row, pair_col = {}, {}
    for i in range(nb):
        for j in range(i):
            # rows in block i, columns in block j: exp(Gam_r - Gam_s) =
            #   exp(c_r) * exp(totals of blocks j+1..i-1) * exp(B_j - c_s)
            mid = np.zeros(D, dt)
            for t in range(j + 1, i):
                mid = mid + btot[t]
            r0, r1 = i * sub, min(L, (i + 1) * sub)
            s0, s1 = j * sub, (j + 1) * sub
            # the row operand is block i's own E; every other factor (each
            # <= 1) is folded into the column operand
            pair_row[(i, j)] = E[r0:r1]
            pair_col[(i, j)] = (Ei[s0:s1] * np.exp(btot[j] - alpha[j])) * (np.exp(alpha[i])
                                                                          * np.exp(mid))
    decay = np.exp(total)
    return dict(E=E, Ei=Ei, g_row=g_row, g_end=g_end, decay=decay,
                pair_row=pair_row, pair_col=pair_col, nb=nb)


def chunk_forward(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                  initial_state, cu_seqlens, C=64, sub=32, mode="anchored",
                  factor_dtype=np.float64, operand_bf16=False, eps=1e-6,
                  check_finite=True):
    """Chunked KDA prefill over packed sequences; returns (out, final_state).

    mode="direct": exp(Gam_r - Gam_s) element by element (no anchoring).
    mode="anchored": the sub-block factorisation above, factors computed in
    ``factor_dtype``; with ``operand_bf16`` every tensor-core operand is
    rounded to bf16 (the state read by the products included), the state
    kept in fp32, and all sums accumulated in fp64.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, H, D = q.shape
    cu = np.asarray(cu_seqlens, np.int64)
    N = len(cu) - 1
    out = np.zeros((T, H, D))
    fin = np.zeros((N, H, D, D))
    rnd = bf16_round if operand_bf16 else (lambda x: np.asarray(x, np.float64))
    for n in range(N):
        for h in range(H):
            S = (np.zeros((D, D)) if initial_state is None
                 else np.array(initial_state[n, h], np.float64))
            if operand_bf16:
                S = S.astype(np.float32).astype(np.float64)
            for c0 in range(cu[n], cu[n + 1], C):
                c1 = min(cu[n + 1], c0 + C)
                L = c1 - c0
                Q, K, V = q[c0:c1, h], k[c0:c1, h], v[c0:c1, h]
                qh = Q / np.sqrt((Q * Q).sum(1, keepdims=True) + eps) * scale
                kh = K / np.sqrt((K * K).sum(1, keepdims=True) + eps)
                a = lower_bound * _sig(math.exp(A_log[h]) * (g[c0:c1, h] + dt_bias[h]))
                b = _sig(beta[c0:c1, h])
                if mode == "direct":
                    Gam = np.cumsum(a, axis=0)
                    Dm = np.exp(Gam[:, None, :] - Gam[None, :, :])
                    Dm = np.where(np.tril(np.ones((L, L), bool))[:, :, None], Dm, 0.0)
                    KK = np.einsum("rd,sd,rsd->rs", kh, kh, Dm)
                    QK = np.einsum("rd,sd,rsd->rs", qh, kh, Dm)
                    g_row = np.exp(Gam)
                    g_end = np.exp(Gam[-1] - Gam)
                    decay = np.exp(Gam[-1])
                else:
                    f = _factors_anchored(a, sub, factor_dtype)
                    if check_finite:
                        for name in ("E", "Ei", "g_row", "g_end", "decay"):
                            assert np.all(np.isfinite(f[name])), name
                    KK = np.zeros((L, L))
                    QK = np.zeros((L, L))
                    # (inside a diagonal block the anti-causal entries, s > r, can overflow:
                    # their factors grow the other way; np.tril below drops them)
                    with np.errstate(over="ignore", invalid="ignore"):
                        for i in range(f["nb"]):
                            r0, r1 = i * sub, min(L, (i + 1) * sub)
                            Er, Eir = f["E"][r0:r1], f["Ei"][r0:r1]
                            KK[r0:r1, r0:r1] = rnd(kh[r0:r1] * Er) @ rnd(kh[r0:r1] * Eir).T
                            QK[r0:r1, r0:r1] = rnd(qh[r0:r1] * Er) @ rnd(kh[r0:r1] * Eir).T
                            for j in range(i):
                                s0, s1 = j * sub, (j + 1) * sub
                                pr, pc = f["pair_row"][(i, j)], f["pair_col"][(i, j)]
                                if check_finite:
                                    assert np.all(np.isfinite(pr)) and np.all(np.isfinite(pc))
                                colop = rnd(kh[s0:s1] * pc)
                                KK[r0:r1, s0:s1] = rnd(kh[r0:r1] * pr) @ colop.T
                                QK[r0:r1, s0:s1] = rnd(qh[r0:r1] * pr) @ colop.T
                    KK = np.tril(KK, -1)
                    QK = np.tril(QK, 0)
                    g_row = np.asarray(f["g_row"], np.float64)
                    g_end = np.asarray(f["g_end"], np.float64)
                    decay = np.asarray(f["decay"], np.float64)
                Amat = b[:, None] * np.tril(KK, -1)
                Tm = np.linalg.inv(np.eye(L) + Amat)
                TB = rnd(Tm * b[None, :])
                W = rnd(TB @ rnd(kh * g_row))
                Up = TB @ rnd(V)
                U = Up - W @ rnd(S)
                Ub = rnd(U)
                O = rnd(qh * g_row) @ rnd(S) + rnd(np.tril(QK, 0)) @ Ub
                S = decay[:, None] * S + rnd(kh * g_end).T @ Ub
                if operand_bf16:
                    S = S.astype(np.float32).astype(np.float64)
                out[c0:c1, h] = O
            fin[n, h] = S
    return out, fin
