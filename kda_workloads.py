"""Seeded synthetic inputs for the KDA chunked prefill.

This module is shared by the tests, the benchmark and the smoke check.  It
holds shapes, seeds and random draws only -- none of the method's
arithmetic -- so that the CUDA path and the CPU oracle can be fed the same
values without sharing any computation.

The workloads follow the shapes the vLLM PR reports on FlashKDA quote
("[Perf][GLM-5.3-Flash] Use FlashKDA for KDA chunked prefill", PR #55737:
8 x 2048 and 1 x 16384 prefills, head_dim 128, bf16 q/k/v/g/beta; "[Kimi-K3]
[Perf] Update FlashKDA for automatic K2 V-split", PR #52458: low-parallelism
batches where 2 * heads * sequences <= SM count; "[KDA] Update flashKDA to
support bf16 checkpoint state", PR #56485: fp32 and bf16 state).  No public
dataset is involved; every value is drawn here:

  q, k, v, g (raw gate logits), beta (raw logits) ~ N(0, 1), drawn in fp32,
  rounded once to bf16.  A_log = log(U[1, 16]) fp32 [H];  dt_bias ~
  N(0, 0.1) fp32 [H, 128];  lower_bound = -5.0;  scale = 128 ** -0.5;
  initial_state ~ N(0, 0.02) (std 0.02) in the state dtype, or zeros.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 128
LOWER_BOUND = -5.0
SCALE = HEAD_DIM ** -0.5


@dataclass(frozen=True)
class Workload:
    name: str
    lengths: tuple
    heads: int
    state_dtype: str          # "f32" or "bf16"
    init: str                 # "zeros" or "normal"
    seed: int
    lower_bound: float = LOWER_BOUND
    scale: float = SCALE
    pad_tokens: int = 0       # extra rows past cu_seqlens[N] (left untouched)
    note: str = field(default="", compare=False)

    @property
    def num_seqs(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths)) + self.pad_tokens


def ragged_lengths(num_seqs: int, total: int, lo: int, hi: int, seed: int) -> list:
    """Log-uniform lengths in [lo, hi], rescaled to sum exactly to ``total``.

    Draw u ~ U(0, 1) per sequence (seeded torch CPU generator), take
    exp(log lo + u (log hi - log lo)), rescale multiplicatively with clipping
    to [lo, hi] until the sum settles, floor, then hand out the remaining
    tokens one at a time to the sequences with the largest fractional parts
    that are still below ``hi``.
    """
    gen = torch.Generator().manual_seed(seed)
    u = torch.rand(num_seqs, generator=gen, dtype=torch.float64)
    x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    for _ in range(200):
        x = torch.clamp(x * (total / float(x.sum())), lo, hi)
    base = torch.floor(x).to(torch.int64)
    rem = total - int(base.sum())
    frac = (x - base.to(torch.float64)).tolist()
    order = sorted(range(num_seqs), key=lambda i: -frac[i])
    lens = base.tolist()
    i = 0
    while rem > 0:
        j = order[i % num_seqs]
        if lens[j] < hi:
            lens[j] += 1
            rem -= 1
        i += 1
    while rem < 0:
        j = order[i % num_seqs]
        if lens[j] > lo:
            lens[j] -= 1
            rem += 1
        i += 1
    return lens


def workload(cfg: int, n: int | None = None) -> Workload:
    """The five prefill workloads (0..4); workload 3 takes n in {1, 2, 3, 7}."""
    if cfg == 0:
        return Workload("tiny_1x128_h2", (128,), 2, "f32", "zeros", 0)
    if cfg == 1:
        return Workload("batched_8x2048_h16", (2048,) * 8, 16, "f32", "normal", 1)
    if cfg == 2:
        return Workload("long_1x16384_h16", (16384,), 16, "f32", "normal", 2)
    if cfg == 3:
        n = 1 if n is None else int(n)
        return Workload(f"vsplit_{n}x4096_h8", (4096,) * n, 8, "f32", "normal", 30 + n)
    if cfg == 4:
        lens = ragged_lengths(64, 65536, 16, 4096, seed=4)
        return Workload("ragged_64seq_65536_h32_bf16state", tuple(lens), 32, "bf16",
                        "normal", 4)
    raise ValueError(f"unknown workload {cfg}")


def custom(lengths, heads, state_dtype="f32", init="normal", seed=0,
           lower_bound=LOWER_BOUND, scale=SCALE, pad_tokens=0) -> Workload:
    """A workload with explicit lengths (edge cases, sweeps)."""
    return Workload(f"custom_{len(lengths)}seq_h{heads}", tuple(int(x) for x in lengths),
                    int(heads), state_dtype, init, int(seed), float(lower_bound),
                    float(scale), int(pad_tokens))


def _randn_bf16(shape, gen, std=1.0, chunk_rows=1 << 14):
    """N(0, std^2) drawn in fp32 row-block by row-block, rounded to bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    inner = 1
    for x in shape[1:]:
        inner *= int(x)
    flat = out.view(shape[0], inner)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        blk = torch.randn((r1 - r0, flat.shape[1]), generator=gen, dtype=torch.float32)
        if std != 1.0:
            blk.mul_(std)
        flat[r0:r1].copy_(blk)
    return out


def make_inputs(w: Workload) -> dict:
    """Host (CPU) tensors for one workload, fully determined by ``w.seed``.

    Returns q, k, v, g [T, H, 128] bf16; beta [T, H] bf16; A_log [H] fp32;
    dt_bias [H, 128] fp32; initial_state [N, H, 128, 128] (state dtype);
    cu_seqlens [N+1] int32; plus lower_bound, scale, state_dtype.
    """
    T, H, D, N = w.total_tokens, w.heads, HEAD_DIM, w.num_seqs
    gen = torch.Generator().manual_seed(w.seed)
    q = _randn_bf16((T, H, D), gen)
    k = _randn_bf16((T, H, D), gen)
    v = _randn_bf16((T, H, D), gen)
    g = _randn_bf16((T, H, D), gen)
    beta = _randn_bf16((T, H), gen)
    A_log = torch.log(torch.rand(H, generator=gen, dtype=torch.float32) * 15.0 + 1.0)
    dt_bias = torch.randn((H, D), generator=gen, dtype=torch.float32) * 0.1
    sdt = torch.float32 if w.state_dtype == "f32" else torch.bfloat16
    if w.init == "zeros":
        s0 = torch.zeros((N, H, D, D), dtype=sdt)
    else:
        s0 = _randn_f32((N * H, D * D), gen, std=0.02).to(sdt).view(N, H, D, D)
    cu = torch.zeros(N + 1, dtype=torch.int32)
    if N:
        cu[1:] = torch.cumsum(torch.tensor(w.lengths, dtype=torch.int64), 0).to(torch.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
                initial_state=s0, cu_seqlens=cu, lower_bound=w.lower_bound,
                scale=w.scale, state_dtype=w.state_dtype)


def _randn_f32(shape, gen, std=1.0, chunk_rows=1 << 12):
    out = torch.empty(shape, dtype=torch.float32)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0, shape[1]), generator=gen, dtype=torch.float32) * std
    return out


def select(inp: dict, seqs, heads) -> dict:
    """The sub-problem made of the chosen sequences and heads, repacked.

    Every (sequence, head) pair is an independent recurrence, so the oracle
    can be run on a sample of pairs of a large workload: this returns the
    inputs of that sample (tokens of the chosen sequences only, chosen head
    columns only), with its own cu_seqlens.
    """
    cu = inp["cu_seqlens"].tolist()
    seqs = list(seqs)
    heads = torch.as_tensor(list(heads), dtype=torch.long)
    rows = torch.cat([torch.arange(cu[n], cu[n + 1]) for n in seqs]) if seqs else \
        torch.zeros(0, dtype=torch.long)
    lens = [cu[n + 1] - cu[n] for n in seqs]
    ncu = torch.zeros(len(seqs) + 1, dtype=torch.int32)
    if seqs:
        ncu[1:] = torch.cumsum(torch.tensor(lens), 0).to(torch.int32)
    pick = lambda x: x.index_select(0, rows).index_select(1, heads)
    return dict(q=pick(inp["q"]), k=pick(inp["k"]), v=pick(inp["v"]), g=pick(inp["g"]),
                beta=inp["beta"].index_select(0, rows).index_select(1, heads),
                A_log=inp["A_log"].index_select(0, heads),
                dt_bias=inp["dt_bias"].index_select(0, heads),
                initial_state=inp["initial_state"].index_select(0, torch.tensor(seqs, dtype=torch.long))
                .index_select(1, heads),
                cu_seqlens=ncu, lower_bound=inp["lower_bound"], scale=inp["scale"],
                state_dtype=inp["state_dtype"], rows=rows)
