"""The seeded input generator against the stated recipe of the five prefill workloads.

Shapes, length mixes, state dtype and initialisation per workload; the value distributions
(q, k, v, g and the beta logits N(0, 1) rounded to bf16 once, A_log = log U[1, 16],
dt_bias N(0, 0.1), the state N(0, 0.02)); lower_bound -5 and scale 128^-0.5; and that the
draw is a function of the seed alone.
"""
import math

import numpy as np
import pytest
import torch

import kda_workloads as W

D = 128


@pytest.mark.parametrize("cfg,n,lengths,H,state,init", [
    (0, None, [128], 2, "f32", "zeros"),
    (1, None, [2048] * 8, 16, "f32", "normal"),
    (2, None, [16384], 16, "f32", "normal"),
    (3, 1, [4096], 8, "f32", "normal"),
    (3, 2, [4096] * 2, 8, "f32", "normal"),
    (3, 3, [4096] * 3, 8, "f32", "normal"),
    (3, 7, [4096] * 7, 8, "f32", "normal"),
])
def test_fixed_shape_workloads(cfg, n, lengths, H, state, init):
    w = W.workload(cfg, n)
    assert list(w.lengths) == lengths and w.heads == H
    assert w.state_dtype == state and w.init == init
    assert w.lower_bound == -5.0 and w.scale == D ** -0.5


def test_ragged_workload_length_mix():
    w = W.workload(4)
    lens = np.array(w.lengths)
    assert len(lens) == 64 and lens.sum() == 65536 and w.heads == 32
    assert w.state_dtype == "bf16" and w.init == "normal"
    assert lens.min() >= 16 and lens.max() <= 4096
    # log-uniform over [16, 4096]: the lengths spread over the whole log range
    logs = np.log(lens)
    assert logs.max() - logs.min() > 0.6 * (math.log(4096) - math.log(16))


def test_value_distributions():
    inp = W.make_inputs(W.workload(1))
    for name in ("q", "k", "v", "g", "beta"):
        x = inp[name]
        assert x.dtype == torch.bfloat16
        x = x.float()
        assert abs(float(x.mean())) < 0.01, name
        assert abs(float(x.std()) - 1.0) < 0.01, name
    a = torch.exp(inp["A_log"])
    assert inp["A_log"].dtype == torch.float32 and inp["A_log"].shape == (16,)
    assert float(a.min()) >= 1.0 and float(a.max()) <= 16.0
    assert inp["dt_bias"].shape == (16, D)
    assert abs(float(inp["dt_bias"].std()) - 0.1) < 0.01
    s = inp["initial_state"]
    assert s.dtype == torch.float32 and s.shape == (8, 16, D, D)
    assert abs(float(s.std()) - 0.02) < 0.001 and abs(float(s.mean())) < 0.001
    assert inp["cu_seqlens"].tolist() == [2048 * i for i in range(9)]
    assert inp["lower_bound"] == -5.0 and inp["scale"] == D ** -0.5


def test_zero_and_bf16_initial_states():
    assert not W.make_inputs(W.workload(0))["initial_state"].any()
    w = W.custom([300, 100], 4, state_dtype="bf16", seed=9)
    s = W.make_inputs(w)["initial_state"]
    assert s.dtype == torch.bfloat16 and abs(float(s.float().std()) - 0.02) < 0.002


def test_draw_depends_on_the_seed_alone():
    a = W.make_inputs(W.custom([200, 57], 3, seed=11))
    b = W.make_inputs(W.custom([200, 57], 3, seed=11))
    c = W.make_inputs(W.custom([200, 57], 3, seed=12))
    for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"):
        assert torch.equal(a[name], b[name]), name
        assert not torch.equal(a[name], c[name]), name
