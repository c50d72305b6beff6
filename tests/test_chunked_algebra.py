"""The chunk algebra and its exponent anchoring, checked against the oracle.

The kernels compute the recurrence chunk by chunk (the WY/UT form named for
FlashKDA-style prefill); ``chunked_ref`` restates that algebra in numpy.
Here it must equal the token-by-token oracle to rounding in fp64, keep every
factor finite in fp32 under the strongest decay the library accepts, and --
with bf16 tensor-core operands emulated -- stay inside the pass bar of 0.01
(fp32 state) that the bf16-checkpoint PR report uses.
"""
import numpy as np
import pytest

import kda_workloads as W
from chunked_ref import chunk_forward


def rand_problem(rng, lengths, H, D, lb=-5.0, gate_shift=0.0, state_std=0.3):
    T = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return dict(
        q=rng.standard_normal((T, H, D)), k=rng.standard_normal((T, H, D)),
        v=rng.standard_normal((T, H, D)), g=rng.standard_normal((T, H, D)) + gate_shift,
        beta=rng.standard_normal((T, H)),
        A_log=np.log(rng.uniform(1, 16, H)), dt_bias=0.1 * rng.standard_normal((H, D)),
        lower_bound=lb, scale=D ** -0.5,
        initial_state=state_std * rng.standard_normal((len(lengths), H, D, D)),
        cu_seqlens=cu)


@pytest.mark.parametrize("C", [16, 32, 64])
def test_direct_chunk_form_equals_oracle(oracle_mod, C):
    rng = np.random.default_rng(100 + C)
    p = rand_problem(rng, [70, 1, 0, 33, 64], 2, 16)
    o_ref, f_ref = oracle_mod.kda_oracle_fwd(**p)
    o, f = chunk_forward(**p, C=C, mode="direct")
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(f, f_ref, rtol=0, atol=1e-10)


@pytest.mark.parametrize("C,sub", [(64, 32), (32, 16), (16, 16)])
def test_anchored_chunk_form_equals_oracle(oracle_mod, C, sub):
    rng = np.random.default_rng(200 + C)
    p = rand_problem(rng, [130, 5, 64, 31, 97], 2, 16)
    o_ref, f_ref = oracle_mod.kda_oracle_fwd(**p)
    o, f = chunk_forward(**p, C=C, sub=sub, mode="anchored")
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(f, f_ref, rtol=0, atol=1e-10)


@pytest.mark.parametrize("lb,shift", [(-5.0, 0.0), (-5.0, 50.0), (-5.5, 50.0)])
def test_anchored_factors_finite_in_fp32(oracle_mod, lb, shift):
    """Saturated gates (a -> lb on every token) at the largest accepted |lb|."""
    rng = np.random.default_rng(300)
    p = rand_problem(rng, [128, 77], 2, 32, lb=lb, gate_shift=shift)
    o_ref, f_ref = oracle_mod.kda_oracle_fwd(**p)
    o, f = chunk_forward(**p, C=64, sub=32, mode="anchored", factor_dtype=np.float32)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=2e-5)
    np.testing.assert_allclose(f, f_ref, rtol=0, atol=2e-5)


def _to64(inp):
    f = lambda t: t.float().double().numpy()
    return dict(q=f(inp["q"]), k=f(inp["k"]), v=f(inp["v"]), g=f(inp["g"]), beta=f(inp["beta"]),
                A_log=f(inp["A_log"]), dt_bias=f(inp["dt_bias"]),
                lower_bound=inp["lower_bound"], scale=inp["scale"],
                initial_state=f(inp["initial_state"]), cu_seqlens=inp["cu_seqlens"].numpy())


def test_bf16_operands_within_fp32_state_tolerance(oracle_mod):
    """Workload 0 (1 x 128, H=2) plus a 300-token state-carrying case:
    bf16 operands, fp32 state, against the oracle's 0.01 bar."""
    for w in (W.workload(0), W.custom([300], 2, seed=5)):
        p = _to64(W.make_inputs(w))
        o_ref, f_ref = oracle_mod.kda_oracle_fwd(**p)
        o, f = chunk_forward(**p, C=64, sub=32, mode="anchored", factor_dtype=np.float32,
                             operand_bf16=True)
        err_o = np.abs(o - o_ref).max()
        err_f = np.abs(f - f_ref).max()
        assert err_o < 0.01 and err_f < 0.01, (w.name, err_o, err_f)
