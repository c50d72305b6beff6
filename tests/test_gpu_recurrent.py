"""GPU parity of the token-by-token form (kda_recurrent_fwd) against the fp64 oracle.

Decode and speculative-verify steps bring a few tokens per sequence; the
recurrent kernel must give what the oracle's token loop gives, write the state
after every token when asked (for rolling back to an accepted prefix), chain
through its own states, and agree with the chunked prefill on the same tokens.
"""
import json
import os

import numpy as np
import pytest
import torch

import kda_gated_delta_chunk_gb300 as kda
import kda_workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOL = json.load(open(os.path.join(ROOT, "tests", "golden", "tolerances.json")))["max_abs"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kda_gated_delta_chunk_gb300 import build as kbuild
    kbuild.build()
    assert kda.device_check(torch.cuda.current_device()) == kda.OK


def dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "rows" else v)
            for k, v in inp.items()}


def f64(t):
    return t.float().double().cpu().numpy()


def oracle_run(oracle_mod, inp, zero_init=False):
    return oracle_mod.kda_oracle_fwd(
        f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]), f64(inp["beta"]),
        f64(inp["A_log"]), f64(inp["dt_bias"]), inp["lower_bound"], inp["scale"],
        None if zero_init else f64(inp["initial_state"]), inp["cu_seqlens"].numpy())


def run(inp, token_states=False, initial_state="keep"):
    d = dev(inp)
    s0 = d["initial_state"] if isinstance(initial_state, str) else initial_state
    out, fin, ts = kda.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                     d["dt_bias"], d["lower_bound"], d["scale"], s0,
                                     d["cu_seqlens"], token_states=token_states,
                                     state_dtype=inp["initial_state"].dtype)
    torch.cuda.synchronize()
    return out, fin, ts


@pytest.mark.parametrize("sd", ["f32", "bf16"])
def test_recurrent_matches_oracle(oracle_mod, sd):
    inp = W.make_inputs(W.custom([1, 2, 3, 7, 1, 0, 5], 4, state_dtype=sd, seed=51))
    out, fin, _ = run(inp)
    o_ref, f_ref = oracle_run(oracle_mod, inp)
    T = inp["q"].shape[0]
    do = np.abs(f64(out[:T]) - o_ref).max()
    df = np.abs(f64(fin) - f_ref).max()
    print(f"recurrent {sd}: out max {do:.3e} state max {df:.3e}")
    assert do <= TOL[sd] and df <= TOL[sd]


def test_token_states_are_the_prefix_states(oracle_mod):
    """token_states[t] is the state after token t: the oracle's final state on the prefix
    ending at t; the last one of each sequence equals final_state bit for bit."""
    inp = W.make_inputs(W.custom([4, 1, 3], 2, seed=52))
    out, fin, ts = run(inp, token_states=True)
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(cu) - 1):
        for m in range(1, cu[n + 1] - cu[n] + 1):
            sub = W.select(inp, [n], [0, 1])
            sub["cu_seqlens"] = torch.tensor([0, m], dtype=torch.int32)
            for key in ("q", "k", "v", "g", "beta"):
                sub[key] = sub[key][:m]
            _, f_ref = oracle_run(oracle_mod, sub)
            got = f64(ts[cu[n] + m - 1])
            assert np.abs(got - f_ref[0]).max() <= TOL["f32"], (n, m)
        assert torch.equal(ts[cu[n + 1] - 1], fin[n])


def test_chaining_one_token_calls_equals_one_call():
    """k tokens in one call == k calls of one token each, threading the state (fp32 state:
    the same arithmetic, so bit for bit)."""
    inp = W.make_inputs(W.custom([6], 3, seed=53))
    out_all, fin_all, _ = run(inp)
    state = dev(inp)["initial_state"]
    outs = []
    for t in range(6):
        step = dict(inp)
        for key in ("q", "k", "v", "g", "beta"):
            step[key] = inp[key][t:t + 1]
        step["cu_seqlens"] = torch.tensor([0, 1], dtype=torch.int32)
        o, state, _ = run(step, initial_state=state)
        outs.append(o)
    assert torch.equal(torch.cat(outs), out_all) and torch.equal(state, fin_all)


def test_recurrent_agrees_with_chunked_prefill(oracle_mod):
    """A sequence long enough for several chunks: the token-by-token kernel and the
    chunked prefill agree within the tolerance (both are checked against the oracle)."""
    inp = W.make_inputs(W.custom([150, 9], 2, seed=54))
    out_r, fin_r, _ = run(inp)
    d = dev(inp)
    out_p, fin_p = kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                         d["dt_bias"], d["lower_bound"], d["scale"],
                                         d["initial_state"], d["cu_seqlens"])
    torch.cuda.synchronize()
    o_ref, f_ref = oracle_run(oracle_mod, inp)
    assert np.abs(f64(out_r) - o_ref).max() <= TOL["f32"]
    assert np.abs(f64(fin_r) - f_ref).max() <= TOL["f32"]
    assert (out_r.float() - out_p.float()).abs().max().item() <= TOL["f32"]
    assert (fin_r - fin_p).abs().max().item() <= TOL["f32"]
