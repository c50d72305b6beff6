"""The allocation-free entry point against the regular one, on the GPU.

kda_chunk_prefill_fwd_noalloc serves callers that cannot allocate device
memory (so cannot pass a workspace): its scratch is a static device array
inside libkda.so.  Called twice in a row through the C ABI, it must give
what kda_chunk_prefill_fwd gives on the same inputs, within the tests'
tolerance (0.01 with an fp32 state, 0.03 with a bf16 state).  This file is
collected last on purpose, and also passes when run alone.
"""
import ctypes
import json
import os

import pytest
import torch

import kda_gated_delta_chunk_gb300 as kda
import kda_workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOL = json.load(open(os.path.join(ROOT, "tests", "golden", "tolerances.json")))["max_abs"]


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kda_gated_delta_chunk_gb300 import build as kbuild
    kbuild.build()
    return kda.lib()


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


@pytest.mark.parametrize("sd", ["f32", "bf16"])
def test_noalloc_matches_regular_entry_point_twice(L, sd):
    w = W.custom([200, 64, 1, 130], 4, state_dtype=sd, seed=41)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in W.make_inputs(w).items()}
    T, H, N = d["q"].shape[0], 4, 4
    stream = torch.cuda.current_stream()
    sdt = kda.STATE_F32 if sd == "f32" else kda.STATE_BF16
    # regular entry point, with its own workspace
    ws = kda.alloc_workspace(T, H, N)
    out_ref = torch.empty_like(d["q"])
    fin_ref = torch.empty_like(d["initial_state"])
    rc = L.kda_chunk_prefill_fwd(
        _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["g"]), _p(d["beta"]), _p(d["A_log"]),
        _p(d["dt_bias"]), float(d["lower_bound"]), float(d["scale"]), _p(d["initial_state"]),
        _p(d["cu_seqlens"]), _p(out_ref), _p(fin_ref), sdt, _p(ws),
        ctypes.c_void_p(stream.cuda_stream), T, N, H, ws.numel())
    assert rc == kda.OK
    for _ in range(2):      # two calls in a row share the static scratch
        out = torch.full_like(d["q"], float("nan"))
        fin = torch.full_like(d["initial_state"], float("nan"))
        rc = L.kda_chunk_prefill_fwd_noalloc(
            _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["g"]), _p(d["beta"]), _p(d["A_log"]),
            _p(d["dt_bias"]), float(d["lower_bound"]), float(d["scale"]),
            _p(d["initial_state"]), _p(d["cu_seqlens"]), _p(out), _p(fin), sdt,
            ctypes.c_void_p(stream.cuda_stream), T, N, H)
        assert rc == kda.OK, kda.status_string(rc)
        torch.cuda.synchronize()
        tol = TOL[sd]
        assert torch.isfinite(out.float()).all() and torch.isfinite(fin.float()).all()
        assert (out.float() - out_ref.float()).abs().max().item() <= tol
        assert (fin.float() - fin_ref.float()).abs().max().item() <= tol


def test_noalloc_binding_and_bad_arguments(L):
    w = W.custom([70], 2, seed=42)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in W.make_inputs(w).items()}
    out = torch.empty_like(d["q"])
    fin = torch.empty_like(d["initial_state"])
    kda.chunk_prefill_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                  d["dt_bias"], d["lower_bound"], d["scale"],
                                  d["initial_state"], d["cu_seqlens"], out, fin)
    out_ref, fin_ref = kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                             d["A_log"], d["dt_bias"], d["lower_bound"],
                                             d["scale"], d["initial_state"], d["cu_seqlens"])
    torch.cuda.synchronize()
    assert (out.float() - out_ref.float()).abs().max().item() <= TOL["f32"]
    assert (fin - fin_ref).abs().max().item() <= TOL["f32"]
    with pytest.raises(kda.KDAError) as e:
        kda.chunk_prefill_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                      d["dt_bias"], -9.0, d["scale"], d["initial_state"],
                                      d["cu_seqlens"], out, fin)
    assert e.value.code == kda.ERR_UNSAFE_LOWER_BOUND
