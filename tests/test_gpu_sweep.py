"""GPU: a seeded sweep of batch shapes across every path.

Each case draws sequence lengths (ragged tails, 1-token and empty sequences, several
chunks), a head count and a state dtype from a fixed seed, runs it through the fused
kernel (P = 1 and a forced value split), the fused kernel with helpers, the split path and
the reference kernel -- some of them through an output row map -- and checks every result
against the fp64 oracle at the tolerance of its state dtype.  The paths must also agree
with each other within that tolerance.
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


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 6))
    pool = [0, 1, 7, 63, 64, 65, 127, 128, 129, 200, 257, 333, 640]
    lengths = [int(rng.choice(pool)) for _ in range(n)]
    if sum(lengths) == 0:
        lengths[0] = 65
    heads = int(rng.choice([1, 2, 3, 4]))
    sd = "bf16" if rng.random() < 0.3 else "f32"
    return lengths, heads, sd


PATHS = [("tc", kda.KERNEL_TC, 1), ("tc_p4", kda.KERNEL_TC, 4), ("helpers", kda.KERNEL_TC_HELPERS, -1),
         ("split", kda.KERNEL_SPLIT, -1), ("split_p2", kda.KERNEL_SPLIT, 2), ("ref", kda.KERNEL_REF, 1),
         ("pipe", kda.KERNEL_PIPE, 1)]


@pytest.mark.parametrize("seed", range(12))
def test_sweep(oracle_mod, seed):
    lengths, H, sd = draw_case(seed)
    inp = W.make_inputs(W.custom(lengths, H, state_dtype=sd, seed=500 + seed))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "rows" else v) for k, v in inp.items()}
    T, N = d["q"].shape[0], len(lengths)
    used = int(inp["cu_seqlens"][-1])
    f = lambda t: t.float().double().cpu().numpy()
    o_ref, s_ref = oracle_mod.kda_oracle_fwd(
        f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["g"]), f(inp["beta"]), f(inp["A_log"]),
        f(inp["dt_bias"]), inp["lower_bound"], inp["scale"], f(inp["initial_state"]),
        inp["cu_seqlens"].numpy())
    ws = torch.zeros(1024 + ((T + 63) // 64 + N) * H * (66560 + 4), dtype=torch.uint8,
                     device="cuda")
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
            d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])
    rng = np.random.default_rng(2000 + seed)
    results = {}
    for name, kern, vs in PATHS:
        if kern == kda.KERNEL_TC_HELPERS and N * H + 1 > torch.cuda.get_device_properties(0).multi_processor_count:
            continue
        mapped = bool(rng.random() < 0.5) and kern != kda.KERNEL_PIPE   # dense outputs only
        if mapped:
            rows = torch.from_numpy(rng.permutation(T + 5)[:T].astype(np.int32)).cuda()
            buf = torch.zeros(T + 5, H, 128, dtype=torch.bfloat16, device="cuda")
            out, fin = kda.chunk_prefill_fwd(*args, out=buf, workspace=ws, kernel=kern,
                                             vsplit=vs, out_index=rows)
            torch.cuda.synchronize()
            out = buf[rows.long()]
        else:
            out, fin = kda.chunk_prefill_fwd(*args, workspace=ws, kernel=kern, vsplit=vs)
            torch.cuda.synchronize()
        assert kda.last_device_status(ws) == kda.OK, name
        do = np.abs(f(out)[:used] - o_ref[:used]).max() if used else 0.0
        ds = np.abs(f(fin) - s_ref).max()
        assert do <= TOL[sd] and ds <= TOL[sd], (name, lengths, H, sd, do, ds)
        results[name] = (out[:used].float(), fin.float())
    base = results["tc"]
    for name, (o, s) in results.items():
        assert (o - base[0]).abs().max().item() <= TOL[sd], name
        assert (s - base[1]).abs().max().item() <= TOL[sd], name
