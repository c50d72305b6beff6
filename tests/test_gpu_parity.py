"""GPU parity: libkda.so's kernels against the fp64 oracle, element by element.

Every workload's inputs come from the seeded generator; the oracle reads
the exact bf16/fp32 values the GPU reads.  The pass bar is the tolerance the
bf16-checkpoint PR report uses (max |delta| 0.01 with an fp32 state, 0.03
with a bf16 state) on both out and final_state; mean |delta| is printed.
Full-size workloads run on the GPU exactly as the benchmark launches them;
the oracle then checks every (sequence, head) pair it can afford (all of
them for the smaller workloads, a sample that always includes the longest
sequence for the largest).
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
KERNELS = [kda.KERNEL_REF, kda.KERNEL_TC, kda.KERNEL_SPLIT, kda.KERNEL_TC_HELPERS,
           kda.KERNEL_PIPE, kda.KERNEL_SPLIT_STREAMED]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kda_gated_delta_chunk_gb300 import build as kbuild
    kbuild.build()
    rc = kda.device_check(torch.cuda.current_device())
    assert rc == kda.OK, kda.status_string(rc)


def to_dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "rows" else v)
            for k, v in inp.items()}


def split_workspace(T, H, N):
    """Workspace with the split path's records for exactly this batch: a 1 KB header and
    66,560 bytes per (chunk slot, head), ceil(T / 64) + N slots."""
    n = 1024 + ((T + 63) // 64 + N) * H * 66560
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def helper_workspace(T, H, N):
    """The same records plus one 4-byte claim word per (chunk slot, head)."""
    n = 1024 + ((T + 63) // 64 + N) * H * (66560 + 4)
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def workspace_for(kernel, T, H, N):
    if kernel == kda.KERNEL_SPLIT:
        return split_workspace(T, H, N)
    if kernel in (kda.KERNEL_TC_HELPERS, kda.KERNEL_SPLIT_STREAMED):
        return helper_workspace(T, H, N)
    return None


def run_gpu(inp, kernel=kda.KERNEL_AUTO, vsplit=-1, out=None, final_state=None, init="keep"):
    d = to_dev(inp)
    s0 = d["initial_state"] if init == "keep" else None
    ws = workspace_for(kernel, d["q"].shape[0], d["q"].shape[1], d["cu_seqlens"].numel() - 1)
    out, fin = kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                     d["dt_bias"], d["lower_bound"], d["scale"], s0,
                                     d["cu_seqlens"], out=out, final_state=final_state,
                                     workspace=ws, state_dtype=inp["initial_state"].dtype,
                                     vsplit=vsplit, kernel=kernel)
    torch.cuda.synchronize()
    return out, fin


def f64(t):
    return t.float().double().cpu().numpy()


def oracle_sub(oracle_mod, inp, seqs, heads, zero_init=False):
    sub = W.select(inp, seqs, heads)
    o, f = oracle_mod.kda_oracle_fwd(
        f64(sub["q"]), f64(sub["k"]), f64(sub["v"]), f64(sub["g"]), f64(sub["beta"]),
        f64(sub["A_log"]), f64(sub["dt_bias"]), sub["lower_bound"], sub["scale"],
        None if zero_init else f64(sub["initial_state"]), sub["cu_seqlens"].numpy())
    return sub["rows"], o, f


def check(oracle_mod, inp, out, fin, seqs=None, heads=None, tol=None, zero_init=False, tag=""):
    N = inp["cu_seqlens"].numel() - 1
    H = inp["q"].shape[1]
    seqs = list(range(N)) if seqs is None else list(seqs)
    heads = list(range(H)) if heads is None else list(heads)
    tol = TOL[inp["state_dtype"]] if tol is None else tol
    rows, o_ref, f_ref = oracle_sub(oracle_mod, inp, seqs, heads, zero_init)
    hidx = torch.tensor(heads)
    o_gpu = f64(out.cpu().index_select(0, rows).index_select(1, hidx))
    f_gpu = f64(fin.cpu().index_select(0, torch.tensor(seqs, dtype=torch.long)).index_select(1, hidx))
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(f_gpu))
    do, df = np.abs(o_gpu - o_ref), np.abs(f_gpu - f_ref)
    print(f"{tag}: out max {do.max() if do.size else 0:.3e} mean {do.mean() if do.size else 0:.3e}"
          f" | state max {df.max():.3e} mean {df.mean():.3e}")
    assert (do.max() if do.size else 0.0) <= tol, ("out", do.max())
    assert df.max() <= tol, ("final_state", df.max())
    return do, df


# ----------------------------------------------------------------- workloads
@pytest.mark.parametrize("kernel", KERNELS)
def test_workload0_tiny(oracle_mod, kernel):
    inp = W.make_inputs(W.workload(0))
    out, fin = run_gpu(inp, kernel)
    check(oracle_mod, inp, out, fin, tag=f"w0 k{kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("vsplit", [1, 2, 4, 8])
def test_ragged_tiles_and_tails(oracle_mod, kernel, vsplit):
    """Several chunks, ragged tails, a 1-token and an empty sequence."""
    if kernel in (kda.KERNEL_TC_HELPERS, kda.KERNEL_PIPE) and vsplit != 1:
        pytest.skip("the helpers and the pipelined kernel run unsplit only")
    if kernel == kda.KERNEL_SPLIT_STREAMED:
        pytest.skip("27 chains need more than the SMs' half at P = 4 (streamed cases below)")
    w = W.custom([1, 63, 64, 65, 130, 0, 200, 17, 129], 3, seed=21)
    inp = W.make_inputs(w)
    out, fin = run_gpu(inp, kernel, vsplit)
    check(oracle_mod, inp, out, fin, tag=f"ragged k{kernel} P{vsplit}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_bf16_state(oracle_mod, kernel):
    w = W.custom([300, 5, 64, 129], 4, state_dtype="bf16", seed=22)
    inp = W.make_inputs(w)
    out, fin = run_gpu(inp, kernel)
    assert fin.dtype == torch.bfloat16
    check(oracle_mod, inp, out, fin, tag=f"bf16 state k{kernel}")


@pytest.mark.parametrize("vsplit", [2, 4, 8])
def test_bf16_state_value_slices(oracle_mod, vsplit):
    """The split path's value-slice chains read and write a bf16 state (P = 2: the tcgen05
    chain, 64 columns a slice in two 32-column halves; P = 4, 8: the warp-level chain)."""
    w = W.custom([300, 5, 64, 129], 4, state_dtype="bf16", seed=23)
    inp = W.make_inputs(w)
    out, fin = run_gpu(inp, kda.KERNEL_SPLIT, vsplit)
    assert fin.dtype == torch.bfloat16
    check(oracle_mod, inp, out, fin, tag=f"bf16 state split P{vsplit}")


@pytest.mark.parametrize("cfg", [1, 2])
@pytest.mark.parametrize("kernel", [kda.KERNEL_AUTO, kda.KERNEL_TC, kda.KERNEL_SPLIT,
                                    kda.KERNEL_TC_HELPERS, kda.KERNEL_PIPE])
def test_workloads_1_2_full_size(oracle_mod, cfg, kernel):
    inp = W.make_inputs(W.workload(cfg))
    out, fin = run_gpu(inp, kernel, 1 if kernel == kda.KERNEL_TC else -1)
    heads = None if cfg == 1 else [0, 5, 11, 15]
    check(oracle_mod, inp, out, fin, heads=heads, tag=f"workload {cfg} k{kernel}")


@pytest.mark.parametrize("n", [1, 2, 3, 7])
def test_workload3_vsplit_vs_unsplit(oracle_mod, n):
    """Split and unsplit paths: same layout, values within tolerance of each
    other and of the oracle (bit identity is not required)."""
    inp = W.make_inputs(W.workload(3, n))
    out_a, fin_a = run_gpu(inp)                 # automatic split
    out_1, fin_1 = run_gpu(inp, vsplit=1)       # forced unsplit
    assert out_a.shape == out_1.shape and fin_a.shape == fin_1.shape
    tol = TOL["f32"]
    assert (out_a.float() - out_1.float()).abs().max().item() <= tol
    assert (fin_a - fin_1).abs().max().item() <= tol
    heads = [0, 3, 7]
    check(oracle_mod, inp, out_a, fin_a, heads=heads, tag=f"w3 n={n} auto")
    check(oracle_mod, inp, out_1, fin_1, heads=heads, tag=f"w3 n={n} P=1")


@pytest.mark.parametrize("cfg,n,P", [(2, None, 4), (3, 2, 4), (3, 3, 2), (3, 7, 1)])
def test_auto_takes_split_path_when_it_triggers(oracle_mod, cfg, n, P):
    """One long sequence (16 heads), 2, 3 and 7 x 4096 (8 heads): AUTO runs the streamed
    split path (the chain beside the k-side kernel; P = 4, 4, 2 and 1, the tcgen05 chains
    at P = 2 and 1) -- the same bits as forcing it, and as the plain split path at the same
    P (the same records and the same chain arithmetic, only started earlier)."""
    inp = W.make_inputs(W.workload(cfg, n) if cfg == 3 else W.workload(cfg))
    T, H, N = inp["q"].shape[0], inp["q"].shape[1], inp["cu_seqlens"].numel() - 1
    assert kda.plan(T, N, H, kda.workspace_size(T, H, N), -1, kda.KERNEL_AUTO)[:2] == \
        (kda.KERNEL_SPLIT_STREAMED, P)
    out_a, fin_a = run_gpu(inp)
    out_s, fin_s = run_gpu(inp, kda.KERNEL_SPLIT_STREAMED)
    assert torch.equal(out_a, out_s) and torch.equal(fin_a, fin_s)
    out_p, fin_p = run_gpu(inp, kda.KERNEL_SPLIT, vsplit=P)
    assert torch.equal(out_a, out_p) and torch.equal(fin_a, fin_p)


@pytest.mark.parametrize("lengths,H,sd,P", [
    ([1, 63, 64, 65, 130, 0, 200], 2, "f32", 4),     # ragged tails, 1-token and empty
    ([300, 5, 64, 129, 900], 3, "bf16", 4),
    ([2048, 2048], 2, "f32", 8),
    ([8192], 4, "f32", 8),
    ([100], 1, "bf16", 8),
    ([1, 63, 64, 65, 130, 0, 200], 2, "f32", 2),     # the tcgen05 chain at P = 2
    ([300, 5, 64, 129, 900], 3, "bf16", 2),
    ([1, 63, 64, 65, 130, 0, 200], 2, "f32", 1),     # the unsplit tcgen05 chain
    ([300, 5, 64, 129, 900], 3, "bf16", 1),
])
def test_streamed_split_against_the_oracle(oracle_mod, lengths, H, sd, P):
    """The streamed split path (chain CTAs copying each record as the k-side kernel
    publishes it) on ragged batches and both state dtypes; one workspace serves a second
    call with new inputs, and the path's header words are back at zero after each call."""
    N, T = len(lengths), sum(lengths)
    ws = helper_workspace(T, H, N)
    for seed in (51, 52):
        inp = W.make_inputs(W.custom(lengths, H, state_dtype=sd, seed=seed))
        d = to_dev(inp)
        out, fin = kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                         d["dt_bias"], d["lower_bound"], d["scale"],
                                         d["initial_state"], d["cu_seqlens"], workspace=ws,
                                         state_dtype=inp["initial_state"].dtype, vsplit=P,
                                         kernel=kda.KERNEL_SPLIT_STREAMED)
        torch.cuda.synchronize()
        assert kda.last_device_status(ws) == kda.OK
        assert ws[512:532].view(torch.int32)[1:].cpu().tolist() == [0, 0, 0, 0]
        check(oracle_mod, inp, out, fin, tag=f"streamed P{P} {lengths} seed {seed}")


def test_streamed_split_dropped_record_times_out():
    """Failure detection on the streamed split path without a GPU fault: with the test hook
    on, the k-side kernel leaves the record of the first chunk of head 0 unpublished; the
    chain CTAs that need it give up after a bounded wait and the call records
    KDA_ERR_DEVICE_TIMEOUT.  The next call on the same workspace is correct: the last chain
    CTA cleared the path's claim words and counters on the way out."""
    inp = W.make_inputs(W.custom([1024, 1024], 2, seed=45))
    d = to_dev(inp)
    T = d["q"].shape[0]
    ws = helper_workspace(T, 2, 2)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
            d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])
    kda.test_drop_one_record(True)
    try:
        kda.chunk_prefill_fwd(*args, workspace=ws, kernel=kda.KERNEL_SPLIT_STREAMED)
        torch.cuda.synchronize()
    finally:
        kda.test_drop_one_record(False)
    assert kda.last_device_status(ws) == kda.ERR_DEVICE_TIMEOUT
    assert ws[512:532].view(torch.int32)[1:].cpu().tolist() == [0, 0, 0, 0]
    out, fin = kda.chunk_prefill_fwd(*args, workspace=ws, kernel=kda.KERNEL_SPLIT_STREAMED)
    torch.cuda.synchronize()
    assert kda.last_device_status(ws) == kda.OK
    out_p, fin_p = run_gpu(inp, kda.KERNEL_SPLIT, vsplit=8)
    assert torch.equal(out, out_p) and torch.equal(fin, fin_p)


def test_split_falls_back_to_fused_on_small_workspace(oracle_mod):
    """AUTO with a workspace below the split path's record area runs one CTA per
    (sequence, head) -- the warp-specialised kernel; forcing the split path with it is
    refused."""
    inp = W.make_inputs(W.custom([150, 70], 2, seed=31))
    d = to_dev(inp)
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
            d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])
    out, fin = kda.chunk_prefill_fwd(*args, workspace=small)
    torch.cuda.synchronize()
    out_t, fin_t = run_gpu(inp, kda.KERNEL_PIPE, vsplit=1)
    assert torch.equal(out, out_t) and torch.equal(fin, fin_t)
    check(oracle_mod, inp, out, fin, tag="small workspace")
    with pytest.raises(kda.KDAError) as e:
        kda.chunk_prefill_fwd(*args, workspace=small, kernel=kda.KERNEL_SPLIT)
    assert e.value.code == kda.ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("kernel", [kda.KERNEL_AUTO, kda.KERNEL_SPLIT, kda.KERNEL_PIPE])
def test_workload4_ragged_bf16_state(oracle_mod, kernel):
    w = W.workload(4)
    inp = W.make_inputs(w)
    out, fin = run_gpu(inp, kernel)
    lens = list(w.lengths)
    longest = int(np.argmax(lens))
    shortest = int(np.argmin(lens))
    seqs = sorted({longest, shortest, 0, 17, 40, 63})
    check(oracle_mod, inp, out, fin, seqs=seqs, heads=[0, 13, 31], tag="workload 4")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("lb,shift", [(-5.0, 40.0), (-5.0, -40.0), (-5.0, 0.0), (0.0, 0.0)])
def test_extreme_gates(oracle_mod, kernel, lb, shift):
    """The gate at its limits: every token decays by e^lb with the largest accepted |lb|
    (sigmoid saturated at 1: the anchored exponents reach 2^(+-16 |lb| log2 e)), no decay
    (sigmoid saturated at 0, or lb = 0), and the largest |lb| with ordinary gates.  The raw
    q/k rows are scaled up by 64 too: the kernels must not depend on normalised inputs."""
    w = W.custom([130, 64, 1, 77], 2, seed=33, lower_bound=lb)
    inp = W.make_inputs(w)
    inp["g"] = (inp["g"].float() + shift).to(torch.bfloat16)
    inp["q"] = (inp["q"].float() * 64.0).to(torch.bfloat16)   # exact: a power of two
    inp["k"] = (inp["k"].float() * 64.0).to(torch.bfloat16)
    out, fin = run_gpu(inp, kernel)
    check(oracle_mod, inp, out, fin, tag=f"gates lb={lb} shift={shift} k{kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_strong_uniform_decay_keeps_adjacent_terms(oracle_mod, kernel):
    """Every channel decays by about 2^-5 per token (lb = -5, sigmoid 0.7), so the anchors of
    the two 32-token blocks lie about 2^-160 apart: a factor formed as their ratio alone
    underflows fp32, while each term it would scale (a token and its neighbour) stays large.
    q = k (one shared key row per head) and values only at token 31 make those neighbour terms
    carry the second block's outputs: a kernel that drops them gets those rows wrong by 100%
    of their size, against bf16-level (< 1%) relative error when they are kept."""
    w = W.custom([70, 64], 2, seed=35, lower_bound=-5.0)
    inp = W.make_inputs(w)
    T, H, D = inp["q"].shape
    gen = torch.Generator().manual_seed(36)
    krow = torch.randn(H, D, generator=gen)
    inp["k"] = krow.expand(T, H, D).to(torch.bfloat16).contiguous()
    inp["q"] = inp["k"].clone()
    # (g + dt_bias) e^A_log = 0.85 in every channel: sigmoid 0.70, decay 5 * 0.70 nats a token
    x = 0.85 / torch.exp(inp["A_log"].float())[:, None] - inp["dt_bias"].float()
    inp["g"] = x[None].expand(T, H, D).to(torch.bfloat16).contiguous()
    v = torch.zeros_like(inp["v"])
    starts = inp["cu_seqlens"][:-1].tolist()
    for st in starts:
        v[st + 31] = inp["v"][st + 31]
    inp["v"] = v
    out, fin = run_gpu(inp, kernel)
    check(oracle_mod, inp, out, fin, tag=f"strong uniform decay k{kernel}")
    rows, o_ref, _ = oracle_sub(oracle_mod, inp, range(len(starts)), range(H), False)
    o_gpu = f64(out.cpu().index_select(0, rows))
    pos = {int(r): i for i, r in enumerate(rows.tolist())}
    for n, st in enumerate(starts):
        idx = [pos[t] for t in range(st + 32, min(st + 64, int(inp["cu_seqlens"][n + 1])))]
        ref, got = o_ref[idx], o_gpu[idx]
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 0.05, (n, rel)


def fused_views(d, extra_cols=64, beta_pad=3):
    """q, k, v, g as views into one fused [T, 4 * H * 128 + extra_cols] buffer and beta as a
    view into a wider [T, H + beta_pad] buffer (the layout of a fused projection output)."""
    T, H, D = d["q"].shape
    fused = torch.zeros(T, 4 * H * D + extra_cols, dtype=torch.bfloat16, device="cuda")
    views = {}
    for j, name in enumerate(("q", "k", "v", "g")):
        fused[:, j * H * D:(j + 1) * H * D] = d[name].reshape(T, H * D)
        views[name] = fused[:, j * H * D:(j + 1) * H * D].view(T, H, D)
    wide = torch.zeros(T, H + beta_pad, dtype=torch.bfloat16, device="cuda")
    wide[:, 1:H + 1] = d["beta"]
    views["beta"] = wide[:, 1:H + 1]
    assert not views["q"].is_contiguous() and not views["beta"].is_contiguous()
    return views


@pytest.mark.parametrize("kernel", KERNELS)
def test_strided_inputs_equal_dense(kernel):
    """The strided entry point gives exactly what the dense call gives (the same
    arithmetic on the same values)."""
    inp = W.make_inputs(W.custom([130, 64, 1, 77], 2, seed=35))
    d = to_dev(inp)
    views = fused_views(d)
    T, H = d["q"].shape[:2]
    ws = workspace_for(kernel, T, H, d["cu_seqlens"].numel() - 1)
    outs = []
    for src in (d, views):
        o, f = kda.chunk_prefill_fwd(src["q"], src["k"], src["v"], src["g"], src["beta"],
                                     d["A_log"], d["dt_bias"], d["lower_bound"], d["scale"],
                                     d["initial_state"], d["cu_seqlens"], workspace=ws,
                                     kernel=kernel)
        torch.cuda.synchronize()
        outs.append((o.clone(), f.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("kernel", KERNELS + [kda.KERNEL_AUTO])
@pytest.mark.parametrize("sd", ["f32", "bf16"])
def test_strided_inputs_against_the_oracle(oracle_mod, kernel, sd):
    """Strided q/k/v/g/beta (views of a fused projection output and of a wider beta
    buffer, as the FlashKDA prefill wrapper passes them) checked element by element
    against the oracle: several sequences over many chunks, ragged tails, a 1-token
    sequence, both state dtypes."""
    inp = W.make_inputs(W.custom([700, 64, 1, 333, 1030], 3, state_dtype=sd, seed=36))
    d = to_dev(inp)
    views = fused_views(d, extra_cols=24, beta_pad=5)
    T, H = d["q"].shape[:2]
    ws = workspace_for(kernel, T, H, d["cu_seqlens"].numel() - 1)
    out, fin = kda.chunk_prefill_fwd(views["q"], views["k"], views["v"], views["g"],
                                     views["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                                     d["scale"], d["initial_state"], d["cu_seqlens"],
                                     workspace=ws, kernel=kernel,
                                     state_dtype=inp["initial_state"].dtype)
    torch.cuda.synchronize()
    check(oracle_mod, inp, out, fin, tag=f"strided {sd} k{kernel}")


# ----------------------------------------------------------------- edge cases
@pytest.mark.parametrize("kernel", [kda.KERNEL_AUTO, kda.KERNEL_PIPE])
def test_inplace_state_update(oracle_mod, kernel):
    inp = W.make_inputs(W.custom([90, 40], 2, seed=23))
    d = to_dev(inp)
    state = d["initial_state"].clone()
    out, fin = kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                     d["dt_bias"], d["lower_bound"], d["scale"], state,
                                     d["cu_seqlens"], final_state=state, kernel=kernel)
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()
    check(oracle_mod, inp, out, fin, tag="in place")


@pytest.mark.parametrize("kernel", [kda.KERNEL_AUTO, kda.KERNEL_PIPE])
def test_null_initial_state(oracle_mod, kernel):
    inp = W.make_inputs(W.custom([70, 3], 2, seed=24))
    out, fin = run_gpu(inp, kernel, init=None)
    check(oracle_mod, inp, out, fin, zero_init=True, tag="null initial state")


@pytest.mark.parametrize("kernel", [kda.KERNEL_AUTO, kda.KERNEL_PIPE])
def test_rows_past_last_sequence_untouched(oracle_mod, kernel):
    inp = W.make_inputs(W.custom([50, 20, 128], 2, seed=25, pad_tokens=9))
    sentinel = torch.full(inp["q"].shape, 7.0, dtype=torch.bfloat16, device="cuda")
    out, fin = run_gpu(inp, kernel, out=sentinel)
    assert torch.all(out[198:].float() == 7.0)
    check(oracle_mod, inp, out, fin, tag="padded")


@pytest.mark.parametrize("kernel", [kda.KERNEL_AUTO, kda.KERNEL_PIPE])
@pytest.mark.parametrize("sd", ["f32", "bf16"])
def test_empty_sequences_pass_state_through(sd, kernel):
    inp = W.make_inputs(W.custom([0, 0, 5, 0], 2, state_dtype=sd, seed=26))
    out, fin = run_gpu(inp, kernel)
    s0 = inp["initial_state"]
    for n in (0, 1, 3):
        assert torch.equal(fin[n].cpu(), s0[n])   # bit-exact copy


def test_no_sequences_is_a_no_op():
    inp = W.make_inputs(W.custom([], 2, seed=27))
    d = to_dev(inp)
    out, fin = kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                     d["dt_bias"], d["lower_bound"], d["scale"],
                                     d["initial_state"], d["cu_seqlens"])
    torch.cuda.synchronize()
    assert fin.shape[0] == 0


@pytest.mark.parametrize("bad", [[0, 40, 20], [5, 20, 40], [0, 20, 999]])
def test_bad_cu_seqlens_reported_on_device(bad):
    inp = W.make_inputs(W.custom([20, 20], 2, seed=28))
    inp["cu_seqlens"] = torch.tensor(bad, dtype=torch.int32)
    d = to_dev(inp)
    ws = kda.alloc_workspace(40, 2, 2)
    out, fin = kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                     d["dt_bias"], d["lower_bound"], d["scale"],
                                     d["initial_state"], d["cu_seqlens"], workspace=ws)
    assert kda.last_device_status(ws) == kda.ERR_BAD_CU_SEQLENS
    assert kda.last_device_status(ws) == kda.OK      # read clears it


def test_errors_returned_with_a_device():
    inp = W.make_inputs(W.custom([20], 2, seed=29))
    d = to_dev(inp)
    with pytest.raises(kda.KDAError) as e:
        kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                              d["dt_bias"], -6.0, d["scale"], d["initial_state"],
                              d["cu_seqlens"])
    assert e.value.code == kda.ERR_UNSAFE_LOWER_BOUND
    with pytest.raises(kda.KDAError) as e:
        kda.chunk_prefill_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                              d["dt_bias"], d["lower_bound"], d["scale"], d["initial_state"],
                              d["cu_seqlens"], workspace=torch.zeros(8, dtype=torch.uint8,
                                                                      device="cuda"))
    assert e.value.code == kda.ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("kernel", [kda.KERNEL_AUTO, kda.KERNEL_PIPE, kda.KERNEL_SPLIT_STREAMED])
def test_cuda_graph_capture_and_replay(oracle_mod, kernel):
    """Capture the call on a side stream, replay it three times, compare with eager (AUTO
    takes the split path on this batch; the streamed split path, forced, runs 12 chains x
    P = 4 beside its k-side kernel)."""
    inp = W.make_inputs(W.custom([200, 64, 3], 4, seed=30))
    d = to_dev(inp)
    out_e, fin_e = run_gpu(inp, kernel)
    out = torch.empty_like(d["q"])
    fin = torch.empty_like(d["initial_state"])
    ws = kda.alloc_workspace(d["q"].shape[0], 4, 3)
    side = torch.cuda.Stream()
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
            d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):        # warm-up outside capture
        kda.chunk_prefill_fwd(*args, out=out, final_state=fin, workspace=ws, stream=side,
                              kernel=kernel)
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        kda.chunk_prefill_fwd(*args, out=out, final_state=fin, workspace=ws, stream=side,
                              kernel=kernel)
    for _ in range(3):
        out.zero_()
        fin.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_e) and torch.equal(fin, fin_e)
    assert kda.last_device_status(ws) == kda.OK


# ----------------------------------------------------------------- k-side helpers
@pytest.mark.parametrize("lengths,H", [([2048] * 8, 16), ([300, 1000, 64, 129, 0, 700], 2),
                                        ([4096, 64, 1, 4000], 4)])
def test_helpers_agree_with_the_fused_kernel_alone(oracle_mod, lengths, H):
    """The fused kernel with helper CTAs computes the chunk-local half of some chunks in
    the helpers' records; which chunks depends on timing.  Its results match the fused
    kernel alone and the oracle, on the benchmark shape and on small batches where the
    helpers take nearly every chunk."""
    inp = W.make_inputs(W.custom(lengths, H, seed=41))
    out_t, fin_t = run_gpu(inp, kda.KERNEL_TC, vsplit=1)
    out_h, fin_h = run_gpu(inp, kda.KERNEL_TC_HELPERS)
    same = torch.equal(out_t, out_h) and torch.equal(fin_t, fin_h)
    d_o = (out_t.float() - out_h.float()).abs().max().item()
    d_f = (fin_t - fin_h).abs().max().item()
    print(f"helpers vs alone: bitwise {same}, out {d_o:.3e}, state {d_f:.3e}")
    assert d_o <= TOL["f32"] and d_f <= TOL["f32"]
    N = len(lengths)
    heads = list(range(H)) if H <= 4 else [0, 7, 15]
    check(oracle_mod, inp, out_h, fin_h, heads=heads, tag=f"helpers {N}x{H}")


def test_auto_dispatch_on_the_device():
    """8 x 2048, H = 16 keeps more than 5/8 of the 152 SMs busy: AUTO runs the
    warp-specialised kernel; 5 x 2048 (80 chains) leaves enough free for helpers."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    max_chains = min(sms - 8, 5 * sms // 8)
    T, N, H = 16384, 8, 16
    path, P, launches = kda.plan(T, N, H, kda.workspace_size(T, H, N), -1, kda.KERNEL_AUTO)
    if N * H > max_chains:
        assert (path, P, launches) == (kda.KERNEL_PIPE, 1, 1)
    T, N = 10240, 5
    path, P, launches = kda.plan(T, N, H, kda.workspace_size(T, H, N), -1, kda.KERNEL_AUTO)
    if N * H <= max_chains and 2 * N * H > sms:
        assert (path, P, launches) == (kda.KERNEL_TC_HELPERS, 1, 2)
    path, P, launches = kda.plan(T, N, H, 256, -1, kda.KERNEL_AUTO)   # no room for records
    assert (path, P, launches) == (kda.KERNEL_PIPE, 1, 1)


def test_helpers_under_cuda_graph_replay(oracle_mod):
    """The helper grid is a programmatic dependent of the fused kernel; a captured call
    replays to the eager result's values."""
    inp = W.make_inputs(W.custom([700, 300, 1000], 2, seed=42))
    d = to_dev(inp)
    T = d["q"].shape[0]
    out = torch.empty_like(d["q"])
    fin = torch.empty_like(d["initial_state"])
    ws = helper_workspace(T, 2, 3)
    side = torch.cuda.Stream()
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
            d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        kda.chunk_prefill_fwd(*args, out=out, final_state=fin, workspace=ws, stream=side,
                              kernel=kda.KERNEL_TC_HELPERS)
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        kda.chunk_prefill_fwd(*args, out=out, final_state=fin, workspace=ws, stream=side,
                              kernel=kda.KERNEL_TC_HELPERS)
    for _ in range(3):
        out.zero_()
        fin.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert kda.last_device_status(ws) == kda.OK
        check(oracle_mod, inp, out, fin, tag="helpers graph replay")


def test_helpers_refused_when_they_cannot_run():
    inp = W.make_inputs(W.custom([100, 50], 2, seed=43))
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
            d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])
    with pytest.raises(kda.KDAError) as e:    # records do not fit
        kda.chunk_prefill_fwd(*args, workspace=split_workspace(150, 2, 2),
                              kernel=kda.KERNEL_TC_HELPERS)
    assert e.value.code == kda.ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(kda.KDAError) as e:    # a value split is not served
        kda.chunk_prefill_fwd(*args, workspace=helper_workspace(150, 2, 2),
                              kernel=kda.KERNEL_TC_HELPERS, vsplit=2)
    assert e.value.code == kda.ERR_INVALID_ARG


def test_bounded_wait_runs_out_and_the_context_survives():
    """Failure detection without a GPU fault: with the library's test hook on
    (kda_test_drop_one_record) the first helper CTA claims its first chunk and never
    publishes the record.  The fused CTA that needs it waits a bounded time (about a
    second), records KDA_ERR_DEVICE_TIMEOUT in the workspace and ends; the next call on the
    same context and workspace is correct."""
    inp = W.make_inputs(W.custom([1024, 1024], 2, seed=44))
    d = to_dev(inp)
    T = d["q"].shape[0]
    ws = helper_workspace(T, 2, 2)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
            d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])
    kda.test_drop_one_record(True)
    try:
        kda.chunk_prefill_fwd(*args, workspace=ws, kernel=kda.KERNEL_TC_HELPERS)
        torch.cuda.synchronize()
    finally:
        kda.test_drop_one_record(False)
    assert kda.last_device_status(ws) == kda.ERR_DEVICE_TIMEOUT
    out, fin = kda.chunk_prefill_fwd(*args, workspace=ws, kernel=kda.KERNEL_TC_HELPERS)
    torch.cuda.synchronize()
    assert kda.last_device_status(ws) == kda.OK
    out_t, fin_t = run_gpu(inp, kda.KERNEL_TC, vsplit=1)
    assert torch.equal(out, out_t) and torch.equal(fin, fin_t)


def test_streamed_split_beside_other_work():
    """The streamed split path relies on no placement: with the warp-specialised kernel of
    another batch filling most SMs from a second stream, and a second streamed call on a
    third, every call still completes with status OK and the same bits as run alone (its
    k-side CTAs that cannot start at once start later; the chains wait for records a bounded
    time, far longer than the other work takes)."""
    inp_a = W.make_inputs(W.custom([4096], 8, seed=71))
    inp_b = W.make_inputs(W.custom([2048] * 8, 16, seed=72))
    inp_c = W.make_inputs(W.custom([4096, 4096], 8, seed=73))
    alone = [run_gpu(inp_a, kda.KERNEL_SPLIT_STREAMED), run_gpu(inp_b, kda.KERNEL_PIPE),
             run_gpu(inp_c, kda.KERNEL_SPLIT_STREAMED)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    calls = []
    for inp, kern, s in zip((inp_a, inp_b, inp_c),
                            (kda.KERNEL_SPLIT_STREAMED, kda.KERNEL_PIPE, kda.KERNEL_SPLIT_STREAMED),
                            streams):
        d = to_dev(inp)
        T, H, N = d["q"].shape[0], d["q"].shape[1], d["cu_seqlens"].numel() - 1
        ws = helper_workspace(T, H, N)
        calls.append((d, kern, s, ws))
    torch.cuda.synchronize()
    results = []
    for _ in range(3):   # several rounds, the three calls in flight together each time
        outs = []
        for d, kern, s, ws in (calls[1], calls[0], calls[2]):   # the big one first
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                outs.append(kda.chunk_prefill_fwd(
                    d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                    d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"],
                    workspace=ws, stream=s, kernel=kern))
        torch.cuda.synchronize()
        for d, kern, s, ws in calls:
            assert kda.last_device_status(ws) == kda.OK
        results.append([outs[1], outs[0], outs[2]])
    for res in results:
        for (o, f), (o_ref, f_ref) in zip(res, alone):
            assert torch.equal(o, o_ref) and torch.equal(f, f_ref)
