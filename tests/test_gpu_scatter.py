"""GPU: outputs written through a row map (kda_chunk_prefill_fwd_scatter,
kda_recurrent_fwd_scatter).

The mixed speculative step of the FlashKDA prefill PR report (PR #55737,
Implementation breakdown item 4) prefills the non-speculative tokens into a
workspace buffer and scatters it into the layer output with index_copy_; the
speculative tokens go through the recurrent form.  With a row map each kernel
writes the layer output directly.  Every path must place exactly the rows the
dense call computes (the same arithmetic, so bit for bit), leave other rows
alone, and report map entries outside the buffer.
"""
import numpy as np
import pytest
import torch

import kda_gated_delta_chunk_gb300 as kda
import kda_workloads as W

pytestmark = pytest.mark.gpu


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


def args_of(d):
    return (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
            d["lower_bound"], d["scale"], d["initial_state"], d["cu_seqlens"])


def records_ws(T, H, N):
    return torch.zeros(1024 + ((T + 63) // 64 + N) * H * (66560 + 4), dtype=torch.uint8,
                       device="cuda")


SENTINEL = 3.0


def scattered(T, H, extra, seed):
    """A random one-to-one map of the T tokens into T + extra rows, and a sentinel buffer."""
    gen = torch.Generator().manual_seed(seed)
    rows = torch.randperm(T + extra, generator=gen)[:T].to(torch.int32)
    buf = torch.full((T + extra, H, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
    return rows.cuda(), buf


def check_placed(buf, rows, dense, T_used):
    rows_c = rows.long().cpu()
    got = buf.cpu()
    assert torch.equal(got[rows_c[:T_used]], dense.cpu()[:T_used])
    untouched = torch.ones(buf.shape[0], dtype=torch.bool)
    untouched[rows_c[:T_used]] = False
    assert torch.all(got[untouched].float() == SENTINEL)


@pytest.mark.parametrize("kernel,vsplit", [(kda.KERNEL_TC, 1), (kda.KERNEL_TC, 2),
                                           (kda.KERNEL_TC_HELPERS, -1), (kda.KERNEL_SPLIT, 1),
                                           (kda.KERNEL_SPLIT, 2), (kda.KERNEL_SPLIT, 4),
                                           (kda.KERNEL_SPLIT, 8), (kda.KERNEL_REF, 1),
                                           (kda.KERNEL_PIPE, 1),
                                           (kda.KERNEL_SPLIT_STREAMED, 4)])
def test_prefill_scatter_places_the_dense_rows(kernel, vsplit):
    """Ragged sequences (a 1-token and an empty one, tails), tokens past cu_seqlens[N]."""
    inp = W.make_inputs(W.custom([130, 1, 0, 64, 257, 70], 2, seed=61, pad_tokens=5))
    d = dev(inp)
    T, H = d["q"].shape[0], 2
    N = d["cu_seqlens"].numel() - 1
    T_used = int(inp["cu_seqlens"][-1])
    ws = records_ws(T, H, N)
    dense, fin_d = kda.chunk_prefill_fwd(*args_of(d), workspace=ws, kernel=kernel, vsplit=vsplit)
    torch.cuda.synchronize()
    rows, buf = scattered(T, H, 11, 62)
    out, fin = kda.chunk_prefill_fwd(*args_of(d), out=buf, workspace=ws, kernel=kernel,
                                     vsplit=vsplit, out_index=rows)
    torch.cuda.synchronize()
    assert kda.last_device_status(ws) == kda.OK
    assert out.data_ptr() == buf.data_ptr()
    check_placed(buf, rows, dense, T_used)
    assert torch.equal(fin, fin_d)


def test_prefill_scatter_on_the_benchmark_shape():
    """8 x 2048, H = 16 through AUTO (the warp-specialised kernel): rows in reverse order."""
    inp = W.make_inputs(W.workload(1))
    d = dev(inp)
    T, H, N = d["q"].shape[0], 16, 8
    ws = kda.alloc_workspace(T, H, N)
    dense, _ = kda.chunk_prefill_fwd(*args_of(d), workspace=ws)
    rows = torch.arange(T - 1, -1, -1, dtype=torch.int32, device="cuda")
    buf = torch.full((T, H, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
    kda.chunk_prefill_fwd(*args_of(d), out=buf, workspace=ws, out_index=rows)
    torch.cuda.synchronize()
    assert kda.last_device_status(ws) == kda.OK
    assert torch.equal(buf.flip(0), dense)


def test_recurrent_scatter_places_the_dense_rows():
    inp = W.make_inputs(W.custom([3, 1, 4, 2], 2, seed=63))
    d = dev(inp)
    T, H = d["q"].shape[0], 2
    dense, fin_d, _ = kda.recurrent_fwd(*args_of(d))
    rows, buf = scattered(T, H, 5, 64)
    out, fin, _ = kda.recurrent_fwd(*args_of(d), out=buf, out_index=rows)
    torch.cuda.synchronize()
    check_placed(buf, rows, dense, T)
    assert torch.equal(fin, fin_d)


def test_mixed_step_writes_one_layer_output(oracle_mod):
    """A mixed step: three prefill sequences and two sequences with 3 speculative tokens,
    interleaved in one layer output [T_all, H, 128].  The prefill writes its rows through
    non_spec_token_indx, the recurrent form through spec_token_indx; together they fill
    every row, each equal to the oracle's output for its token."""
    H = 2
    pre = W.make_inputs(W.custom([150, 70, 9], H, seed=65))
    spec = W.make_inputs(W.custom([3, 3], H, seed=66))
    Tp, Ts = pre["q"].shape[0], spec["q"].shape[0]
    order = torch.randperm(Tp + Ts, generator=torch.Generator().manual_seed(67)).to(torch.int32)
    non_spec_idx, spec_idx = order[:Tp].cuda(), order[Tp:].cuda()
    layer_out = torch.full((Tp + Ts, H, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
    dp, ds = dev(pre), dev(spec)
    kda.chunk_prefill_fwd(*args_of(dp), out=layer_out, out_index=non_spec_idx)
    kda.recurrent_fwd(*args_of(ds), out=layer_out, out_index=spec_idx)
    torch.cuda.synchronize()
    f = lambda t: t.float().double().numpy()
    tol = 0.01
    for inp, idx in ((pre, non_spec_idx), (spec, spec_idx)):
        o_ref, _ = oracle_mod.kda_oracle_fwd(
            f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["g"]), f(inp["beta"]),
            f(inp["A_log"]), f(inp["dt_bias"]), inp["lower_bound"], inp["scale"],
            f(inp["initial_state"]), inp["cu_seqlens"].numpy())
        got = layer_out.cpu()[idx.long().cpu()].float().double().numpy()
        assert np.abs(got - o_ref).max() <= tol


@pytest.mark.parametrize("kernel", [kda.KERNEL_TC, kda.KERNEL_SPLIT, kda.KERNEL_REF,
                                    kda.KERNEL_PIPE])
def test_out_of_range_rows_are_reported_and_skipped(kernel):
    inp = W.make_inputs(W.custom([100, 40], 2, seed=68))
    d = dev(inp)
    T, H = d["q"].shape[0], 2
    ws = records_ws(T, H, 2)
    dense, _ = kda.chunk_prefill_fwd(*args_of(d), workspace=ws, kernel=kernel, vsplit=1)
    torch.cuda.synchronize()
    rows = torch.arange(T, dtype=torch.int32)
    rows[7] = -1
    rows[90] = T      # one past the buffer
    buf = torch.full((T, H, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
    kda.chunk_prefill_fwd(*args_of(d), out=buf, workspace=ws, kernel=kernel, vsplit=1,
                          out_index=rows.cuda())
    assert kda.last_device_status(ws) == kda.ERR_BAD_OUT_INDEX
    keep = torch.ones(T, dtype=torch.bool)
    keep[7] = keep[90] = False
    assert torch.equal(buf.cpu()[keep], dense.cpu()[keep])
    assert torch.all(buf.cpu()[7].float() == SENTINEL) and torch.all(buf.cpu()[90].float() == SENTINEL)
