"""Host-side checks of libkda.so that need no GPU.

The library must load, export every function include/kda.h declares, size
the workspace, choose the value split as the V-split PR report states, and
refuse bad arguments with its documented codes before touching a device.
"""
import ctypes
import json
import os
import re

import pytest

import kda_gated_delta_chunk_gb300 as kda
import kda_workloads as W
from kda_gated_delta_chunk_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kda.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert len(names) >= 7
    for name in names:
        assert hasattr(L, name), name
    assert set(names) == set(kda.EXPORTS)


def test_workspace_size(L):
    n = kda.workspace_size(16384, 16, 8)
    assert n >= 16 and n % 16 == 0
    assert kda.workspace_size(-1, 16, 8) == 0
    assert kda.workspace_size(0, 0, 0) >= 0


SLOT_HEAD_BYTES = 66560      # one split-path record: 3 tiles 64x128 + 2 tiles 64x64 bf16 + 1 KB


def _sms():
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    except Exception:
        pass
    return 152               # the library's assumption when no device answers


def test_workspace_size_holds_split_records(L):
    """Records for ceil(T/64) + N chunk slots per head whenever some batch of up to
    max_seqs sequences would take the value split (2 H N <= SMs) or the k-side helpers
    (H N <= min(SMs - 8, 5 SMs / 8), N <= 128; plus a 4-byte claim word per slot and head),
    else 256 bytes; rounded up to 16."""
    sms = _sms()
    cases = [(1000, 2, 3), (16384, 16, 1), (16384, 16, 8), (4096, 8, 7), (64, 1, 500),
             (65536, 32, 64), (65536, 160, 2)]
    for T, H, N in cases:
        got = kda.workspace_size(T, H, N)
        need = 256
        if 2 * H <= sms:
            n_split = min(N, sms // (2 * H))
            need = max(need, 1024 + ((T + 63) // 64 + n_split) * H * SLOT_HEAD_BYTES)
        max_chains = min(sms - 8, 5 * sms // 8)
        if H <= max_chains:
            n_help = min(N, 128, max_chains // H)
            need = max(need, 1024 + ((T + 63) // 64 + n_help) * H * (SLOT_HEAD_BYTES + 4))
        assert got == (need + 15) // 16 * 16, (T, H, N)
        assert got % 16 == 0
    assert kda.workspace_size(0, 4, 2) == 256          # no tokens, no records
    assert kda.workspace_size(100, 4, 0) == 256


def test_vsplit_boundary_matches_pages(L):
    g = json.load(open(os.path.join(GOLDEN, "vsplit_boundary.json")))
    for case in g["cases"]:
        for h in case["heads"]:
            split = [n for n in range(1, 40) if kda.choose_vsplit(n, h, case["sm_count"]) > 1]
            assert split == list(range(1, case["max_split_seqs"] + 1)), (case, h)


def test_vsplit_factor_values(L):
    assert kda.choose_vsplit(8, 16, 152) == 1        # 8x2048, H=16: 256 > 152
    assert kda.choose_vsplit(1, 16, 152) == 8        # 1x16384, H=16
    assert kda.choose_vsplit(7, 8, 152) == 2
    assert kda.choose_vsplit(3, 8, 152) == 4
    assert kda.choose_vsplit(1, 8, 152) == 8
    assert kda.choose_vsplit(0, 8, 152) == 1
    for n in range(1, 30):
        for h in (1, 4, 8, 16, 32):
            p = kda.choose_vsplit(n, h, 152)
            assert p in (1, 2, 4, 8)
            assert p == 1 or p * n * h <= 152


# ------------------------------------------------------------------ dispatch, no device
GB300_SMS = 152


def _auto(lengths, H, ws=None, sms=GB300_SMS, **kw):
    T, N = sum(lengths), len(lengths)
    ws = kda.workspace_size(T, H, N) if ws is None else ws
    return kda.plan_for(T, N, H, ws, sms, **kw)


def _records_only(lengths, H):
    """Bytes of the split path's header and records, without the helpers' claim words."""
    T, N = sum(lengths), len(lengths)
    return 1024 + ((T + 63) // 64 + N) * H * 66560


@pytest.mark.parametrize("shape,H,want", [
    ("tiny", 2, (kda.KERNEL_SPLIT, 8, 2)),                 # 1 x 128: too short to stream
    ("batched", 16, (kda.KERNEL_PIPE, 1, 1)),              # 128 chains: over 5/8 of the SMs
    ("long", 16, (kda.KERNEL_SPLIT_STREAMED, 4, 2)),       # 1 x 16384: 64 chain CTAs
    ("v1", 8, (kda.KERNEL_SPLIT_STREAMED, 8, 2)),          # N x 4096, H = 8
    ("v2", 8, (kda.KERNEL_SPLIT_STREAMED, 4, 2)),
    ("v3", 8, (kda.KERNEL_SPLIT_STREAMED, 2, 2)),          # 24 x 2 chain CTAs
    ("v7", 8, (kda.KERNEL_SPLIT_STREAMED, 1, 2)),          # 56 unsplit chain CTAs
    ("ragged", 32, (kda.KERNEL_PIPE, 1, 1)),               # 2048 chains: no SM left over
])
def test_auto_dispatch_of_the_benchmark_shapes(L, shape, H, want):
    lengths = {"tiny": [128], "batched": [2048] * 8, "long": [16384], "v1": [4096],
               "v2": [4096] * 2, "v3": [4096] * 3, "v7": [4096] * 7,
               "ragged": list(W.workload(4).lengths)}[shape]
    assert _auto(lengths, H) == want


def test_auto_helper_conditions(L):
    # helpers while at most min(SMs - 8, 5 SMs / 8) chains run (95 of 152), else the
    # warp-specialised kernel: 11 x 8 = 88 chains and 12 x 8 = 96
    assert _auto([2048] * 11, 8)[0] == kda.KERNEL_TC_HELPERS
    assert _auto([2048] * 12, 8) == (kda.KERNEL_PIPE, 1, 1)
    # 5 x 16 = 80 chains: 5/8 of 128 SMs is 80, of 127 it is 79
    assert _auto([2048] * 5, 16, sms=128)[0] == kda.KERNEL_TC_HELPERS
    assert _auto([2048] * 5, 16, sms=127)[0] == kda.KERNEL_PIPE
    # on a small part the 8 free SMs bind first: 5/8 of 20 is 12, 20 - 8 = 12 as well;
    # 13 chains of 1 head exceed both
    assert _auto([256] * 12, 1, sms=20)[0] == kda.KERNEL_TC_HELPERS
    assert _auto([256] * 13, 1, sms=20)[0] == kda.KERNEL_PIPE
    # sequences of at least 4 chunks on average
    assert _auto([256] * 5, 16)[0] == kda.KERNEL_TC_HELPERS
    assert _auto([255] * 5, 16)[0] == kda.KERNEL_PIPE
    # the claim words must fit as well as the records
    lengths = [2048] * 5
    assert _auto(lengths, 16, ws=_records_only(lengths, 16)) == (kda.KERNEL_PIPE, 1, 1)
    claims = ((sum(lengths) + 63) // 64 + len(lengths)) * 16 * 4   # a word per (slot, head)
    assert _auto(lengths, 16, ws=_records_only(lengths, 16) + claims - 4)[0] == kda.KERNEL_PIPE
    assert _auto(lengths, 16, ws=_records_only(lengths, 16) + claims)[0] == \
        kda.KERNEL_TC_HELPERS


def test_auto_streamed_split_conditions(L):
    # P = 8 while 2 N H 8 <= SMs, else P = 4 while 2 N H 4 <= SMs, else P = 2 while
    # 2 N H 2 <= SMs, else the plain split
    assert _auto([4096] * 9, 1) == (kda.KERNEL_SPLIT_STREAMED, 8, 2)
    # sequences of 2048 tokens or more on average
    assert _auto([2048], 8) == (kda.KERNEL_SPLIT_STREAMED, 8, 2)
    assert _auto([2047], 8) == (kda.KERNEL_SPLIT, 8, 2)
    assert _auto([4000, 96], 4) == (kda.KERNEL_SPLIT_STREAMED, 8, 2)
    assert _auto([4000, 95], 4) == (kda.KERNEL_SPLIT, 8, 2)
    assert _auto([4096] * 10, 1) == (kda.KERNEL_SPLIT_STREAMED, 4, 2)
    assert _auto([4096] * 19, 1) == (kda.KERNEL_SPLIT_STREAMED, 4, 2)
    assert _auto([4096] * 20, 1) == (kda.KERNEL_SPLIT_STREAMED, 2, 2)
    assert _auto([4096] * 38, 1) == (kda.KERNEL_SPLIT_STREAMED, 2, 2)
    assert _auto([4096] * 39, 1) == (kda.KERNEL_SPLIT_STREAMED, 1, 2)   # 8 x 39 <= 3 x 152
    assert _auto([4096] * 57, 1) == (kda.KERNEL_SPLIT_STREAMED, 1, 2)
    assert _auto([4096] * 58, 1) == (kda.KERNEL_SPLIT, 2, 2)
    # the claim words must fit as well as the records
    lengths = [4096] * 2
    assert _auto(lengths, 8, ws=_records_only(lengths, 8)) == (kda.KERNEL_SPLIT, 8, 2)
    claims = ((sum(lengths) + 63) // 64 + len(lengths)) * 8 * 4
    assert _auto(lengths, 8, ws=_records_only(lengths, 8) + claims - 4) == (kda.KERNEL_SPLIT, 8, 2)
    assert _auto(lengths, 8, ws=_records_only(lengths, 8) + claims) == \
        (kda.KERNEL_SPLIT_STREAMED, 4, 2)
    # at most 128 sequences (shown on a part with enough SMs for the split)
    def full(lengths, H):   # records and claim words
        return 1024 + ((sum(lengths) + 63) // 64 + len(lengths)) * H * (66560 + 4)
    assert _auto([2048] * 128, 1, sms=4096, ws=full([2048] * 128, 1)) == \
        (kda.KERNEL_SPLIT_STREAMED, 8, 2)
    assert _auto([2048] * 129, 1, sms=4096, ws=full([2048] * 129, 1)) == \
        (kda.KERNEL_SPLIT, 8, 2)
    # a split factor given by the caller keeps the plain split under AUTO
    assert _auto([16384], 16, vsplit=4) == (kda.KERNEL_SPLIT, 4, 2)


def test_forced_streamed_split(L):
    assert _auto([16384], 16, kernel=kda.KERNEL_SPLIT_STREAMED) == (kda.KERNEL_SPLIT_STREAMED, 4, 2)
    assert _auto([16384], 16, kernel=kda.KERNEL_SPLIT_STREAMED, vsplit=2) == \
        (kda.KERNEL_SPLIT_STREAMED, 2, 2)
    assert _auto([16384], 16, kernel=kda.KERNEL_SPLIT_STREAMED, vsplit=1) == \
        (kda.KERNEL_SPLIT_STREAMED, 1, 2)
    assert _auto([4096], 8, kernel=kda.KERNEL_SPLIT_STREAMED, vsplit=4) == \
        (kda.KERNEL_SPLIT_STREAMED, 4, 2)
    refused = [
        (dict(vsplit=3), kda.ERR_INVALID_ARG),
        (dict(vsplit=8), kda.ERR_INVALID_ARG),                 # 2 x 16 x 8 > 152
        (dict(sms=127, vsplit=4), kda.ERR_INVALID_ARG),        # 2 x 16 x 4 > 127
        (dict(sms=63, vsplit=2), kda.ERR_INVALID_ARG),         # 2 x 16 x 2 > 63
        (dict(sms=42), kda.ERR_INVALID_ARG),                   # and 8 x 16 > 3 x 42
        (dict(ws=_records_only([16384], 16)), kda.ERR_WORKSPACE_TOO_SMALL),
    ]
    for kw, code in refused:
        with pytest.raises(kda.KDAError) as e:
            _auto([16384], 16, kernel=kda.KERNEL_SPLIT_STREAMED, **kw)
        assert e.value.code == code, kw
    # no tokens: one launch writes the states
    ws = 1024 + (0 + 1) * 8 * (66560 + 4)   # one slot per sequence
    assert kda.plan_for(0, 1, 8, ws, GB300_SMS, kernel=kda.KERNEL_SPLIT_STREAMED) == \
        (kda.KERNEL_SPLIT_STREAMED, 8, 1)


def test_auto_without_room_for_records_runs_the_fused_kernel(L):
    # the value split triggers, but a bare status workspace holds no records
    assert _auto([16384], 16, ws=256) == (kda.KERNEL_PIPE, 1, 1)
    # a split factor given by the caller stays, on the fused kernel
    assert _auto([16384], 16, ws=256, vsplit=4) == (kda.KERNEL_TC, 4, 1)
    assert _auto([16384], 16, ws=_records_only([16384], 16)) == (kda.KERNEL_SPLIT, 8, 2)


def test_forced_kernels_and_refusals(L):
    # a forced split with records for all eight sequences (more than the default workspace
    # of eight sequences holds: AUTO takes neither the split nor helpers there)
    assert _auto([2048] * 8, 16, kernel=kda.KERNEL_SPLIT, ws=_records_only([2048] * 8, 16)) == \
        (kda.KERNEL_SPLIT, 1, 2)
    assert _auto([2048] * 8, 16, kernel=kda.KERNEL_TC) == (kda.KERNEL_TC, 1, 1)
    assert _auto([2048] * 8, 16, kernel=kda.KERNEL_REF) == (kda.KERNEL_REF, 1, 1)
    assert _auto([16384], 16, kernel=kda.KERNEL_TC_HELPERS) == (kda.KERNEL_TC_HELPERS, 1, 2)
    refused = [
        (dict(kernel=kda.KERNEL_SPLIT, ws=256), kda.ERR_WORKSPACE_TOO_SMALL),
        (dict(kernel=kda.KERNEL_TC_HELPERS, ws=256), kda.ERR_WORKSPACE_TOO_SMALL),
        (dict(kernel=kda.KERNEL_TC_HELPERS, vsplit=2), kda.ERR_INVALID_ARG),
        (dict(kernel=kda.KERNEL_TC_HELPERS, sms=128), kda.ERR_INVALID_ARG),   # no SM free
        (dict(vsplit=3), kda.ERR_INVALID_ARG),
        (dict(kernel=99), kda.ERR_INVALID_ARG),
        (dict(sms=0), kda.ERR_INVALID_ARG),
        (dict(ws=255), kda.ERR_WORKSPACE_TOO_SMALL),
    ]
    for kw, code in refused:
        with pytest.raises(kda.KDAError) as e:
            _auto([2048] * 8, 16, **kw)
        assert e.value.code == code, kw
    with pytest.raises(kda.KDAError) as e:
        kda.plan_for(2048, 1, 0, 1 << 20, GB300_SMS)     # no heads
    assert e.value.code == kda.ERR_INVALID_ARG


def test_launch_counts_of_degenerate_batches(L):
    assert kda.plan_for(0, 0, 16, 256, GB300_SMS) == (kda.KERNEL_PIPE, 1, 0)   # no sequences
    # sequences that are all empty: no records to make, one launch writes the states
    assert kda.plan_for(0, 3, 8, 1 << 20, GB300_SMS) == (kda.KERNEL_PIPE, 1, 1)
    # a forced split path keeps its documented record area, a slot per sequence included
    ws = _records_only([0, 0, 0], 8)
    assert kda.plan_for(0, 3, 8, ws, GB300_SMS, kernel=kda.KERNEL_SPLIT) == (kda.KERNEL_SPLIT, 4, 1)
    with pytest.raises(kda.KDAError) as e:
        kda.plan_for(0, 3, 8, 1 << 20, GB300_SMS, kernel=kda.KERNEL_SPLIT)
    assert e.value.code == kda.ERR_WORKSPACE_TOO_SMALL


def test_status_strings(L):
    for code in range(-10, 1):
        assert kda.status_string(code) and kda.status_string(code) != "unknown status"
    assert kda.status_string(-99) == "unknown status"


def _call(L, **over):
    """Call kda_chunk_prefill_fwd_ex with fake (never dereferenced) pointers."""
    a = dict(q=0x10000, k=0x20000, v=0x30000, g=0x40000, beta=0x50000, A_log=0x60000,
             dt_bias=0x70000, lb=-5.0, scale=128 ** -0.5, s0=0x80000, cu=0x90000,
             out=0xA0000, fin=0xB0000, sd=0, ws=0xC0000, stream=None, T=64, N=1, H=2,
             wsb=kda.workspace_size(64, 2, 1), vsplit=-1, kernel=0)
    a.update(over)
    P = ctypes.c_void_p
    return L.kda_chunk_prefill_fwd_ex(
        P(a["q"]), P(a["k"]), P(a["v"]), P(a["g"]), P(a["beta"]), P(a["A_log"]),
        P(a["dt_bias"]), a["lb"], a["scale"], P(a["s0"]), P(a["cu"]), P(a["out"]),
        P(a["fin"]), a["sd"], P(a["ws"]), P(a["stream"]), a["T"], a["N"], a["H"], a["wsb"],
        a["vsplit"], a["kernel"])


@pytest.mark.parametrize("over,code", [
    (dict(lb=-6.0), kda.ERR_UNSAFE_LOWER_BOUND),
    (dict(lb=-5.01), kda.ERR_UNSAFE_LOWER_BOUND),
    (dict(lb=0.5), kda.ERR_UNSAFE_LOWER_BOUND),
    (dict(lb=float("nan")), kda.ERR_INVALID_ARG),
    (dict(scale=float("inf")), kda.ERR_INVALID_ARG),
    (dict(H=0), kda.ERR_INVALID_ARG),
    (dict(T=-1), kda.ERR_INVALID_ARG),
    (dict(N=-1), kda.ERR_INVALID_ARG),
    (dict(sd=2), kda.ERR_INVALID_ARG),
    (dict(q=0), kda.ERR_INVALID_ARG),
    (dict(out=0), kda.ERR_INVALID_ARG),
    (dict(cu=0), kda.ERR_INVALID_ARG),
    (dict(fin=0), kda.ERR_INVALID_ARG),
    (dict(fin=0, N=0, T=0), kda.ERR_CUDA),
    (dict(ws=0), kda.ERR_INVALID_ARG),
    (dict(wsb=8), kda.ERR_WORKSPACE_TOO_SMALL),
    (dict(q=0x10008), kda.ERR_MISALIGNED),
    (dict(fin=0xB0004), kda.ERR_MISALIGNED),
    (dict(beta=0x50001), kda.ERR_MISALIGNED),
    (dict(vsplit=3), kda.ERR_INVALID_ARG),
    (dict(kernel=7), kda.ERR_INVALID_ARG),
    (dict(kernel=-1), kda.ERR_INVALID_ARG),
])
def test_argument_gate(L, over, code):
    assert _call(L, **over) == code


def _call_strided(L, strides):
    P = ctypes.c_void_p
    return L.kda_chunk_prefill_fwd_strided(
        P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000), P(0x60000), P(0x70000),
        -5.0, 128 ** -0.5, P(0x80000), P(0x90000), P(0xA0000), P(0xB0000), 0, P(0xC0000),
        P(None), 64, 1, 2, kda.workspace_size(64, 2, 1), *strides, -1, 0)


@pytest.mark.parametrize("strides,code", [
    ((255, 256, 256, 256, 2), kda.ERR_INVALID_ARG),      # q rows overlap (H * 128 = 256)
    ((256, 256, 256, 256, 1), kda.ERR_INVALID_ARG),      # beta rows overlap (H = 2)
    ((260, 256, 256, 256, 2), kda.ERR_MISALIGNED),       # 16-byte TMA rows: multiple of 8
    ((256, 256, 260, 256, 2), kda.ERR_MISALIGNED),
    ((0, 256, 256, 256, 2), kda.ERR_INVALID_ARG),
])
def test_strided_argument_gate(L, strides, code):
    assert _call_strided(L, strides) == code


def test_valid_arguments_reach_the_device_check(L):
    """Valid arguments pass validation; without an sm_103 GPU the call then
    stops at the device check and enqueues nothing."""
    rc = _call(L)
    import torch
    if not torch.cuda.is_available():
        assert rc in (kda.ERR_CUDA, kda.ERR_UNSUPPORTED_DEVICE)


def test_recurrent_argument_gate(L):
    """kda_recurrent_fwd refuses bad arguments on the host, before any device work."""
    P = ctypes.c_void_p
    base = [P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000), P(0x60000),
            P(0x70000), -5.0, 128 ** -0.5, P(0x80000), P(0x90000), P(0xA0000), P(0xB0000), 0]
    assert L.kda_recurrent_fwd(*base, P(0xD0004), P(0xC0000), P(None), 4, 1, 2, 256) == \
        kda.ERR_MISALIGNED                                   # token_states not 16-byte aligned
    assert L.kda_recurrent_fwd(*base, P(None), P(0xC0000), P(None), 4, 1, 2, 8) == \
        kda.ERR_WORKSPACE_TOO_SMALL
    base[7] = -7.0
    assert L.kda_recurrent_fwd(*base, P(None), P(0xC0000), P(None), 4, 1, 2, 256) == \
        kda.ERR_UNSAFE_LOWER_BOUND


def _call_scatter(L, index, rows):
    P = ctypes.c_void_p
    return L.kda_chunk_prefill_fwd_scatter(
        P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000), P(0x60000), P(0x70000),
        -5.0, 128 ** -0.5, P(0x80000), P(0x90000), P(0xA0000), P(0xB0000), 0, P(0xC0000),
        P(None), 64, 1, 2, kda.workspace_size(64, 2, 1), 256, 256, 256, 256, 2, P(index),
        rows, -1, 0)


@pytest.mark.parametrize("index,rows,code", [
    (None, 64, kda.ERR_INVALID_ARG),        # the map is required
    (0xD0000, -1, kda.ERR_INVALID_ARG),     # negative row count
    (0xD0002, 64, kda.ERR_MISALIGNED),      # int32 map: 4-byte aligned
])
def test_scatter_argument_gate(L, index, rows, code):
    """kda_chunk_prefill_fwd_scatter / kda_recurrent_fwd_scatter refuse a missing or
    misaligned row map and a negative row count on the host."""
    assert _call_scatter(L, index, rows) == code
    P = ctypes.c_void_p
    base = [P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000), P(0x60000),
            P(0x70000), -5.0, 128 ** -0.5, P(0x80000), P(0x90000), P(0xA0000), P(0xB0000), 0,
            P(None), P(0xC0000), P(None), 4, 1, 2, 256]
    assert L.kda_recurrent_fwd_scatter(*base, P(index), rows) == code


def test_scatter_valid_arguments_reach_the_device_check(L):
    import torch
    rc = _call_scatter(L, 0xD0000, 64)
    if not torch.cuda.is_available():
        assert rc in (kda.ERR_CUDA, kda.ERR_UNSUPPORTED_DEVICE)
