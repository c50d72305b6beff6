"""The roofline arithmetic of bench.py, rebuilt independently on the host.

`algorithmic_bytes` is checked against a sum over the tensors the prefill must read or
write once, each sized from its shape and dtype; `algorithmic_flops` against the sum of
the chunked form's products, step by step (Gram products, WY factors, inter-chunk read,
state update), for full 64-token chunks.  The batched workload's figures are the ones the
measured tables quote.
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench                      # noqa: E402
import kda_workloads as W         # noqa: E402

D, C = 128, 64
BF16, F32, I32 = 2, np.dtype(np.float32).itemsize, np.dtype(np.int32).itemsize


def bytes_by_tensor(w):
    T, N, H = sum(w.lengths), len(w.lengths), w.heads
    state = F32 if w.state_dtype == "f32" else BF16
    tensors = {
        "q": T * H * D * BF16, "k": T * H * D * BF16, "v": T * H * D * BF16,
        "g": T * H * D * BF16, "out": T * H * D * BF16, "beta": T * H * BF16,
        "A_log": H * F32, "dt_bias": H * D * F32, "cu_seqlens": (N + 1) * I32,
        "initial_state": N * H * D * D * state, "final_state": N * H * D * D * state,
    }
    return sum(tensors.values())


def flops_by_step(tokens, heads):
    """Multiply-adds x 2 of one 64-token chunk and head, per step of the chunked form."""
    steps = {
        "A = K K^T (decay-weighted)": 2 * C * C * D,
        "QK = Q K^T (decay-weighted)": 2 * C * C * D,
        "W = T diag(b) K": 2 * C * C * D,
        "U' = T diag(b) V": 2 * C * C * D,
        "U = U' - W S": 2 * C * D * D,
        "O = Qg S": 2 * C * D * D,
        "O += QK U": 2 * C * C * D,
        "S += Ke^T U": 2 * C * D * D,
    }
    assert tokens % C == 0
    return tokens // C * heads * sum(steps.values())


@pytest.mark.parametrize("cfg", [0, 1, 2, 4])
def test_algorithmic_bytes(cfg):
    w = W.workload(cfg)
    assert bench.algorithmic_bytes(w) == bytes_by_tensor(w)


def test_algorithmic_bytes_of_the_batched_workload():
    assert bench.algorithmic_bytes(W.workload(1)) == 352_854_116


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_algorithmic_flops(cfg):
    w = W.workload(cfg)
    assert bench.algorithmic_flops(w) == flops_by_step(sum(w.lengths), w.heads)


def test_algorithmic_flops_of_the_batched_workload():
    assert bench.algorithmic_flops(W.workload(1)) == 47_244_640_256


def test_the_batched_workload_is_bound_by_hbm():
    """flop per byte below the measured ridge point: the HBM roofline is the slower one."""
    w = W.workload(1)
    hbm_gbs, bf16_tflops, _ = bench.load_peaks()
    t_hbm = bench.algorithmic_bytes(w) / (hbm_gbs * 1e9)
    t_tensor = bench.algorithmic_flops(w) / (bf16_tflops * 1e12)
    assert t_hbm > t_tensor


def test_kernel_source_sets_name_existing_device_sources():
    """Every file a per-kernel source hash covers exists, so a renamed or removed file cannot
    leave a committed traffic figure keyed to sources that are no longer built."""
    csrc = os.path.join(ROOT, "kda_gated_delta_chunk_gb300", "csrc")
    for name, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.isfile(os.path.join(csrc, f)), (name, f)
            assert f not in bench.HOST_ONLY_SOURCES, (name, f)


def test_committed_traffic_entries_name_their_capture():
    """Each traffic figure names the profile summary it came from, and that file is committed."""
    import json
    t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for name, ent in t.items():
        assert ent["dram_bytes_per_launch"] > 0, name
        assert os.path.isfile(os.path.join(ROOT, ent["capture"])), (name, ent["capture"])
        assert len(ent["source_hash"]) == 16, name
