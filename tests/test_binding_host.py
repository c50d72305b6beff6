"""The Python binding on a host without a GPU: it marshals arguments and nothing else.

There is no CPU fallback: host tensors are refused before anything is computed, and a
missing libkda.so is an error, not a slower path.  Importing the package loads no oracle
code.
"""
import os
import subprocess
import sys

import pytest
import torch

import kda_gated_delta_chunk_gb300 as kda
import kda_workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _host_inputs():
    inp = W.make_inputs(W.custom([70, 30], 2, seed=1))
    assert inp["q"].device.type == "cpu"
    return (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"], inp["dt_bias"],
            inp["lower_bound"], inp["scale"], inp["initial_state"], inp["cu_seqlens"])


def test_prefill_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA tensor"):
        kda.chunk_prefill_fwd(*_host_inputs())


def test_recurrent_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA tensor"):
        kda.recurrent_fwd(*_host_inputs())


def test_skinny_proj_refuses_host_tensors():
    x = torch.zeros(14, 256, dtype=torch.bfloat16)
    w_ab = torch.zeros(144, 256, dtype=torch.bfloat16)
    w_b = torch.zeros(512, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        kda.skinny_proj(x, w_ab, w_b)


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(kda, "_lib_path", str(tmp_path / "libkda.so"))
    monkeypatch.setattr(kda, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        kda.workspace_size(128, 2, 1)


def test_package_imports_no_oracle_code():
    code = ("import sys, kda_gated_delta_chunk_gb300\n"
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]\n"
            "sys.exit(1 if bad else 0)\n")
    assert subprocess.run([sys.executable, "-c", code], cwd=ROOT).returncode == 0
