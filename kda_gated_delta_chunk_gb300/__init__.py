"""Python binding of libkda.so (chunked KDA prefill on GB300 / sm_103a).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  The
names follow the C ABI in ``include/kda.h``:

    workspace_size(total_tokens, heads, max_seqs) -> int
    chunk_prefill_fwd(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                      initial_state, cu_seqlens, out=None, final_state=None,
                      workspace=None, ...) -> (out, final_state)
    choose_vsplit(num_seqs, heads, sm_count) -> int
    chunk_prefill_fwd(..., vsplit=-1, kernel=KERNEL_AUTO): strided views of q, k, v, g,
        beta are passed through kda_chunk_prefill_fwd_strided
    recurrent_fwd(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                  cu_seqlens, token_states=False, ...) -> (out, final_state, token_states)
    plan(total_tokens, num_seqs, heads, workspace_bytes, vsplit, kernel)
        -> (kernel, vsplit, launches)
    KERNEL_AUTO / KERNEL_TC / KERNEL_TC_HELPERS / KERNEL_SPLIT / KERNEL_SPLIT_STREAMED /
    KERNEL_REF / KERNEL_PIPE
    last_device_status(workspace) -> int
    status_string(code) -> str

There is no CPU fallback: if the library is missing or the device is not an
sm_103 GPU, these calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

HEAD_DIM = 128
STATE_F32, STATE_BF16 = 0, 1
KERNEL_AUTO, KERNEL_TC, KERNEL_REF, KERNEL_SPLIT, KERNEL_TC_HELPERS, KERNEL_PIPE = 0, 1, 2, 3, 4, 5
KERNEL_SPLIT_STREAMED = 6
OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED_DEVICE = -2
ERR_WORKSPACE_TOO_SMALL = -3
ERR_UNSAFE_LOWER_BOUND = -4
ERR_MISALIGNED = -5
ERR_LAUNCH_FAILED = -6
ERR_DEVICE_TIMEOUT = -7
ERR_BAD_CU_SEQLENS = -8
ERR_CUDA = -9
ERR_BAD_OUT_INDEX = -10

# every symbol include/kda.h declares
EXPORTS = ("kda_workspace_size", "kda_chunk_prefill_fwd", "kda_chunk_prefill_fwd_ex",
           "kda_choose_vsplit", "kda_status_string", "kda_last_device_status",
           "kda_device_check", "kda_plan", "kda_plan_for", "kda_chunk_prefill_fwd_strided",
           "kda_recurrent_fwd", "kda_chunk_prefill_fwd_noalloc", "kda_chunk_prefill_fwd_scatter",
           "kda_recurrent_fwd_scatter", "kda_skinny_proj_workspace_size", "kda_skinny_proj",
           "kda_test_drop_one_record")

_lib = None
_lock = threading.Lock()


class KDAError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = int(code)
        super().__init__(f"{what}: {status_string(code)} ({code})" if what else
                         f"{status_string(code)} ({code})")


_lib_path = LIB_PATH


def use_library(path: str) -> None:
    """Load ``path`` instead of libkda.so (the phase-stamp build, for profiling); must come
    before the first call into the library."""
    global _lib_path
    with _lock:
        if _lib is not None and path != _lib_path:
            raise RuntimeError("the library is already loaded")
        _lib_path = path


def lib() -> ctypes.CDLL:
    """Load libkda.so (built in-tree by ``build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_lib_path):
                raise RuntimeError(f"{_lib_path} is missing: build it with "
                                   "kda_gated_delta_chunk_gb300.build.build()")
            L = ctypes.CDLL(_lib_path)
            P, I32, I64, SZ, F = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_size_t, ctypes.c_float)
            L.kda_workspace_size.restype = SZ
            L.kda_workspace_size.argtypes = [I64, I32, I32]
            fwd_args = [P, P, P, P, P, P, P, F, F, P, P, P, P, ctypes.c_int, P, P,
                        I64, I32, I32, SZ]
            L.kda_chunk_prefill_fwd.restype = ctypes.c_int
            L.kda_chunk_prefill_fwd.argtypes = fwd_args
            L.kda_chunk_prefill_fwd_ex.restype = ctypes.c_int
            L.kda_chunk_prefill_fwd_ex.argtypes = fwd_args + [ctypes.c_int, ctypes.c_int]
            L.kda_chunk_prefill_fwd_strided.restype = ctypes.c_int
            L.kda_chunk_prefill_fwd_strided.argtypes = fwd_args + [I64] * 5 + [ctypes.c_int,
                                                                             ctypes.c_int]
            L.kda_chunk_prefill_fwd_scatter.restype = ctypes.c_int
            L.kda_chunk_prefill_fwd_scatter.argtypes = fwd_args + [I64] * 5 + [P, I64,
                                                                             ctypes.c_int,
                                                                             ctypes.c_int]
            L.kda_choose_vsplit.restype = ctypes.c_int
            L.kda_choose_vsplit.argtypes = [I32, I32, I32]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_status_string.argtypes = [ctypes.c_int]
            L.kda_last_device_status.restype = ctypes.c_int
            L.kda_last_device_status.argtypes = [P, P]
            L.kda_device_check.restype = ctypes.c_int
            L.kda_device_check.argtypes = [ctypes.c_int]
            L.kda_recurrent_fwd.restype = ctypes.c_int
            L.kda_recurrent_fwd.argtypes = [P, P, P, P, P, P, P, F, F, P, P, P, P, ctypes.c_int,
                                            P, P, P, I64, I32, I32, SZ]
            L.kda_recurrent_fwd_scatter.restype = ctypes.c_int
            L.kda_recurrent_fwd_scatter.argtypes = L.kda_recurrent_fwd.argtypes + [P, I64]
            L.kda_plan.restype = ctypes.c_int
            L.kda_plan.argtypes = [I64, I32, I32, SZ, ctypes.c_int, ctypes.c_int, P, P, P]
            L.kda_plan_for.restype = ctypes.c_int
            L.kda_plan_for.argtypes = [I64, I32, I32, SZ, ctypes.c_int, ctypes.c_int, I32, P, P, P]
            L.kda_skinny_proj_workspace_size.restype = SZ
            L.kda_skinny_proj_workspace_size.argtypes = [I32, I32]
            L.kda_skinny_proj.restype = ctypes.c_int
            L.kda_skinny_proj.argtypes = [P, I64, P, P, P, I64, P, I64, I32, I32, I32, I32, I32,
                                          P, SZ, P]
            L.kda_test_drop_one_record.restype = None
            L.kda_test_drop_one_record.argtypes = [ctypes.c_int]
            L.kda_chunk_prefill_fwd_noalloc.restype = ctypes.c_int
            L.kda_chunk_prefill_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, F, F, P, P, P, P,
                                                        ctypes.c_int, P, I64, I32, I32]
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().kda_status_string(int(code)).decode()


def workspace_size(total_tokens: int, heads: int, max_seqs: int) -> int:
    return int(lib().kda_workspace_size(int(total_tokens), int(heads), int(max_seqs)))


def choose_vsplit(num_seqs: int, heads: int, sm_count: int) -> int:
    return int(lib().kda_choose_vsplit(int(num_seqs), int(heads), int(sm_count)))


def device_check(device: int = 0) -> int:
    return int(lib().kda_device_check(int(device)))


def test_drop_one_record(on: bool) -> None:
    """Test hook (failure detection): while on, helper-path calls leave one record
    unpublished so the waiting CTA's bounded wait runs out."""
    lib().kda_test_drop_one_record(1 if on else 0)


def plan(total_tokens: int, num_seqs: int, heads: int, workspace_bytes: int,
         vsplit: int = -1, kernel: int = KERNEL_AUTO):
    """``kda_plan``: (kernel, vsplit, launches) a call would use on the current device."""
    k, p, n = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().kda_plan(int(total_tokens), int(num_seqs), int(heads), int(workspace_bytes),
                        int(vsplit), int(kernel), ctypes.byref(k), ctypes.byref(p),
                        ctypes.byref(n))
    if rc != OK:
        raise KDAError(rc, "kda_plan")
    return k.value, p.value, n.value


def plan_for(total_tokens: int, num_seqs: int, heads: int, workspace_bytes: int, sm_count: int,
             vsplit: int = -1, kernel: int = KERNEL_AUTO):
    """``kda_plan_for``: (kernel, vsplit, launches) a call would use on a device with
    ``sm_count`` multiprocessors; touches no device."""
    k, p, n = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().kda_plan_for(int(total_tokens), int(num_seqs), int(heads), int(workspace_bytes),
                            int(vsplit), int(kernel), int(sm_count), ctypes.byref(k),
                            ctypes.byref(p), ctypes.byref(n))
    if rc != OK:
        raise KDAError(rc, "kda_plan_for")
    return k.value, p.value, n.value


def alloc_workspace(total_tokens: int, heads: int, max_seqs: int, device=None) -> torch.Tensor:
    """A zero-filled uint8 workspace of ``workspace_size`` bytes (16-byte aligned)."""
    n = workspace_size(total_tokens, heads, max_seqs)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def last_device_status(workspace: torch.Tensor, stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    return int(lib().kda_last_device_status(ctypes.c_void_p(workspace.data_ptr()),
                                            ctypes.c_void_p(s.cuda_stream)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, shape=None, token_strided=False):
    """Type/device/shape checks.  With token_strided, only the leading (token) dimension may
    be strided: the rest must be dense (views into a wider buffer, e.g. a fused projection)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and t.shape != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.is_contiguous():
        return
    if token_strided:
        inner = 1
        for size, stride in zip(reversed(t.shape[1:]), reversed(t.stride()[1:])):
            if size > 1 and stride != inner:
                raise ValueError(f"{name}: only the token dimension may be strided")
            inner *= size
    else:
        raise ValueError(f"{name} must be contiguous")


def _out_rows(out, out_index, T, H, D, dev):
    """The destination of the outputs: dense [T, H, D] (allocated if None), or with a row
    map, ``out`` [R, H, D] given by the caller and out_index int32 [T]."""
    if out_index is None:
        if out is None:
            out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
        _need(out, "out", torch.bfloat16, (T, H, D))
        return out, 0
    if out is None:
        raise ValueError("out_index needs the destination tensor out")
    _need(out_index, "out_index", torch.int32, (T,))
    _need(out, "out", torch.bfloat16, (out.shape[0], H, D))
    return out, int(out.shape[0])


def chunk_prefill_fwd(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                      initial_state, cu_seqlens, out=None, final_state=None,
                      workspace=None, state_dtype=None, stream=None, vsplit: int = -1,
                      kernel: int = KERNEL_AUTO, out_index=None):
    """Run ``kda_chunk_prefill_fwd`` (``_ex`` when vsplit/kernel are overridden,
    ``_strided`` for views, ``_scatter`` with a row map).

    q, k, v, g: bf16 [T, H, 128] (a leading batch dim of 1 is accepted);
    beta: bf16 [T, H]; A_log: fp32 [H]; dt_bias: fp32 [H, 128];
    initial_state: [N, H, 128, 128] fp32/bf16 or None; cu_seqlens: int32 [N+1].
    out_index: None, or int32 [T] -- token t's output goes to out[out_index[t]], out being
    a caller's [R, H, 128] buffer.  Returns (out, final_state).  Asynchronous on ``stream``
    (default: the current torch stream).
    """
    squeeze = q.dim() == 4
    if squeeze:
        q, k, v, g = (x.view(x.shape[1:]) for x in (q, k, v, g))
        if out is not None:
            out = out.view(out.shape[1:])
        if beta.dim() == 3:
            beta = beta.view(beta.shape[1:])
        if out_index is not None and out_index.dim() == 2:
            out_index = out_index.view(out_index.shape[1:])
    T, H, D = q.shape
    if D != HEAD_DIM:
        raise KDAError(ERR_INVALID_ARG, f"head_dim {D} (only {HEAD_DIM} is supported)")
    N = cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g)):
        _need(t, name, torch.bfloat16, (T, H, D), token_strided=True)
    _need(beta, "beta", torch.bfloat16, (T, H), token_strided=True)
    _need(A_log, "A_log", torch.float32, (H,))
    _need(dt_bias, "dt_bias", torch.float32, (H, D))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,))
    tok_strides = [int(t.stride(0)) if T > 1 else H * D for t in (q, k, v, g)]
    tok_strides.append(int(beta.stride(0)) if T > 1 else H)
    dense = tok_strides == [H * D] * 4 + [H]
    if state_dtype is None:
        state_dtype = initial_state.dtype if initial_state is not None else torch.float32
    sd = {torch.float32: STATE_F32, torch.bfloat16: STATE_BF16}.get(state_dtype)
    if sd is None:
        raise TypeError("state dtype must be float32 or bfloat16")
    if initial_state is not None:
        _need(initial_state, "initial_state", state_dtype, (N, H, D, D))
    out, out_rows = _out_rows(out, out_index, T, H, D, q.device)
    if final_state is None:
        final_state = torch.empty((N, H, D, D), dtype=state_dtype, device=q.device)
    _need(final_state, "final_state", state_dtype, (N, H, D, D))
    if workspace is None:
        workspace = alloc_workspace(T, H, N, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
            float(lower_bound), float(scale), _ptr(initial_state), _ptr(cu_seqlens),
            _ptr(out), _ptr(final_state), sd, _ptr(workspace), ctypes.c_void_p(s.cuda_stream),
            int(T), int(N), int(H), int(workspace.numel()))
    if out_index is not None:
        rc = lib().kda_chunk_prefill_fwd_scatter(*args, *tok_strides, _ptr(out_index), out_rows,
                                                 int(vsplit), int(kernel))
    elif not dense:
        rc = lib().kda_chunk_prefill_fwd_strided(*args, *tok_strides, int(vsplit), int(kernel))
    elif vsplit == -1 and kernel == KERNEL_AUTO:
        rc = lib().kda_chunk_prefill_fwd(*args)
    else:
        rc = lib().kda_chunk_prefill_fwd_ex(*args, int(vsplit), int(kernel))
    if rc != OK:
        raise KDAError(rc, "kda_chunk_prefill_fwd")
    if squeeze:
        out = out.unsqueeze(0)
    return out, final_state


def recurrent_fwd(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                  cu_seqlens, out=None, final_state=None, token_states=False, workspace=None,
                  state_dtype=None, stream=None, out_index=None):
    """Run ``kda_recurrent_fwd`` (decode / speculative verify: a few tokens per sequence;
    ``_scatter`` with a row map).

    Same tensors as chunk_prefill_fwd (dense).  token_states: False (none), True (allocate
    [T, H, 128, 128] in the state dtype) or a tensor to fill with the state after every
    token.  out_index as in chunk_prefill_fwd.  Returns (out, final_state, token_states or
    None).
    """
    if q.dim() == 4:
        q, k, v, g = (x.view(x.shape[1:]) for x in (q, k, v, g))
        if beta.dim() == 3:
            beta = beta.view(beta.shape[1:])
    T, H, D = q.shape
    N = cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g)):
        _need(t, name, torch.bfloat16, (T, H, D))
    _need(beta, "beta", torch.bfloat16, (T, H))
    _need(A_log, "A_log", torch.float32, (H,))
    _need(dt_bias, "dt_bias", torch.float32, (H, D))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,))
    if state_dtype is None:
        state_dtype = initial_state.dtype if initial_state is not None else torch.float32
    sd = {torch.float32: STATE_F32, torch.bfloat16: STATE_BF16}.get(state_dtype)
    if sd is None:
        raise TypeError("state dtype must be float32 or bfloat16")
    if initial_state is not None:
        _need(initial_state, "initial_state", state_dtype, (N, H, D, D))
    out, out_rows = _out_rows(out, out_index, T, H, D, q.device)
    if final_state is None:
        final_state = torch.empty((N, H, D, D), dtype=state_dtype, device=q.device)
    _need(final_state, "final_state", state_dtype, (N, H, D, D))
    if token_states is True:
        token_states = torch.empty((T, H, D, D), dtype=state_dtype, device=q.device)
    elif token_states is False:
        token_states = None
    if token_states is not None:
        _need(token_states, "token_states", state_dtype, (T, H, D, D))
    if workspace is None:
        workspace = torch.zeros(256, dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
            float(lower_bound), float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
            _ptr(final_state), sd, _ptr(token_states), _ptr(workspace),
            ctypes.c_void_p(s.cuda_stream), int(T), int(N), int(H), int(workspace.numel()))
    if out_index is not None:
        rc = lib().kda_recurrent_fwd_scatter(*args, _ptr(out_index), out_rows)
    else:
        rc = lib().kda_recurrent_fwd(*args)
    if rc != OK:
        raise KDAError(rc, "kda_recurrent_fwd")
    return out, final_state, token_states


def skinny_proj_workspace_size(k: int, n_ab: int) -> int:
    return int(lib().kda_skinny_proj_workspace_size(int(k), int(n_ab)))


def skinny_proj(x, w_ab, w_b, r: int = 128, y=None, z=None, workspace=None, stream=None):
    """Run ``kda_skinny_proj``: y = x w_ab^T, z = y[:, :r] w_b^T (bf16, fp32 accumulation).

    x: bf16 [m, k] (rows may be strided), w_ab: bf16 [n_ab, k], w_b: bf16 [n_b, r];
    y / z: optional bf16 [m, n_ab] / [m, n_b] outputs (rows may be strided, e.g. views into
    the buffers the next kernels read).  workspace: a zero-filled uint8 buffer of
    ``skinny_proj_workspace_size(k, n_ab)`` bytes, reusable across calls on one stream.
    Returns (y, z).
    """
    if x.dim() != 2 or w_ab.dim() != 2 or w_b.dim() != 2:
        raise ValueError("x, w_ab and w_b must be 2-D")
    m, k = x.shape
    n_ab, n_b = w_ab.shape[0], w_b.shape[0]
    _need(x, "x", torch.bfloat16, (m, k), token_strided=True)
    _need(w_ab, "w_ab", torch.bfloat16, (n_ab, k))
    _need(w_b, "w_b", torch.bfloat16, (n_b, int(r)))
    if y is None:
        y = torch.empty((m, n_ab), dtype=torch.bfloat16, device=x.device)
    if z is None:
        z = torch.empty((m, n_b), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, (m, n_ab), token_strided=True)
    _need(z, "z", torch.bfloat16, (m, n_b), token_strided=True)
    if workspace is None:
        workspace = torch.zeros(skinny_proj_workspace_size(k, n_ab), dtype=torch.uint8,
                                device=x.device)
    _need(workspace, "workspace", torch.uint8)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    ld = lambda t, n: int(t.stride(0)) if t.shape[0] > 1 else n
    rc = lib().kda_skinny_proj(_ptr(x), ld(x, k), _ptr(w_ab), _ptr(w_b), _ptr(y), ld(y, n_ab),
                               _ptr(z), ld(z, n_b), int(m), int(k), int(n_ab), int(r), int(n_b),
                               _ptr(workspace), int(workspace.numel()),
                               ctypes.c_void_p(s.cuda_stream))
    if rc != OK:
        raise KDAError(rc, "kda_skinny_proj")
    return y, z


def chunk_prefill_fwd_noalloc(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                              initial_state, cu_seqlens, out, final_state, stream=None):
    """Run ``kda_chunk_prefill_fwd_noalloc``: no workspace, no allocation.

    For callers that cannot allocate device memory.  ``out`` and
    ``final_state`` must be given (this wrapper allocates nothing either);
    the library keeps its small scratch in a static device array shared by
    all calls, so calls that overlap on the GPU race.
    """
    if q.dim() == 4:
        q, k, v, g = (x.view(x.shape[1:]) for x in (q, k, v, g))
        out = out.view(out.shape[1:])
        if beta.dim() == 3:
            beta = beta.view(beta.shape[1:])
    T, H, D = q.shape
    N = cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("out", out)):
        _need(t, name, torch.bfloat16, (T, H, D))
    _need(beta, "beta", torch.bfloat16, (T, H))
    _need(A_log, "A_log", torch.float32, (H,))
    _need(dt_bias, "dt_bias", torch.float32, (H, D))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,))
    sd = {torch.float32: STATE_F32, torch.bfloat16: STATE_BF16}.get(final_state.dtype)
    if sd is None:
        raise TypeError("state dtype must be float32 or bfloat16")
    _need(final_state, "final_state", final_state.dtype, (N, H, D, D))
    if initial_state is not None:
        _need(initial_state, "initial_state", final_state.dtype, (N, H, D, D))
    # the library finds its static scratch on the current device: every tensor must live there
    cur = torch.cuda.current_device()
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("A_log", A_log),
                    ("dt_bias", dt_bias), ("cu_seqlens", cu_seqlens), ("out", out),
                    ("final_state", final_state), ("initial_state", initial_state)):
        if t is not None and t.device.index != cur:
            raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{cur}")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    rc = lib().kda_chunk_prefill_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
        float(lower_bound), float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
        _ptr(final_state), sd, ctypes.c_void_p(s.cuda_stream), int(T), int(N), int(H))
    if rc != OK:
        raise KDAError(rc, "kda_chunk_prefill_fwd_noalloc")
    return out, final_state
