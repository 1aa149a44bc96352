"""Python binding of libjfa (ctypes).  Argument marshalling only.

Every function here has the name of the C entry point it calls (see
include/jfa.h).  Tensors are torch tensors; PyTorch supplies device memory
(outputs, workspace) and the current CUDA stream.  No arithmetic of the method
happens in Python: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import functools
import inspect
import math
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libjfa.so")

JFA_OP_FWD, JFA_OP_BWD, JFA_OP_BLOCK_FWD, JFA_OP_BLOCK_BWD, JFA_OP_TOPK_SELECT, JFA_OP_FWD_TOPK = 0, 1, 2, 3, 4, 5
JFA_OP_BLOCK_FWD_ROPE, JFA_OP_BLOCK_BWD_ROPE = 6, 7
STATUS = {0: "JFA_OK", 1: "JFA_ERR_INVALID_ARG", 2: "JFA_ERR_UNSUPPORTED", 3: "JFA_ERR_BAD_OFFSETS",
          4: "JFA_ERR_WORKSPACE_TOO_SMALL", 5: "JFA_ERR_ARCH", 6: "JFA_ERR_CUDA", 7: "JFA_ERR_DEVICE_TIMEOUT",
          8: "JFA_ERR_TOO_LARGE"}

# exported symbols and their ctypes signatures
_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "jfa_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _S, _P]),
    "jfa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _S, _P]),
    "jfa_fwd_window": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _S, _P]),
    "jfa_bwd_window": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _S,
                            _P]),
    "jfa_plan_window": (_I, [_I, _P, _I, _I, _I, _I, _I, _P, _P]),
    "jfa_topk_rows": (_I, [_P, _I, _I, _I, _I]),
    "jfa_topk_select": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _S, _P]),
    "jfa_fwd_topk": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "block_attn_fwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _S, _P]),
    "block_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _S, _P]),
    "block_attn_fwd_rope": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _F, _P, _S, _P]),
    "block_attn_bwd_rope": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _F, _P, _S,
                                 _P]),
    "jfa_workspace_size": (_S, [_I, _P, _I, _I, _I, _I, _I, _I]),
    "jfa_status_string": (ctypes.c_char_p, [_I]),
    "jfa_device_status": (_I, [_P, _P]),
    "jfa_plan_fwd": (_I, [_P, _I, _I, _I, _I, _I, _P, _P]),
    "jfa_plan_bwd": (_I, [_P, _I, _I, _I, _I, _I, _P, _P]),
    "block_plan": (_I, [_P, _I, _I, _I, _P, _P]),
    "jfa_fwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "jfa_fwd_noalloc_capacity": (_S, []),
    "jfa_fwd_noalloc_status": (_I, [_P]),
    "jfa_selftest_wait_timeout_noalloc": (_I, [_P]),
    "jfa_set_schedule": (_I, [_I]),
    "jfa_get_schedule": (_I, []),
    "jfa_set_bwd_schedule": (_I, [_I]),
    "jfa_get_bwd_schedule": (_I, []),
    "jfa_set_block_schedule": (_I, [_I]),
    "jfa_get_block_schedule": (_I, []),
    "jfa_profile_enable": (_I, [_I]),
    "jfa_selftest_wait_timeout": (_I, [_P, _S, _P]),
    "jfa_profile_select": (_I, [_I]),
    "jfa_profile_read": (_I, [_I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
}
KERNEL_KINDS = {"fwd": 0, "bwd_prep": 1, "bwd_main": 2, "dq_convert": 3, "block_fwd": 4, "block_bwd": 5,
                "fill": 6, "topk_select": 7, "rope": 8}

_lock = threading.Lock()
_lib = None


class JfaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


def load(path: str | None = None):
    """Load libjfa.so (built by ``variable_length_attention_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libjfa.so is not built ({p}); run variable_length_attention_gb300.build.build()")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype, f.argtypes = res, args
            _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else t.data_ptr()


def _host_offsets(offsets, offsets_host):
    if offsets_host is None:
        offsets_host = offsets.detach().to("cpu")
    h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int32))
    return h


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream():
    """Handle of the current CUDA stream of the current device (the direct
    query where this torch has it: it skips building a Stream object)."""
    if _raw_stream is not None and _cur_device is not None:
        return _raw_stream(_cur_device())
    return torch.cuda.current_stream().cuda_stream


def _check(name, st):
    if st != 0:
        raise JfaError(name, st)


def _on_tensor_device(fn):
    """Run a call under the CUDA device of its first tensor argument, as a torch
    op does: the library launches on the current device and its current
    stream, so calling with tensors of another device would otherwise launch
    kernels on the wrong GPU."""
    first_name = next(iter(inspect.signature(fn).parameters))

    @functools.wraps(fn)
    def call(*args, **kwargs):
        first = args[0] if args else kwargs.get(first_name)
        if isinstance(first, torch.Tensor) and first.is_cuda:
            with torch.cuda.device(first.device):
                return fn(*args, **kwargs)
        return fn(*args, **kwargs)  # the argument checks reject a tensor that is not on a GPU
    return call


def _expect(name, t, shape, dtype=torch.bfloat16, device=None):
    """The C ABI sees only pointers; check here that each tensor really is the
    contiguous device buffer the call will read or write, on the call's device."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, but the call runs on {device}")


def _check_problem(q, k, v, offsets, offs_h, nq, *, o=None, dout=None, lse=None, dq=None, dk=None, dv=None):
    batch = len(offs_h) - 1
    T = int(offs_h[-1]) if batch >= 0 else 0
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    q_rows = nq if nq > 0 else T
    o_rows = batch * nq if nq > 0 else T
    _expect("q", q, (q_rows, H, D))
    dev = q.device
    _expect("k", k, (T, Hkv, D), device=dev)
    _expect("v", v, (T, Hkv, D), device=dev)
    _expect("offsets", offsets, (batch + 1,), torch.int32, device=dev)
    _expect("o", o, (o_rows, H, D), device=dev)
    _expect("dout", dout, (o_rows, H, D), device=dev)
    _expect("lse", lse, (H, o_rows), torch.float32, device=dev)
    _expect("dq", dq, (q_rows, H, D), device=dev)
    _expect("dk", dk, (T, Hkv, D), device=dev)
    _expect("dv", dv, (T, Hkv, D), device=dev)


def _workspace(op, offs_h, batch, nq, H, D, causal, bq, workspace, device):
    """The caller's workspace as given (the library checks its size and returns
    JFA_ERR_WORKSPACE_TOO_SMALL), or a new one of the size the library asks for."""
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace: must be a contiguous CUDA tensor")
        if workspace.device != device:
            raise ValueError(f"workspace: on {workspace.device}, but the call runs on {device}")
        return workspace
    need = load().jfa_workspace_size(op, offs_h.ctypes.data, batch, nq, H, D, int(causal), int(bq))
    return torch.empty(max(need, 256), dtype=torch.uint8, device=device)


def jfa_workspace_size(op, offsets_host, batch, nq_broadcast, num_heads, head_dim, causal, broadcast_q):
    h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int32))
    return load().jfa_workspace_size(op, h.ctypes.data_as(ctypes.c_void_p), batch, nq_broadcast, num_heads,
                                     head_dim, int(causal), int(broadcast_q))


def jfa_status_string(status: int) -> str:
    return load().jfa_status_string(status).decode()


@_on_tensor_device
def jfa_device_status(workspace) -> int:
    return load().jfa_device_status(_ptr(workspace), _stream())


def _window_args(window):
    """(left, right) of a sliding window; None or a negative side is open (-1)."""
    left, right = window
    return (-1 if left is None or left < 0 else int(left)), (-1 if right is None or right < 0 else int(right))


@_on_tensor_device
def jfa_fwd(q, k, v, offsets, offsets_host=None, *, max_len=None, nq_broadcast=0, causal=False, scale=None,
            out=None, lse=None, return_lse=True, workspace=None, window=None):
    """Forward.  Returns (o, lse); lse is None if return_lse is False.
    ``window=(left, right)``: query i sees keys i-left .. i+right of its
    sequence (jfa_fwd_window; self-attention; causal closes the right side)."""
    L = load()
    offs_h = _host_offsets(offsets, offsets_host)
    batch = len(offs_h) - 1
    bq = nq_broadcast > 0
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    if max_len is None:
        max_len = int(np.max(np.diff(offs_h))) if batch > 0 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o_rows = batch * nq_broadcast if bq else int(offs_h[-1])
    if out is None:
        out = torch.empty((o_rows, H, D), dtype=torch.bfloat16, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty((H, o_rows), dtype=torch.float32, device=q.device)
    if not return_lse:
        lse = None
    _check_problem(q, k, v, offsets, offs_h, nq_broadcast, o=out, lse=lse)
    workspace = _workspace(JFA_OP_FWD, offs_h, batch, nq_broadcast, H, D, causal, bq, workspace, q.device)
    if window is not None:
        if bq:
            raise ValueError("a window applies to self-attention only")
        wl, wr = _window_args(window)
        if causal:
            wr = 0 if wr < 0 else min(wr, 0)
        st = L.jfa_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(offsets), offs_h.ctypes.data,
                              batch, int(max_len), H, Hkv, D, float(scale), wl, wr, workspace.data_ptr(),
                              workspace.nbytes, _stream())
        _check("jfa_fwd_window", st)
        return out, lse
    st = L.jfa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(offsets),
                   offs_h.ctypes.data, batch, int(max_len), int(nq_broadcast), H, Hkv, D,
                   float(scale), int(causal), int(bq), workspace.data_ptr(), workspace.nbytes, _stream())
    _check("jfa_fwd", st)
    return out, lse


@_on_tensor_device
def jfa_bwd(q, k, v, o, dout, lse, offsets, offsets_host=None, *, max_len=None, nq_broadcast=0, causal=False,
            scale=None, dq=None, dk=None, dv=None, workspace=None, window=None):
    """Backward.  Returns (dq, dk, dv).  ``window`` as in jfa_fwd."""
    L = load()
    offs_h = _host_offsets(offsets, offsets_host)
    batch = len(offs_h) - 1
    bq = nq_broadcast > 0
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    if max_len is None:
        max_len = int(np.max(np.diff(offs_h))) if batch > 0 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_problem(q, k, v, offsets, offs_h, nq_broadcast, o=o, dout=dout, lse=lse, dq=dq, dk=dk, dv=dv)
    workspace = _workspace(JFA_OP_BWD, offs_h, batch, nq_broadcast, H, D, causal, bq, workspace, q.device)
    if window is not None:
        if bq:
            raise ValueError("a window applies to self-attention only")
        wl, wr = _window_args(window)
        if causal:
            wr = 0 if wr < 0 else min(wr, 0)
        st = L.jfa_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                              _ptr(dv), _ptr(offsets), offs_h.ctypes.data, batch, int(max_len), H, Hkv, D,
                              float(scale), wl, wr, workspace.data_ptr(), workspace.nbytes, _stream())
        _check("jfa_bwd_window", st)
        return dq, dk, dv
    st = L.jfa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                   _ptr(offsets), offs_h.ctypes.data, batch, int(max_len), int(nq_broadcast),
                   H, Hkv, D, float(scale), int(causal), int(bq), workspace.data_ptr(), workspace.nbytes, _stream())
    _check("jfa_bwd", st)
    return dq, dk, dv


def _rope_tables(rope, D, device):
    if rope is None:
        return None
    cos, sin = rope
    for name, t in (("rope cos", cos), ("rope sin", sin)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.dim() != 2 or \
                t.shape[1] != D // 2 or t.device != device:
            raise ValueError(f"{name}: expected a contiguous float32 CUDA tensor [positions, {D // 2}] on {device}")
    if cos.shape != sin.shape:
        raise ValueError("rope cos and sin must have the same shape")
    return cos, sin


def jfa_topk_rows(offsets_host, num_heads, nq_broadcast=0) -> int:
    """Query blocks (rows of a top-k selection) of a problem."""
    h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int32))
    n = load().jfa_topk_rows(h.ctypes.data_as(ctypes.c_void_p), len(h) - 1, int(nq_broadcast), int(num_heads),
                             int(nq_broadcast > 0))
    if n < 0:
        raise JfaError("jfa_topk_rows", -n)
    return n


@_on_tensor_device
def jfa_topk_select(q, k, offsets, offsets_host=None, *, topk, max_len=None, nq_broadcast=0, selection=None,
                    workspace=None):
    """First stage of the block-sparse forward: int32 [query blocks, topk],
    each row's chosen key blocks ascending, -1 padded."""
    L = load()
    offs_h = _host_offsets(offsets, offsets_host)
    batch = len(offs_h) - 1
    bq = nq_broadcast > 0
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    if max_len is None:
        max_len = int(np.max(np.diff(offs_h))) if batch > 0 else 0
    rows = jfa_topk_rows(offs_h, H, nq_broadcast)
    if selection is None:
        selection = torch.empty((rows, topk), dtype=torch.int32, device=q.device)
    _expect("selection", selection, (rows, topk), torch.int32, device=q.device)
    _check_problem(q, k, k, offsets, offs_h, nq_broadcast)
    workspace = _workspace(JFA_OP_TOPK_SELECT, offs_h, batch, nq_broadcast, H, D, False, bq, workspace, q.device)
    st = L.jfa_topk_select(_ptr(q), _ptr(k), _ptr(offsets), offs_h.ctypes.data, batch, int(max_len),
                           int(nq_broadcast), H, Hkv, D, int(topk), int(bq), _ptr(selection), workspace.data_ptr(),
                           workspace.nbytes, _stream())
    _check("jfa_topk_select", st)
    return selection


@_on_tensor_device
def jfa_fwd_topk(q, k, v, offsets, selection, offsets_host=None, *, topk, max_len=None, nq_broadcast=0, scale=None,
                 out=None, lse=None, workspace=None):
    """Second stage of the block-sparse forward: attention over each query
    block's chosen key blocks.  Returns (o, lse)."""
    L = load()
    offs_h = _host_offsets(offsets, offsets_host)
    batch = len(offs_h) - 1
    bq = nq_broadcast > 0
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    if max_len is None:
        max_len = int(np.max(np.diff(offs_h))) if batch > 0 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o_rows = batch * nq_broadcast if bq else int(offs_h[-1])
    if out is None:
        out = torch.empty((o_rows, H, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((H, o_rows), dtype=torch.float32, device=q.device)
    _expect("selection", selection, (jfa_topk_rows(offs_h, H, nq_broadcast), topk), torch.int32, device=q.device)
    _check_problem(q, k, v, offsets, offs_h, nq_broadcast, o=out, lse=lse)
    workspace = _workspace(JFA_OP_FWD_TOPK, offs_h, batch, nq_broadcast, H, D, False, bq, workspace, q.device)
    st = L.jfa_fwd_topk(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(selection), int(topk), _ptr(offsets),
                        offs_h.ctypes.data, batch, int(max_len), int(nq_broadcast), H, Hkv, D, float(scale), int(bq),
                        workspace.data_ptr(), workspace.nbytes, _stream())
    _check("jfa_fwd_topk", st)
    return out, lse


@_on_tensor_device
def block_attn_fwd(q, k, v, offsets, offsets_host=None, *, max_len=None, scale=None, out=None, workspace=None,
                   rope=None):
    """Block-diagonal (64-token blocks) forward.  Returns o.  ``rope=(cos, sin)``
    (fp32 [positions, D/2]) fuses the rotary embedding of q and k
    (block_attn_fwd_rope)."""
    L = load()
    offs_h = _host_offsets(offsets, offsets_host)
    batch = len(offs_h) - 1
    H, D = q.shape[1], q.shape[2]
    if max_len is None:
        max_len = int(np.max(np.diff(offs_h))) if batch > 0 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = torch.empty_like(q) if out is None else out
    _check_problem(q, k, v, offsets, offs_h, 0, o=out)
    tables = _rope_tables(rope, D, q.device)
    op = JFA_OP_BLOCK_FWD if tables is None else JFA_OP_BLOCK_FWD_ROPE
    workspace = _workspace(op, offs_h, batch, 0, H, D, False, False, workspace, q.device)
    if tables is not None:
        st = L.block_attn_fwd_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(tables[0]), _ptr(tables[1]),
                                   tables[0].shape[0], _ptr(offsets), offs_h.ctypes.data, batch, int(max_len), H, D,
                                   float(scale), workspace.data_ptr(), workspace.nbytes, _stream())
        _check("block_attn_fwd_rope", st)
        return out
    st = L.block_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(offsets), offs_h.ctypes.data,
                          batch, int(max_len), H, D, float(scale), workspace.data_ptr(), workspace.nbytes, _stream())
    _check("block_attn_fwd", st)
    return out


@_on_tensor_device
def block_attn_bwd(q, k, v, o, dout, offsets, offsets_host=None, *, max_len=None, scale=None, dq=None, dk=None,
                   dv=None, workspace=None, rope=None):
    """Block-diagonal backward.  Returns (dq, dk, dv); with ``rope`` (as in
    block_attn_fwd) dq and dk are with respect to the unrotated q and k."""
    L = load()
    offs_h = _host_offsets(offsets, offsets_host)
    batch = len(offs_h) - 1
    H, D = q.shape[1], q.shape[2]
    if max_len is None:
        max_len = int(np.max(np.diff(offs_h))) if batch > 0 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_problem(q, k, v, offsets, offs_h, 0, o=o, dout=dout, dq=dq, dk=dk, dv=dv)
    tables = _rope_tables(rope, D, q.device)
    op = JFA_OP_BLOCK_BWD if tables is None else JFA_OP_BLOCK_BWD_ROPE
    workspace = _workspace(op, offs_h, batch, 0, H, D, False, False, workspace, q.device)
    if tables is not None:
        st = L.block_attn_bwd_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                   _ptr(tables[0]), _ptr(tables[1]), tables[0].shape[0], _ptr(offsets),
                                   offs_h.ctypes.data, batch, int(max_len), H, D, float(scale),
                                   workspace.data_ptr(), workspace.nbytes, _stream())
        _check("block_attn_bwd_rope", st)
        return dq, dk, dv
    st = L.block_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                          _ptr(offsets), offs_h.ctypes.data, batch, int(max_len), H, D,
                          float(scale), workspace.data_ptr(), workspace.nbytes, _stream())
    _check("block_attn_bwd", st)
    return dq, dk, dv


def _plan(fn_name, offsets_host, num_heads, nq, causal, n_cta):
    L = load()
    h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int32))
    fn = getattr(L, fn_name)
    n = fn(h.ctypes.data_as(ctypes.c_void_p), len(h) - 1, num_heads, nq, int(causal), n_cta, None, None)
    if n < 0:
        raise JfaError(fn_name, -n)
    units = np.zeros(4 * n, dtype=np.int32)
    start = np.zeros(n_cta + 1, dtype=np.int32)
    n2 = fn(h.ctypes.data_as(ctypes.c_void_p), len(h) - 1, num_heads, nq, int(causal), n_cta,
            units.ctypes.data_as(ctypes.c_void_p), start.ctypes.data_as(ctypes.c_void_p))
    assert n2 == n
    return units, start


def jfa_plan_fwd(offsets_host, num_heads, n_cta, *, nq=0, causal=False):
    """Host forward plan: (units int32[4n], cta_start int32[n_cta+1])."""
    return _plan("jfa_plan_fwd", offsets_host, num_heads, nq, causal, n_cta)


def jfa_plan_bwd(offsets_host, num_heads, n_cta, *, nq=0, causal=False):
    """Host backward plan: (units int32[4n], cta_start int32[n_cta+1])."""
    return _plan("jfa_plan_bwd", offsets_host, num_heads, nq, causal, n_cta)


def jfa_plan_window(which, offsets_host, num_heads, n_cta, window):
    """Window planners (0 forward, 1 backward): (units int32[4n], cta_start
    int32[n_cta+1])."""
    L = load()
    h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int32))
    wl, wr = _window_args(window)
    n = L.jfa_plan_window(which, h.ctypes.data_as(ctypes.c_void_p), len(h) - 1, num_heads, wl, wr, n_cta, None,
                          None)
    if n < 0:
        raise JfaError("jfa_plan_window", -n)
    units = np.zeros(4 * n, dtype=np.int32)
    start = np.zeros(n_cta + 1, dtype=np.int32)
    L.jfa_plan_window(which, h.ctypes.data_as(ctypes.c_void_p), len(h) - 1, num_heads, wl, wr, n_cta,
                      units.ctypes.data_as(ctypes.c_void_p), start.ctypes.data_as(ctypes.c_void_p))
    return units, start


def block_plan(offsets_host, num_heads, n_sm):
    """Block plan: (block_per_batch int32[B+1], prog_start int32[P+1])."""
    L = load()
    h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int32))
    P = L.block_plan(h.ctypes.data_as(ctypes.c_void_p), len(h) - 1, num_heads, n_sm, None, None)
    if P < 0:
        raise JfaError("block_plan", -P)
    bpb = np.zeros(len(h), dtype=np.int32)
    ps = np.zeros(P + 1, dtype=np.int32)
    L.block_plan(h.ctypes.data_as(ctypes.c_void_p), len(h) - 1, num_heads, n_sm,
                 bpb.ctypes.data_as(ctypes.c_void_p), ps.ctypes.data_as(ctypes.c_void_p))
    return bpb, ps


def jfa_set_schedule(mode):
    """Work distribution of the jagged forward: 0 / "static" (host plan, one CTA
    per SM) or 1 / "clc" (Cluster Launch Control)."""
    m = {"static": 0, "clc": 1}.get(mode, mode)
    _check("jfa_set_schedule", load().jfa_set_schedule(int(m)))


def jfa_get_schedule() -> int:
    return load().jfa_get_schedule()


def jfa_set_bwd_schedule(mode):
    """Work distribution of the jagged backward: 0 / "static" (host plan, one
    CTA per SM) or 1 / "clc" (Cluster Launch Control)."""
    m = {"static": 0, "clc": 1}.get(mode, mode)
    _check("jfa_set_bwd_schedule", load().jfa_set_bwd_schedule(int(m)))


def jfa_get_bwd_schedule() -> int:
    return load().jfa_get_bwd_schedule()


def jfa_set_block_schedule(mode):
    """Work distribution of the block-diagonal kernels: 0 / "static" (closed-form
    ranges, one CTA per SM) or 1 / "clc" (Cluster Launch Control over chunks)."""
    m = {"static": 0, "clc": 1}.get(mode, mode)
    _check("jfa_set_block_schedule", load().jfa_set_block_schedule(int(m)))


def jfa_get_block_schedule() -> int:
    return load().jfa_get_block_schedule()


@_on_tensor_device
def jfa_selftest_wait_timeout(workspace) -> None:
    """Launch the bounded-wait self-test into ``workspace`` (a CUDA uint8 tensor);
    jfa_device_status(workspace) then reports JFA_ERR_DEVICE_TIMEOUT."""
    if not workspace.is_cuda:
        raise ValueError("workspace: must be a CUDA tensor")
    _check("jfa_selftest_wait_timeout",
           load().jfa_selftest_wait_timeout(workspace.data_ptr(), workspace.nbytes, _stream()))


def jfa_profile_enable(on: bool = True):
    """Start (or stop) bracketing every library kernel launch with CUDA events."""
    _check("jfa_profile_enable", load().jfa_profile_enable(int(on)))


def jfa_profile_select(kinds=None):
    """Limit the events to these kernel kinds (names or numbers; None = all)."""
    if kinds is None:
        mask = (1 << len(KERNEL_KINDS)) - 1
    else:
        mask = 0
        for k in kinds:
            mask |= 1 << (KERNEL_KINDS[k] if isinstance(k, str) else int(k))
    _check("jfa_profile_select", load().jfa_profile_select(mask))


def jfa_profile_read(kind) -> tuple[float, int]:
    """(summed device milliseconds, launches) of one kernel kind since enabling."""
    k = KERNEL_KINDS[kind] if isinstance(kind, str) else int(kind)
    ms, n = ctypes.c_double(0.0), ctypes.c_int(0)
    _check("jfa_profile_read", load().jfa_profile_read(k, ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


@_on_tensor_device
def jfa_fwd_noalloc(q, k, v, offsets, offsets_host=None, *, max_len=None, nq_broadcast=0, causal=False,
                    scale=None, out=None, lse=None):
    """jfa_fwd without a workspace, for callers that cannot allocate device
    memory: the library's own fixed 1 MiB static scratch holds the plan.  Outputs
    must still be supplied by the caller (or are allocated here by torch, for
    convenience).  Calls that overlap on the GPU race on the shared scratch."""
    L = load()
    offs_h = _host_offsets(offsets, offsets_host)
    batch = len(offs_h) - 1
    bq = nq_broadcast > 0
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    if max_len is None:
        max_len = int(np.max(np.diff(offs_h))) if batch > 0 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o_rows = batch * nq_broadcast if bq else int(offs_h[-1])
    if out is None:
        out = torch.empty((o_rows, H, D), dtype=torch.bfloat16, device=q.device)
    _check_problem(q, k, v, offsets, offs_h, nq_broadcast, o=out, lse=lse)
    st = L.jfa_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(offsets),
                           offs_h.ctypes.data, batch, int(max_len), int(nq_broadcast), H, Hkv,
                           D, float(scale), int(causal), int(bq), _stream())
    _check("jfa_fwd_noalloc", st)
    return out, lse


def jfa_fwd_noalloc_status() -> int:
    """Status recorded in jfa_fwd_noalloc's static scratch on the current device
    (synchronises the current stream): 0 or a JFA_ERR_* code."""
    return load().jfa_fwd_noalloc_status(_stream())


def jfa_selftest_wait_timeout_noalloc() -> None:
    """The bounded-wait self-test with its error word in jfa_fwd_noalloc's static
    scratch; jfa_fwd_noalloc_status() then reports JFA_ERR_DEVICE_TIMEOUT."""
    _check("jfa_selftest_wait_timeout_noalloc", load().jfa_selftest_wait_timeout_noalloc(_stream()))
