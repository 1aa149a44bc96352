"""The C ABI: the library loads on a machine without a GPU, exports every entry
point include/jfa.h declares, and rejects bad arguments before any device work."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import jfa as J

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "jfa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol():
    lib = J.load()
    names = _declared()
    assert "jfa_fwd" in names and "jfa_bwd" in names and "block_attn_fwd" in names and "block_attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    # and the binding knows every one of them
    assert set(names) <= set(J.SIGNATURES), set(names) - set(J.SIGNATURES)


def test_status_strings():
    for code in range(8):
        s = V.jfa_status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert V.jfa_status_string(99) == "unknown status"


FAKE = ctypes.c_void_p(0x10000)        # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x10008)


def _fwd(offsets, *, q=FAKE, D=128, H=2, Hkv=2, causal=0, bq=0, nq=0, scale=0.1, max_len=None, batch=None):
    lib = J.load()
    h = np.ascontiguousarray(np.asarray(offsets, dtype=np.int32))
    if max_len is None:
        max_len = int(np.max(np.diff(h))) if len(h) > 1 else 0
    if batch is None:
        batch = len(h) - 1
    return lib.jfa_fwd(q, FAKE, FAKE, FAKE, None, FAKE, h.ctypes.data_as(ctypes.c_void_p), batch, max_len, nq, H,
                       Hkv, D, scale, causal, bq, FAKE, 1 << 20, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(D=96), 2),                          # head_dim not 64/128
    (dict(H=3, Hkv=2), 2),                    # heads not a multiple of kv heads
    (dict(causal=1, bq=1, nq=8), 2),          # causal broadcast is undefined
    (dict(bq=1, nq=0), 1),                    # broadcast without query rows
    (dict(scale=0.0), 1),                     # scale must be positive
    (dict(scale=float("nan")), 1),
    (dict(q=MISALIGNED), 1),                  # TMA needs 16-byte aligned bases
    (dict(max_len=10), 3),                    # a sequence longer than max_len
    (dict(batch=-1), 1),
])
def test_fwd_argument_errors(kwargs, status):
    assert _fwd([0, 17, 40], **kwargs) == status


@pytest.mark.parametrize("left,right", [(-2, 0), (0, -2), (-5, -5)])
@pytest.mark.parametrize("bwd", [False, True])
def test_window_bounds_below_minus_one_rejected(left, right, bwd):
    # -1 leaves a side open; anything lower is an argument error, found before
    # any device work
    lib = J.load()
    h = np.array([0, 17, 40], dtype=np.int32)
    hp = h.ctypes.data_as(ctypes.c_void_p)
    if bwd:
        st = lib.jfa_bwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, hp, 2, 23, 2, 2, 128,
                                0.1, left, right, FAKE, 1 << 20, None)
    else:
        st = lib.jfa_fwd_window(FAKE, FAKE, FAKE, FAKE, None, FAKE, hp, 2, 23, 2, 2, 128, 0.1, left, right, FAKE,
                                1 << 20, None)
    assert st == 1


def test_window_plan_rejects_bad_bounds():
    h = np.array([0, 17, 40], dtype=np.int32)
    assert J.load().jfa_plan_window(0, h.ctypes.data_as(ctypes.c_void_p), 2, 2, -2, 0, 4, None, None) == -1
    assert J.load().jfa_plan_window(2, h.ctypes.data_as(ctypes.c_void_p), 2, 2, 0, 0, 4, None, None) == -1


def test_broadcast_row_count_overflow_rejected():
    # batch * nq broadcast output rows past the 32-bit row index range: rejected
    # before any device work (the empty sequences need no data)
    lib = J.load()
    h = np.zeros(70001, dtype=np.int32)
    st = lib.jfa_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, h.ctypes.data_as(ctypes.c_void_p), 70000, 0, 40000,
                     2, 2, 64, 0.125, 0, 1, FAKE, 1 << 20, None)
    assert st == 2


@pytest.mark.parametrize("offsets", [[5, 10], [0, 10, 4], [0, -1]])
def test_bad_offsets(offsets):
    assert _fwd(offsets, max_len=100) == 3


@pytest.mark.parametrize("H,Hkv,causal,bq,status", [
    (3, 2, 0, 0, 2),   # query heads not a multiple of key/value heads
    (4, 2, 1, 1, 2),   # causal broadcast-Q is undefined
    (4, 0, 0, 0, 1),   # no key/value heads
])
def test_bwd_argument_errors_before_device_work(H, Hkv, causal, bq, status):
    # every case returns before the device is touched, so the fake pointers are never used
    lib = J.load()
    h = np.array([0, 10, 20], dtype=np.int32)
    st = lib.jfa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, h.ctypes.data_as(ctypes.c_void_p),
                     2, 10, 16 if bq else 0, H, Hkv, 64, 0.125, causal, bq, FAKE, 1 << 20, None)
    assert st == status


def _bwd(**kw):
    # jfa_bwd with fake pointers; every case below is rejected before device work
    lib = J.load()
    h = np.array([0, 10, 20], dtype=np.int32)
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, D=64)
    a.update(kw)
    return lib.jfa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"], FAKE,
                       h.ctypes.data_as(ctypes.c_void_p), 2, 10, 0, 2, 2, a["D"], 0.125, 0, 0, FAKE, 1 << 20, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(do=None), 1), (dict(lse=None), 1), (dict(dq=None), 1), (dict(dk=None), 1), (dict(dv=None), 1),
    (dict(dq=MISALIGNED), 1), (dict(dk=MISALIGNED), 1), (dict(do=MISALIGNED), 1), (dict(D=96), 2),
])
def test_bwd_buffer_errors_before_device_work(kwargs, status):
    assert _bwd(**kwargs) == status


def _block(bwd, offsets=(0, 64, 100), D=128, scale=0.1, **kw):
    lib = J.load()
    h = np.ascontiguousarray(np.asarray(offsets, dtype=np.int32))
    batch = len(h) - 1
    max_len = int(np.max(np.diff(h))) if batch > 0 else 0
    hp = h.ctypes.data_as(ctypes.c_void_p)
    a = dict(dq=FAKE, dk=FAKE, dv=FAKE, do=FAKE)
    a.update(kw)
    if bwd:
        return lib.block_attn_bwd(FAKE, FAKE, FAKE, FAKE, a["do"], a["dq"], a["dk"], a["dv"], FAKE, hp, batch, max_len,
                                  2, D, scale, FAKE, 1 << 20, None)
    return lib.block_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, hp, batch, max_len, 2, D, scale, FAKE, 1 << 20, None)


@pytest.mark.parametrize("bwd", [False, True])
@pytest.mark.parametrize("kwargs,status", [
    (dict(D=96), 2), (dict(offsets=(0, 64, 30)), 3), (dict(offsets=(4, 64)), 3), (dict(scale=float("nan")), 1),
    (dict(scale=0.0), 1),
])
def test_block_argument_errors_before_device_work(bwd, kwargs, status):
    assert _block(bwd, **kwargs) == status


@pytest.mark.parametrize("kwargs", [dict(dq=None), dict(do=None), dict(dk=MISALIGNED), dict(dv=MISALIGNED)])
def test_block_bwd_buffer_errors_before_device_work(kwargs):
    assert _block(True, **kwargs) == 1


@pytest.mark.parametrize("which", ["schedule", "bwd_schedule", "block_schedule"])
def test_schedule_switches(which):
    # host-side state only: no device work
    lib = J.load()
    set_, get_ = getattr(lib, f"jfa_set_{which}"), getattr(lib, f"jfa_get_{which}")
    old = get_()
    try:
        assert set_(2) == 1 and set_(-1) == 1 and get_() == old
        for mode in (1, 0):
            assert set_(mode) == 0 and get_() == mode
    finally:
        set_(old)


def test_planner_hooks_reject_bad_input():
    lib = J.load()
    h = np.array([1, 5], dtype=np.int32)
    assert lib.jfa_plan_fwd(h.ctypes.data_as(ctypes.c_void_p), 1, 2, 0, 0, 4, None, None) == -3
    h = np.array([0, 5], dtype=np.int32)
    assert lib.jfa_plan_fwd(h.ctypes.data_as(ctypes.c_void_p), 1, 0, 0, 0, 4, None, None) == -1
    assert lib.block_plan(h.ctypes.data_as(ctypes.c_void_p), 1, 2, 0, None, None) == -1


def test_python_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        J._lib_missing = True
        ctypes_path = str(tmp_path / "nope.so")
        # a fresh loader pointed at a missing file must raise, never fall back
        saved = J._lib
        J._lib = None
        try:
            J.load(ctypes_path)
        finally:
            J._lib = saved


def test_binding_rejects_mismatched_shapes():
    # broadcast-Q called without nq_broadcast: q has the shared rows only, so the
    # binding must refuse before the library is asked to read past its end
    import torch
    offs = torch.tensor([0, 300, 700], dtype=torch.int32)
    q = torch.zeros((256, 2, 64), dtype=torch.bfloat16)
    k = torch.zeros((700, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="q: expected shape"):
        J._check_problem(q, k, k, offs, offs.numpy(), 0)
    with pytest.raises(ValueError, match="CUDA"):  # right shapes, but host tensors
        J._check_problem(q, k, k, offs, offs.numpy(), 256)


@pytest.mark.parametrize("by_keyword", [False, True])
def test_binding_rejects_host_tensors(by_keyword):
    # the entry points run under their tensors' CUDA device; host tensors are
    # rejected by the argument checks before the library is called
    q = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    offs = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        if by_keyword:
            V.jfa_fwd(q=q, k=q, v=q, offsets=offs, offsets_host=[0, 4])
        else:
            V.jfa_fwd(q, q, q, offs, [0, 4])


def test_topk_rows_count_query_blocks():
    # one row per (sequence with keys, query head, 256-row query block)
    import oracle
    from variable_length_attention_gb300 import workloads as W
    for w in (W.custom([1, 63, 128, 129, 255, 256, 257, 513, 1000], 2, 64), W.custom([300, 0, 900, 129], 3, 128, nq=300),
              W.jagged()):
        assert V.jfa_topk_rows(w.offsets, w.num_heads, w.nq) == len(oracle._topk_units(w.offsets, w.num_heads, w.nq))
