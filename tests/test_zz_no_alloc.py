"""jfa_fwd_noalloc: the forward for callers that cannot allocate device memory.

Callers inside a framework whose memory manager owns every device allocation,
or serving loops that must never allocate, cannot give the library a
workspace.  jfa_fwd_noalloc keeps its plan in the library's own fixed static
scratch instead.  These tests call it through the C ABI (ctypes, device
pointers from torch tensors that the test itself allocates as inputs and
outputs) and check it against the fp64 oracle and against jfa_fwd, the
workspace-taking entry point, on two calls in a row and on a sequence of
different problems that share the scratch, with the tolerances of the forward
parity tests; after every call jfa_fwd_noalloc_status() must report JFA_OK.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import jfa as J
from variable_length_attention_gb300 import workloads as W
from tests.parity import LSE_MAX_ABS, O_MAX_ABS, O_REL_L2, rel_l2, rows_of, sample_units, to64

pytestmark = pytest.mark.gpu


def _noalloc_raw(w, q, k, v, offs, o, lse):
    """One call of jfa_fwd_noalloc through the C ABI."""
    lib = J.load()
    h = np.ascontiguousarray(w.offsets.astype(np.int32))
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.jfa_fwd_noalloc(p(q), p(k), p(v), p(o), p(lse), p(offs), h.ctypes.data_as(ctypes.c_void_p),
                               w.batch, w.max_len, w.nq, w.num_heads, w.num_kv_heads, w.head_dim, w.scale,
                               int(w.causal), int(w.nq > 0),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _status():
    return J.load().jfa_fwd_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(og, lg, o_ref, lse_ref):
    assert np.all(np.isfinite(og))
    assert np.max(np.abs(og - o_ref)) <= O_MAX_ABS
    assert rel_l2(og, o_ref) <= O_REL_L2
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    if fin.any():
        assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= LSE_MAX_ABS


def _run(w, q, k, v, offs):
    o = torch.full((w.o_rows, w.num_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.num_heads, w.o_rows), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc_raw(w, q, k, v, offs, o, lse) == 0
    assert _status() == 0
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


CASES = [W.jagged(False), W.jagged(True), W.custom([5, 0, 130, 700, 64], 2, 128, nq=300),
         W.custom([1, 63, 64, 65, 129, 257], 2, 64)]


@pytest.mark.parametrize("w", CASES, ids=["jagged", "jagged_causal", "broadcast_with_empty", "edges_d64"])
def test_noalloc_matches_oracle_and_workspace_entry_point(w):
    q, k, v, _ = w.tensors("cpu")
    # the oracle on every unit of the small cases, on a seeded sample of
    # (sequence, head) units, the first and last sequence included, at full size
    sel = sample_units(w.batch, w.num_heads, 12, seed=21) if w.total_tokens > 10000 else None
    o_or, lse_or, _ = oracle.attn_fwd(to64(q), to64(k), to64(v), w.offsets, scale=w.scale, causal=w.causal,
                                      nq=w.nq, sel=sel)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    offs = torch.from_numpy(w.offsets).cuda()
    o_ws, lse_ws = V.jfa_fwd(q, k, v, offs, w.offsets, causal=w.causal, nq_broadcast=w.nq)
    o_ws, lse_ws = o_ws.double().cpu().numpy(), lse_ws.double().cpu().numpy()
    m = rows_of(w.offsets, sel, w.num_heads, w.nq) if sel is not None else None
    for _ in range(2):  # two calls in a row share (and overwrite) the static scratch
        og, lg = _run(w, q, k, v, offs)
        _close(og, lg, o_ws, lse_ws)
        if m is None:
            _close(og, lg, o_or, lse_or)
        else:
            _close(og[m], lg.T[m], o_or[m], lse_or.T[m])


def test_noalloc_sequence_of_different_problems():
    """Problems of different sizes and modes, one after another on the same
    static scratch: a large plan, then a tiny one (a stale tail of the larger
    plan must not be read), broadcast-Q with empty sequences, then
    self-attention without any."""
    seq = [W.jagged(False), W.tiny(), W.custom([0, 300, 0, 17], 2, 128, nq=129, seed_base=31),
           W.custom([200, 1, 65], 4, 128, num_kv_heads=2, causal=True, seed_base=32), W.tiny()]
    for w in seq:
        q, k, v, _ = [t.cuda() for t in w.tensors("cpu")]
        offs = torch.from_numpy(w.offsets).cuda()
        o_ws, lse_ws = V.jfa_fwd(q, k, v, offs, w.offsets, causal=w.causal, nq_broadcast=w.nq)
        og, lg = _run(w, q, k, v, offs)
        _close(og, lg, o_ws.double().cpu().numpy(), lse_ws.double().cpu().numpy())


def test_noalloc_status_reports_a_timed_out_wait():
    """The bounded-wait self-test with its error word in the static scratch: the
    status call reports the timeout (after about 2 s, with no fault), and the
    next jfa_fwd_noalloc call clears it and still computes the right result."""
    J.load()
    assert J.load().jfa_selftest_wait_timeout_noalloc(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    assert _status() == 7  # JFA_ERR_DEVICE_TIMEOUT
    w = W.tiny()
    q, k, v, _ = w.tensors("cpu")
    o_or, lse_or, _ = oracle.attn_fwd(to64(q), to64(k), to64(v), w.offsets, scale=w.scale)
    og, lg = _run(w, q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(w.offsets).cuda())
    _close(og, lg, o_or, lse_or)


def test_noalloc_rejects_a_plan_beyond_its_capacity():
    cap = J.load().jfa_fwd_noalloc_capacity()
    assert cap == 1 << 20
    # 300,000 single-token sequences need 300,000 forward units (16 bytes each)
    w = W.custom([1] * 300000, 1, 64)
    q, k, v, _ = [t.cuda() for t in w.tensors("cpu")]
    offs = torch.from_numpy(w.offsets).cuda()
    o = torch.empty((w.o_rows, 1, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, w.o_rows), dtype=torch.float32, device="cuda")
    assert _noalloc_raw(w, q, k, v, offs, o, lse) == 8  # JFA_ERR_TOO_LARGE
