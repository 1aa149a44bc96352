"""jfa_fwd_noalloc: the forward for callers that cannot allocate device memory.

Callers inside a framework whose memory manager owns every device allocation,
or serving loops that must never allocate, cannot give the library a
workspace.  jfa_fwd_noalloc keeps its plan in the library's own fixed static
scratch instead.  This test calls it through the C ABI (ctypes, device pointers
from torch tensors that the test itself allocates as inputs and outputs) and
checks it against jfa_fwd, the workspace-taking entry point, on two calls in a
row, with the same tolerances as the forward parity tests.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import jfa as J
from variable_length_attention_gb300 import workloads as W
from tests.parity import O_MAX_ABS, O_REL_L2, LSE_MAX_ABS, rel_l2

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


@pytest.mark.parametrize("w", [W.jagged(False), W.jagged(True), W.custom([5, 0, 130, 700, 64], 2, 128, nq=300),
                               W.custom([1, 63, 64, 65, 129, 257], 2, 64)],
                         ids=["jagged", "jagged_causal", "broadcast_with_empty", "edges_d64"])
def test_noalloc_matches_workspace_entry_point(w):
    q, k, v, _ = [t.cuda() for t in w.tensors("cpu")]
    offs = torch.from_numpy(w.offsets).cuda()
    o_ref, lse_ref = V.jfa_fwd(q, k, v, offs, w.offsets, causal=w.causal, nq_broadcast=w.nq)
    o_ref, lse_ref = o_ref.double().cpu().numpy(), lse_ref.double().cpu().numpy()
    for _ in range(2):  # two calls in a row share (and overwrite) the static scratch
        o = torch.full((w.o_rows, w.num_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.num_heads, w.o_rows), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc_raw(w, q, k, v, offs, o, lse) == 0
        torch.cuda.synchronize()
        og, lg = o.double().cpu().numpy(), lse.double().cpu().numpy()
        assert np.all(np.isfinite(og))
        assert np.max(np.abs(og - o_ref)) <= O_MAX_ABS
        assert rel_l2(og, o_ref) <= O_REL_L2
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
        assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= LSE_MAX_ABS


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
