"""Failure detection on the GPU without faulting it: a wait that nothing
completes runs out its bound, the error word says so, and the context keeps
working for the next call."""
import time

import pytest
import torch

import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from tests.parity import assert_fwd_ok, check_fwd

pytestmark = pytest.mark.gpu

JFA_OK, JFA_ERR_DEVICE_TIMEOUT = 0, 7


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    V.jfa_selftest_wait_timeout(ws)
    assert V.jfa_device_status(ws) == JFA_ERR_DEVICE_TIMEOUT
    waited = time.perf_counter() - t0
    assert 1.0 < waited < 30.0, waited  # the 2 s bound, not a hang
    # the same context runs a normal call afterwards, and its status is clean
    res, _ = check_fwd(W.tiny())
    assert_fwd_ok(res)
    w = W.tiny()
    q, k, v, _ = (t.cuda() for t in w.tensors("cpu"))
    offs = torch.from_numpy(w.offsets).cuda()
    ws2 = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    V.jfa_fwd(q, k, v, offs, w.offsets, workspace=ws2)
    assert V.jfa_device_status(ws2) == JFA_OK


def test_selftest_rejects_small_workspace():
    with pytest.raises(V.jfa.JfaError):
        V.jfa_selftest_wait_timeout(torch.zeros(2, dtype=torch.uint8, device="cuda"))
