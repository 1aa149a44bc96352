"""GPU parity of the sliding-window entry points (jfa_fwd_window,
jfa_bwd_window) against the fp64 oracle, through the C ABI.

Query i of a sequence sees keys i - left .. i + right of its sequence (None:
that side open).  The windows cover one key (the identity), causal windows
shorter, equal to and longer than a 128-key block, two-sided windows, and
windows open on one side, on sequence lengths around every tile size, at head
size 64 and 128, with grouped K/V heads, and at full size on the jagged
workload."""
import pytest
import torch

import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from tests.parity import assert_bwd_ok, assert_fwd_ok, check_bwd, check_fwd, gpu_inputs, sample_units

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 511, 513]
WINDOWS = [(0, 0), (63, 0), (127, 0), (128, 0), (255, 0), (300, 40), (None, 129), (1000, None), (5, 5),
           (130, 260)]


@pytest.mark.parametrize("window", WINDOWS, ids=[str(x) for x in WINDOWS])
@pytest.mark.parametrize("D", [64, 128])
def test_window_forward_edges(window, D):
    w = W.custom(EDGE_LENGTHS, 2, D, seed_base=1100 + D)
    res, _ = check_fwd(w, window=window)
    assert_fwd_ok(res)


@pytest.mark.parametrize("window", WINDOWS, ids=[str(x) for x in WINDOWS])
@pytest.mark.parametrize("D", [64, 128])
def test_window_backward_edges(window, D):
    w = W.custom([1, 63, 129, 256, 257, 513, 700], 2, D, seed_base=1200 + D)
    assert_bwd_ok(check_bwd(w, window=window))


@pytest.mark.parametrize("window", [(127, 0), (200, 30)], ids=["causal127", "two_sided"])
def test_window_grouped_heads(window):
    w = W.custom([300, 1, 129, 700], 4, 128, num_kv_heads=2, seed_base=1300)
    res, _ = check_fwd(w, window=window)
    assert_fwd_ok(res)
    assert_bwd_ok(check_bwd(w, window=window))


def test_window_jagged_full_size():
    # the jagged workload (B=32, lengths 32..4096, H=8, D=128) under a causal
    # window of 1024 keys: a seeded sample of (sequence, head) units
    w = W.jagged(False)
    sel = sample_units(w.batch, w.num_heads, 12, seed=31)
    res, _ = check_fwd(w, sel=sel, window=(1023, 0))
    assert_fwd_ok(res)
    assert_bwd_ok(check_bwd(w, sel=sel, window=(1023, 0)))


def test_wide_window_equals_full_attention():
    # a window wider than every sequence is plain attention: the same outputs as
    # jfa_fwd / jfa_bwd within the kernels' rounding
    w = W.custom([700, 33, 300], 2, 128, seed_base=1400)
    (q, k, v, do), offs, _ = gpu_inputs(w)
    o1, l1 = V.jfa_fwd(q, k, v, offs, w.offsets)
    o2, l2 = V.jfa_fwd(q, k, v, offs, w.offsets, window=(5000, 5000))
    g1 = V.jfa_bwd(q, k, v, o1, do, l1, offs, w.offsets)
    g2 = V.jfa_bwd(q, k, v, o2, do, l2, offs, w.offsets, window=(5000, 5000))
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() < 1e-2
    assert (l1 - l2).abs().max().item() < 1e-3
    for a, b in zip(g1, g2):
        assert ((a.float() - b.float()).norm() / b.float().norm()).item() < 1e-2
