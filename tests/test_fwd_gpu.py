"""GPU parity of jfa_fwd against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from tests.parity import assert_fwd_ok, check_fwd, sample_units

pytestmark = pytest.mark.gpu


def test_tiny_workload():
    res, _ = check_fwd(W.tiny())
    assert_fwd_ok(res)


EDGE_LENGTHS = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 511, 513]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(D, causal):
    w = W.custom(EDGE_LENGTHS, 2, D, causal=causal, seed_base=100 + D + int(causal))
    res, _ = check_fwd(w)
    assert_fwd_ok(res)


@pytest.mark.parametrize("H,Hkv", [(4, 2), (4, 1), (8, 8)])
def test_gqa(H, Hkv):
    w = W.custom([300, 77, 129, 1], H, 128, num_kv_heads=Hkv, seed_base=200 + H + Hkv)
    res, _ = check_fwd(w)
    assert_fwd_ok(res)


@pytest.mark.parametrize("nq", [1, 100, 256, 300])
def test_broadcast_small(nq):
    w = W.custom([5, 0, 130, 700, 64], 2, 128, nq=nq, seed_base=300 + nq)
    res, _ = check_fwd(w)
    assert_fwd_ok(res)


def test_empty_batch_and_empty_sequences():
    w = W.custom([0, 0, 40, 0], 2, 64, seed_base=400)
    res, _ = check_fwd(w)
    assert_fwd_ok(res)


def test_jagged_full_size():
    w = W.jagged(False)
    res, _ = check_fwd(w, sel=sample_units(w.batch, w.num_heads, 24, seed=1))
    assert_fwd_ok(res)


def test_jagged_causal_full_size():
    w = W.jagged(True)
    res, _ = check_fwd(w, sel=sample_units(w.batch, w.num_heads, 24, seed=2))
    assert_fwd_ok(res)


def test_broadcast_full_size():
    w = W.broadcast()
    res, _ = check_fwd(w, sel=sample_units(w.batch, w.num_heads, 64, seed=3))
    assert_fwd_ok(res)


def test_dense_gqa_full_size():
    w = W.dense(gqa=True)
    res, _ = check_fwd(w, sel=sample_units(w.batch, w.num_heads, 6, seed=4))
    assert_fwd_ok(res)


def test_repeatable_and_no_lse():
    w = W.custom([700, 33], 2, 128, seed_base=500)
    (q, k, v, _), offs, _ = __import__("tests.parity", fromlist=["gpu_inputs"]).gpu_inputs(w)
    o1, l1 = V.jfa_fwd(q, k, v, offs, w.offsets)
    o2, l2 = V.jfa_fwd(q, k, v, offs, w.offsets)
    o3, none = V.jfa_fwd(q, k, v, offs, w.offsets, return_lse=False)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)
