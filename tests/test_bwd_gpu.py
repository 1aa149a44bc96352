"""GPU parity of jfa_bwd (dQ, dK, dV) against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from tests.parity import assert_bwd_ok, check_bwd, gpu_inputs, sample_units

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 511, 513]


def test_tiny_workload():
    assert_bwd_ok(check_bwd(W.tiny()))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(D, causal):
    w = W.custom(EDGE_LENGTHS, 2, D, causal=causal, seed_base=600 + D + int(causal))
    assert_bwd_ok(check_bwd(w))


@pytest.mark.parametrize("nq", [1, 100, 256, 300])
@pytest.mark.parametrize("D", [64, 128])
def test_broadcast_small(nq, D):
    w = W.custom([5, 0, 130, 700, 64], 2, D, nq=nq, seed_base=700 + nq + D)
    assert_bwd_ok(check_bwd(w))


def test_jagged_full_size():
    w = W.jagged(False)
    assert_bwd_ok(check_bwd(w, sel=sample_units(w.batch, w.num_heads, 16, seed=11)))


def test_jagged_causal_full_size():
    w = W.jagged(True)
    assert_bwd_ok(check_bwd(w, sel=sample_units(w.batch, w.num_heads, 16, seed=12)))


def test_broadcast_full_size():
    # dQ of the shared Q needs every sequence: full oracle
    assert_bwd_ok(check_bwd(W.broadcast()))


def test_dense_full_size():
    w = W.dense(gqa=False)
    assert_bwd_ok(check_bwd(w, sel=sample_units(w.batch, w.num_heads, 4, seed=13)))


def test_gqa_backward_is_rejected():
    w = W.custom([100, 50], 4, 64, num_kv_heads=2)
    (q, k, v, do), offs, _ = gpu_inputs(w)
    o, lse = V.jfa_fwd(q, k, v, offs, w.offsets)
    with pytest.raises(V.jfa.JfaError) as e:
        V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets)
    assert e.value.status == 2


def test_backward_repeatable_except_dq_order():
    w = W.custom([700, 33, 300], 2, 128, seed_base=800)
    (q, k, v, do), offs, _ = gpu_inputs(w)
    o, lse = V.jfa_fwd(q, k, v, offs, w.offsets)
    g1 = V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets)
    g2 = V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets)
    torch.cuda.synchronize()
    # dK and dV are owned by one CTA each: bit-identical; dQ sums in arrival order
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert (g1[0].float() - g2[0].float()).abs().max().item() < 1e-2
