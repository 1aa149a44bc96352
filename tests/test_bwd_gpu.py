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
    # dQ, dK, dV of a seeded sample of (sequence, head) units, at least 8, the
    # first and last sequences among them
    w = W.dense(gqa=False)
    sel = sample_units(w.batch, w.num_heads, 8, seed=13)
    assert sel[0].any() and sel[w.batch - 1].any() and sel.sum() >= 8
    assert_bwd_ok(check_bwd(w, sel=sel))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv,D", [(4, 2, 64), (4, 1, 128), (8, 2, 128)])
def test_gqa(H, Hkv, D, causal):
    # dK and dV of a key/value head sum the gradients of its H/Hkv query heads;
    # sequences of several key blocks and query tiles, ragged tails, a 1-token one
    w = W.custom([300, 1, 129, 700, 256], H, D, num_kv_heads=Hkv, causal=causal,
                 seed_base=900 + 10 * H + Hkv + D + int(causal))
    assert_bwd_ok(check_bwd(w))


@pytest.mark.parametrize("Hkv", [1, 2])
def test_gqa_broadcast(Hkv):
    # broadcast-Q with groups: dQ of each query head sums over all sequences,
    # dK/dV of each key/value head over its group; an empty sequence included
    w = W.custom([200, 0, 77, 513, 129], 4, 128, num_kv_heads=Hkv, nq=192, seed_base=950 + Hkv)
    assert_bwd_ok(check_bwd(w))


def test_gqa_group_sum_identity():
    # the grouped call equals the ungrouped call on K/V repeated per query head,
    # with dK/dV summed over each group (checked on the GPU results themselves)
    w = W.custom([300, 129, 513], 4, 128, num_kv_heads=2, seed_base=960)
    (q, k, v, do), offs, _ = gpu_inputs(w)
    o, lse = V.jfa_fwd(q, k, v, offs, w.offsets)
    dq, dk, dv = V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets)
    kr, vr = k.repeat_interleave(2, dim=1).contiguous(), v.repeat_interleave(2, dim=1).contiguous()
    o2, lse2 = V.jfa_fwd(q, kr, vr, offs, w.offsets)
    dq2, dk2, dv2 = V.jfa_bwd(q, kr, vr, o2, do, lse2, offs, w.offsets)
    torch.cuda.synchronize()
    T = int(w.offsets[-1])
    dk2 = dk2.float().view(T, 2, 2, 128).sum(2)
    dv2 = dv2.float().view(T, 2, 2, 128).sum(2)
    for a, b in ((dq.float(), dq2.float()), (dk.float(), dk2), (dv.float(), dv2)):
        assert ((a - b).norm() / b.norm()).item() < 1e-2


@pytest.mark.parametrize("Hkv", [2, 1])
def test_backward_repeatable_except_dq_order(Hkv):
    w = W.custom([700, 33, 300], 2, 128, num_kv_heads=Hkv, seed_base=800)
    (q, k, v, do), offs, _ = gpu_inputs(w)
    o, lse = V.jfa_fwd(q, k, v, offs, w.offsets)
    g1 = V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets)
    g2 = V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets)
    torch.cuda.synchronize()
    # dK and dV are owned by one CTA each: bit-identical; dQ sums in arrival order
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert (g1[0].float() - g2[0].float()).abs().max().item() < 1e-2
