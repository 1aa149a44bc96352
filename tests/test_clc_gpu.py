"""The jagged forward and backward under Cluster Launch Control scheduling: same
results as the static plan (parity with the oracle, and bit-identical outputs
where each output is owned by one unit, since a unit is computed by one CTA in
the same way whichever CTA takes it; the backward's dQ sums units in arrival
order)."""
import pytest
import torch

import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from tests.parity import assert_bwd_ok, assert_fwd_ok, check_bwd, check_fwd, gpu_inputs, sample_units

pytestmark = pytest.mark.gpu


@pytest.fixture
def clc_mode():
    old = V.jfa_get_schedule()
    V.jfa_set_schedule("clc")
    yield
    V.jfa_set_schedule(old)


@pytest.mark.parametrize("w", [W.tiny(), W.custom([1, 63, 129, 257, 513, 1000], 2, 128, causal=True, seed_base=40),
                               W.custom([5, 0, 130, 700], 2, 64, nq=300, seed_base=41)],
                         ids=["tiny", "causal_edges", "broadcast"])
def test_clc_parity(clc_mode, w):
    res, _ = check_fwd(w)
    assert_fwd_ok(res)


def test_clc_full_size_matches_static(clc_mode):
    w = W.jagged(False)
    (q, k, v, _), offs, _ = gpu_inputs(w)
    o_clc, l_clc = V.jfa_fwd(q, k, v, offs, w.offsets)
    V.jfa_set_schedule("static")
    o_st, l_st = V.jfa_fwd(q, k, v, offs, w.offsets)
    torch.cuda.synchronize()
    assert torch.equal(o_clc, o_st) and torch.equal(l_clc, l_st)
    V.jfa_set_schedule("clc")
    res, _ = check_fwd(w, sel=sample_units(w.batch, w.num_heads, 8, seed=5))
    assert_fwd_ok(res)


@pytest.fixture
def bwd_clc_mode():
    old = V.jfa_get_bwd_schedule()
    V.jfa_set_bwd_schedule("clc")
    yield
    V.jfa_set_bwd_schedule(old)


@pytest.mark.parametrize("w", [W.tiny(), W.custom([1, 63, 129, 257, 513, 1000], 2, 128, causal=True, seed_base=42),
                               W.custom([5, 0, 130, 700], 2, 64, nq=300, seed_base=43),
                               W.custom([300, 129, 700], 4, 128, num_kv_heads=2, seed_base=44)],
                         ids=["tiny", "causal_edges", "broadcast", "gqa"])
def test_bwd_clc_parity(bwd_clc_mode, w):
    assert_bwd_ok(check_bwd(w))


def test_bwd_clc_full_size_matches_static(bwd_clc_mode):
    # causal: units of very different costs, so CTAs take over many units
    w = W.jagged(True)
    (q, k, v, do), offs, _ = gpu_inputs(w)
    o, lse = V.jfa_fwd(q, k, v, offs, w.offsets, causal=True)
    g_clc = V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets, causal=True)
    V.jfa_set_bwd_schedule("static")
    g_st = V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets, causal=True)
    torch.cuda.synchronize()
    V.jfa_set_bwd_schedule("clc")
    # dK and dV are owned by one unit each: bit-identical; dQ sums in arrival order
    assert torch.equal(g_clc[1], g_st[1]) and torch.equal(g_clc[2], g_st[2])
    assert (g_clc[0].float() - g_st[0].float()).abs().max().item() < 1e-2
    assert_bwd_ok(check_bwd(w, sel=sample_units(w.batch, w.num_heads, 8, seed=6)))


@pytest.fixture
def block_clc_mode():
    old = V.jfa_get_block_schedule()
    V.jfa_set_block_schedule("clc")
    yield
    V.jfa_set_block_schedule(old)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lengths", [[64, 128, 192], [130, 64, 7, 1, 0, 63, 65, 200], [4032] * 3, [0, 150, 0]])
def test_block_clc_parity(block_clc_mode, D, lengths):
    # chunks of 16 tiles taken under Cluster Launch Control: parity with the
    # oracle, including tail blocks, empty sequences and an odd block count
    from tests.test_block_gpu import _assert, _compare, _run
    w = W.custom(lengths, 3, D, mode="block", seed_base=970 + D + len(lengths))
    q, k, v, do = [t.cuda() for t in w.tensors("cpu")]
    o, dq, dk, dv = _run(w, q, k, v, do)
    _assert(_compare(w, [b for b in range(w.batch) if w.lengths[b] > 0], q, k, v, do, o, dq, dk, dv))


@pytest.mark.parametrize("D", [64, 128])
def test_block_clc_matches_static(block_clc_mode, D):
    # every tile owns its outputs, so the two schedules give identical bits
    from tests.test_block_gpu import _run
    w = W.block(D, batch=96)
    q, k, v, do = w.tensors("cuda")
    r_clc = _run(w, q, k, v, do)
    V.jfa_set_block_schedule("static")
    r_st = _run(w, q, k, v, do)
    V.jfa_set_block_schedule("clc")
    for a, b in zip(r_clc, r_st):
        assert torch.equal(a, b)
