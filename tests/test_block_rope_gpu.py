"""GPU parity of the rotary block-diagonal entry points (block_attn_fwd_rope,
block_attn_bwd_rope) against the fp64 oracle, through the C ABI.

The cos/sin tables handed to the kernels are inputs: built here from the
rotate-half convention (angle p * base^(-2i/D) for position p and pair i),
rounded to fp32.  The oracle rotates the exact bf16 inputs in fp64 from the
same convention on its own (oracle.rope) and differentiates through it."""
import math

import numpy as np
import pytest
import torch

import oracle
import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from variable_length_attention_gb300.workloads import offsets_from_lengths
from tests.parity import GRAD_REL_L2, O_MAX_ABS, O_REL_L2, rel_l2, to64

pytestmark = pytest.mark.gpu

BASE = 10000.0


def _tables(positions, D, device="cuda"):
    ang = np.arange(positions)[:, None] * BASE ** (-2.0 * np.arange(D // 2) / D)[None, :]
    return (torch.from_numpy(np.cos(ang)).float().to(device).contiguous(),
            torch.from_numpy(np.sin(ang)).float().to(device).contiguous())


def _run(w, q, k, v, do):
    offs = torch.from_numpy(w.offsets).to(q.device)
    rope = _tables(max(w.max_len, 1), w.head_dim, q.device)
    o = V.block_attn_fwd(q, k, v, offs, w.offsets, scale=w.scale, rope=rope)
    dq, dk, dv = V.block_attn_bwd(q, k, v, o, do, offs, w.offsets, scale=w.scale, rope=rope)
    torch.cuda.synchronize()
    return o, dq, dk, dv


def _compare(w, seqs, q, k, v, do, o, dq, dk, dv):
    offs = w.offsets
    rows = np.concatenate([np.arange(offs[b], offs[b + 1]) for b in seqs])
    sub = offsets_from_lengths([offs[b + 1] - offs[b] for b in seqs])
    idx = torch.from_numpy(rows).to(q.device)
    pick = lambda t: to64(t.index_select(0, idx))  # noqa: E731
    q64, k64, v64, do64 = pick(q), pick(k), pick(v), pick(do)
    o_ref, _ = oracle.block_fwd(q64, k64, v64, sub, scale=w.scale, rope_base=BASE)
    g_ref = oracle.block_bwd(q64, k64, v64, do64, sub, scale=w.scale, rope_base=BASE)
    og = pick(o)
    res = {"o_max_abs": float(np.max(np.abs(og - o_ref))), "o_rel_l2": rel_l2(og, o_ref)}
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref[:3]):
        res[name] = rel_l2(pick(g), r)
    return res


# The kernels round the rotated q and k rows to bf16 before the score GEMM (its
# operands are bf16), one rounding more than the unrotated kernels and the
# fp64 oracle make: each score moves by up to about scale * |q| |k| 2^-8, and
# on the largest outputs the maximum deviation grows accordingly, so the
# rotary variant's O max-abs bound is twice the plain one; its relative L2
# bounds are the plain ones.
ROPE_O_MAX_ABS = 2 * O_MAX_ABS


def _assert(res):
    assert res["o_max_abs"] <= ROPE_O_MAX_ABS and res["o_rel_l2"] <= O_REL_L2, res
    for name in ("dq", "dk", "dv"):
        assert res[name] <= GRAD_REL_L2, res


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lengths", [[64, 128, 192], [130, 64, 7, 1, 0, 63, 65, 200], [4032] * 3, [0, 150, 0]])
def test_rope_block_small(D, lengths):
    w = W.custom(lengths, 2, D, mode="block", seed_base=1500 + D + len(lengths))
    q, k, v, do = [t.cuda() for t in w.tensors("cpu")]
    o, dq, dk, dv = _run(w, q, k, v, do)
    _assert(_compare(w, [b for b in range(w.batch) if w.lengths[b] > 0], q, k, v, do, o, dq, dk, dv))


@pytest.mark.parametrize("sched", ["static", "clc"])
def test_rope_block_schedules_agree(sched):
    # both schedules, positions up to 4031: bit-identical results (each tile owns its rows)
    w = W.block(128, batch=48)
    q, k, v, do = w.tensors("cuda")
    old = V.jfa_get_block_schedule()
    try:
        V.jfa_set_block_schedule(sched)
        r1 = _run(w, q, k, v, do)
        V.jfa_set_block_schedule("clc" if sched == "static" else "static")
        r2 = _run(w, q, k, v, do)
    finally:
        V.jfa_set_block_schedule(old)
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)
    _assert(_compare(w, [0, 47], q, k, v, do, *r1))


@pytest.mark.parametrize("D", [64, 128])
def test_rope_block_full_size(D):
    """Batch 1152 x 4032 tokens, H=4, rotary fused: a seeded sample of
    sequences (the first and the last among them) against the oracle."""
    w = W.block(D)
    q, k, v, do = w.tensors("cuda")
    o, dq, dk, dv = _run(w, q, k, v, do)
    rng = np.random.default_rng(D + 7)
    seqs = sorted(set([0, w.batch - 1] + rng.choice(w.batch, 3, replace=False).tolist()))
    _assert(_compare(w, seqs, q, k, v, do, o, dq, dk, dv))


def test_rope_tables_must_cover_every_position():
    w = W.custom([100, 30], 1, 64, mode="block", seed_base=1600)
    q, k, v, _ = [t.cuda() for t in w.tensors("cpu")]
    offs = torch.from_numpy(w.offsets).cuda()
    with pytest.raises(V.jfa.JfaError):
        V.block_attn_fwd(q, k, v, offs, w.offsets, rope=_tables(99, 64))  # positions 0..99 needed


def test_rope_workspace_holds_the_packed_table():
    """The rotary calls pack the tables as (cos, sin) half2 pairs into the
    workspace: their size exceeds the plain block calls' by one table of
    longest-sequence x D/2 x 4 bytes (rounded up to 256), and a workspace of the
    plain size is refused before any work."""
    from variable_length_attention_gb300 import jfa as J
    w = W.custom([100, 0, 30, 64], 2, 64, mode="block", seed_base=1700)
    table = -(-(100 * (w.head_dim // 2) * 4) // 256) * 256
    for plain, rot in ((J.JFA_OP_BLOCK_FWD, J.JFA_OP_BLOCK_FWD_ROPE), (J.JFA_OP_BLOCK_BWD, J.JFA_OP_BLOCK_BWD_ROPE)):
        a = V.jfa_workspace_size(plain, w.offsets, w.batch, 0, w.num_heads, w.head_dim, 0, 0)
        b = V.jfa_workspace_size(rot, w.offsets, w.batch, 0, w.num_heads, w.head_dim, 0, 0)
        assert a > 0 and b == a + table
    q, k, v, _ = [t.cuda() for t in w.tensors("cpu")]
    offs = torch.from_numpy(w.offsets).cuda()
    small = torch.empty(V.jfa_workspace_size(J.JFA_OP_BLOCK_FWD, w.offsets, w.batch, 0, w.num_heads, w.head_dim, 0, 0),
                        dtype=torch.uint8, device="cuda")
    with pytest.raises(V.jfa.JfaError, match="WORKSPACE"):
        V.block_attn_fwd(q, k, v, offs, w.offsets, rope=_tables(100, 64), workspace=small)
