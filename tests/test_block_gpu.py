"""GPU parity of block_attn_fwd / block_attn_bwd (64-token block-diagonal
attention) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from variable_length_attention_gb300.workloads import offsets_from_lengths
from tests.parity import GRAD_REL_L2, O_MAX_ABS, O_REL_L2, rel_l2, to64

pytestmark = pytest.mark.gpu


def _run(w, q, k, v, do):
    offs = torch.from_numpy(w.offsets).to(q.device)
    o = V.block_attn_fwd(q, k, v, offs, w.offsets, scale=w.scale)
    dq, dk, dv = V.block_attn_bwd(q, k, v, o, do, offs, w.offsets, scale=w.scale)
    torch.cuda.synchronize()
    return o, dq, dk, dv


def _compare(w, seqs, q, k, v, do, o, dq, dk, dv):
    """Oracle on the chosen sequences only (blocks never cross sequences)."""
    offs = w.offsets
    rows = np.concatenate([np.arange(offs[b], offs[b + 1]) for b in seqs])
    sub = offsets_from_lengths([offs[b + 1] - offs[b] for b in seqs])
    idx = torch.from_numpy(rows).to(q.device)
    pick = lambda t: to64(t.index_select(0, idx))  # noqa: E731
    q64, k64, v64, do64 = pick(q), pick(k), pick(v), pick(do)
    o_ref, _ = oracle.block_fwd(q64, k64, v64, sub, scale=w.scale)
    g_ref = oracle.block_bwd(q64, k64, v64, do64, sub, scale=w.scale)
    og = pick(o)
    res = {"o_max_abs": float(np.max(np.abs(og - o_ref))), "o_rel_l2": rel_l2(og, o_ref)}
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref[:3]):
        res[name] = rel_l2(pick(g), r)
    return res


def _assert(res):
    assert res["o_max_abs"] <= O_MAX_ABS and res["o_rel_l2"] <= O_REL_L2, res
    for name in ("dq", "dk", "dv"):
        assert res[name] <= GRAD_REL_L2, res


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lengths", [[64, 128, 192], [130, 64, 7, 1, 0, 63, 65, 200], [4032] * 3])
def test_block_small(D, lengths):
    w = W.custom(lengths, 2, D, mode="block", seed_base=900 + D + len(lengths))
    q, k, v, do = [t.cuda() for t in w.tensors("cpu")]
    o, dq, dk, dv = _run(w, q, k, v, do)
    _assert(_compare(w, range(w.batch), q, k, v, do, o, dq, dk, dv))


def test_block_odd_block_count_and_empty():
    # 3 blocks in total: the last tile has no second block
    w = W.custom([0, 150, 0], 3, 64, mode="block", seed_base=950)
    q, k, v, do = [t.cuda() for t in w.tensors("cpu")]
    o, dq, dk, dv = _run(w, q, k, v, do)
    _assert(_compare(w, [1], q, k, v, do, o, dq, dk, dv))


@pytest.mark.parametrize("D", [64, 128])
def test_block_full_size(D):
    """Batch 1152 x 4032 tokens (63 blocks each), H=4: inputs drawn on the GPU,
    a seeded sample of sequences checked against the oracle."""
    w = W.block(D)
    q, k, v, do = w.tensors("cuda")
    o, dq, dk, dv = _run(w, q, k, v, do)
    rng = np.random.default_rng(D)
    seqs = sorted(set([0, w.batch - 1] + rng.choice(w.batch, 4, replace=False).tolist()))
    _assert(_compare(w, seqs, q, k, v, do, o, dq, dk, dv))
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
