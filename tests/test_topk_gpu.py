"""GPU parity of the two-stage block-sparse forward (jfa_topk_select,
jfa_fwd_topk) against the fp64 oracle, through the C ABI.

Stage one decides integers (which key blocks) from floating-point scores, and
the GPU forms its block means in fp32 while the oracle uses fp64, so near-ties
may be broken either way: the test checks that the GPU's choice is a valid
top-k under the oracle's scores (every chosen score at least every unchosen
one, up to the fp32 rounding of the scores), that it equals the oracle's
choice wherever the k-th and (k+1)-th scores are apart, and its format
(ascending, in range, -1 padded).  Stage two is compared with the oracle's
block-sparse attention on the GPU's own choice, at the forward tolerances."""
import numpy as np
import pytest
import torch

import oracle
import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from tests.parity import LSE_MAX_ABS, O_MAX_ABS, O_REL_L2, rel_l2, to64

pytestmark = pytest.mark.gpu


def _check_selection(sel, scores, topk):
    sel = sel.cpu().numpy()
    assert sel.shape == (len(scores), topk)
    exact = 0
    for row, sc in zip(sel, scores):
        cnt = min(topk, len(sc))
        chosen = row[:cnt]
        assert np.all(row[cnt:] == -1)
        assert np.all(np.diff(chosen) > 0) and chosen.min() >= 0 and chosen.max() < len(sc)
        rest = np.setdiff1d(np.arange(len(sc)), chosen)
        tol = 1e-4 * np.max(np.abs(sc)) + 1e-6
        if len(rest):
            assert sc[chosen].min() >= sc[rest].max() - tol, (sc, chosen)
        want = oracle.topk_select([sc], topk)[0]
        ordered = np.sort(sc)[::-1]
        if len(sc) <= topk or ordered[cnt - 1] - ordered[cnt] > tol:
            assert list(chosen) == want
            exact += 1
    return exact


def _run(w, topk):
    q, k, v, _ = w.tensors("cpu")
    offs = torch.from_numpy(w.offsets).cuda()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    sel = V.jfa_topk_select(qd, kd, offs, w.offsets, topk=topk, nq_broadcast=w.nq)
    o, lse = V.jfa_fwd_topk(qd, kd, vd, offs, sel, w.offsets, topk=topk, nq_broadcast=w.nq, scale=w.scale)
    torch.cuda.synchronize()
    q64, k64, v64 = to64(q), to64(k), to64(v)
    scores = oracle.topk_scores(q64, k64, w.offsets, nq=w.nq)
    exact = _check_selection(sel, scores, topk)
    selection = [[int(j) for j in row if j >= 0] for row in sel.cpu().numpy()]
    o_ref, lse_ref = oracle.attn_fwd_topk(q64, k64, v64, w.offsets, selection, scale=w.scale, nq=w.nq)
    og, lg = to64(o), to64(lse)
    assert np.all(np.isfinite(og))
    assert np.max(np.abs(og - o_ref)) <= O_MAX_ABS
    assert rel_l2(og, o_ref) <= O_REL_L2
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= LSE_MAX_ABS
    return exact, len(scores)


@pytest.mark.parametrize("topk", [1, 2, 3, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_topk_edges(topk, D):
    w = W.custom([1, 63, 128, 129, 255, 256, 257, 513, 1000], 2, D, seed_base=1700 + D + topk)
    exact, rows = _run(w, topk)
    assert exact >= rows // 2


def test_topk_grouped_heads():
    w = W.custom([700, 129, 2000], 4, 128, num_kv_heads=2, seed_base=1710)
    _run(w, 4)


@pytest.mark.parametrize("topk", [2, 5])
def test_topk_broadcast_with_empty_sequence(topk):
    w = W.custom([300, 0, 900, 129], 2, 128, nq=300, seed_base=1720 + topk)
    _run(w, topk)


def test_topk_jagged_full_size():
    # the jagged workload (lengths 32..4096, H=8, D=128) keeping half of at most 32 blocks
    w = W.jagged(False)
    exact, rows = _run(w, 8)
    assert exact >= 0.9 * rows


def test_topk_covering_every_block_is_full_attention():
    w = W.custom([700, 33, 300], 2, 128, seed_base=1730)
    q, k, v, _ = [t.cuda() for t in w.tensors("cpu")]
    offs = torch.from_numpy(w.offsets).cuda()
    sel = V.jfa_topk_select(q, k, offs, w.offsets, topk=6)
    o1, l1 = V.jfa_fwd_topk(q, k, v, offs, sel, w.offsets, topk=6)
    o2, l2 = V.jfa_fwd(q, k, v, offs, w.offsets)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() < 1e-2
    assert (l1 - l2).abs().max().item() < 1e-3


def test_topk_longest_sequence_limit():
    """The selection keeps one score per key block of the longest sequence in
    shared memory (48 KB): a sequence of 12,288 key blocks (1,572,864 keys) runs,
    one key more is refused before any work.  The inputs make the answer exact:
    every query row is the same vector u, every key row zero except in four key
    blocks, whose rows are c u with distinct c > 0, so every query block picks
    those four blocks (bf16-exact values, no near-ties)."""
    n_blk, D, topk = 12288, 64, 4
    T = n_blk * 128
    u = torch.full((D,), 0.125, dtype=torch.bfloat16, device="cuda")
    q = u.expand(T + 1, 1, D).contiguous()
    k = torch.zeros((T + 1, 1, D), dtype=torch.bfloat16, device="cuda")
    chosen = [5, 100, 7777, n_blk - 1]
    for blk, c in zip(chosen, [1.0, 0.875, 0.75, 0.625]):
        k[128 * blk:128 * (blk + 1), 0] = (u.float() * c).to(torch.bfloat16)
    offs_h = np.array([0, T], dtype=np.int32)
    sel = V.jfa_topk_select(q[:T], k[:T], torch.from_numpy(offs_h).cuda(), offs_h, topk=topk)
    torch.cuda.synchronize()
    assert sel.shape == (T // 256, topk)
    assert torch.equal(sel.cpu(), torch.tensor(chosen, dtype=torch.int32).expand(T // 256, topk))
    offs_h1 = np.array([0, T + 1], dtype=np.int32)
    with pytest.raises(V.jfa.JfaError, match="UNSUPPORTED"):
        V.jfa_topk_select(q, k, torch.from_numpy(offs_h1).cuda(), offs_h1, topk=topk)
