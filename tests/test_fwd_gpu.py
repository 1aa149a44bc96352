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


def test_dense_full_size():
    # the dense-equivalent stress shape (B=8 x 8192, H=16, D=128): O and LSE of a
    # seeded sample of 10 (sequence, head) units, sequences 0 and 7 among them
    w = W.dense(gqa=False)
    sel = sample_units(w.batch, w.num_heads, 8, seed=14)
    assert sel[0].any() and sel[w.batch - 1].any() and sel.sum() >= 8
    res, _ = check_fwd(w, sel=sel)
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


@pytest.mark.parametrize("causal", [False, True])
def test_running_max_growth(causal):
    """Scores that climb along the keys, for some rows and not others: the running
    maximum of those rows grows by more than 2^8 several times, so the O rescale
    path runs, with rows of one warp taking different decisions ("TLX Block
    Attention", section 2.1: the correction factor when m grows)."""
    import oracle
    from tests.parity import rel_l2, to64
    lengths = [700, 300, 129]
    H, D = 2, 64
    offs_h = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(offs_h[-1])
    g = torch.Generator().manual_seed(4242 + int(causal))
    q = torch.randn(T, H, D, generator=g)
    k = torch.randn(T, H, D, generator=g)
    v = torch.randn(T, H, D, generator=g)
    q[:, :, 0] = torch.where(torch.arange(T) % 2 == 0, 3.0, 0.0)[:, None]  # every other row climbs
    for b in range(len(lengths)):
        j = torch.arange(lengths[b], dtype=torch.float32)
        k[offs_h[b]:offs_h[b + 1], :, 0] = (0.07 * j)[:, None]
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = 1.0 / np.sqrt(D)
    offs = torch.from_numpy(offs_h).cuda()
    o, lse = V.jfa_fwd(q.cuda(), k.cuda(), v.cuda(), offs, offs_h, causal=causal, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref, _ = oracle.attn_fwd(to64(q), to64(k), to64(v), offs_h, scale=scale, causal=causal)
    o_g, lse_g = to64(o), to64(lse)
    res = {"o_max_abs": float(np.max(np.abs(o_g - o_ref))), "o_rel_l2": rel_l2(o_g, o_ref),
           "lse_max_abs": float(np.max(np.abs(lse_g - lse_ref))), "lse_inf_match": True,
           "finite": bool(np.all(np.isfinite(o_g)))}
    # the growth is real: for a climbing row near the end of the first sequence, the
    # maximum over all its keys exceeds the first block's by more than two steps of 2^8
    s_row = to64(k[:lengths[0] - 1, 0]) @ to64(q[lengths[0] - 2, 0]) * scale
    assert (s_row.max() - s_row[:128].max()) * np.log2(np.e) > 16.0
    assert_fwd_ok(res)
