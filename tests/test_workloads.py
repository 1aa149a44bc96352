"""The seeded input recipe and the FLOP count the metric is quoted in.  CPU only.

The generators are the one module both the oracle and the CUDA path read, so
their recipe (lengths, seeds, shapes, value distribution) is checked here, and
the valid-pair count behind every TFLOP/s figure is checked against brute-force
enumeration of the (query, key) pairs each mode scores.
"""
import math

import numpy as np
import pytest
import torch

from variable_length_attention_gb300 import workloads as W


def test_offsets_are_an_exclusive_prefix_sum():
    offs = W.offsets_from_lengths([128, 4096, 512, 2048])
    assert offs.dtype == np.int32 and offs.tolist() == [0, 128, 4224, 4736, 6784]
    assert W.offsets_from_lengths([]).tolist() == [0]
    with pytest.raises(ValueError):
        W.offsets_from_lengths([2**30, 2**30])


def test_jagged_lengths_recipe():
    a, b = W.jagged(False), W.jagged(True)
    assert np.array_equal(a.lengths, b.lengths)           # the causal variant shares the lengths
    assert np.array_equal(a.lengths, W.jagged(False).lengths)  # seeded
    assert a.batch == 32 and a.num_heads == 8 and a.head_dim == 128
    assert a.lengths.min() >= 32 and a.lengths.max() <= 4096
    # log-uniform on [32, 4096]: ln L is uniform with mean (ln 32 + ln 4096) / 2
    mean_log = np.mean(np.log(a.lengths))
    assert abs(mean_log - 0.5 * (math.log(32) + math.log(4096))) < 0.5


def test_broadcast_lengths_recipe():
    w = W.broadcast()
    assert w.batch == 256 and w.nq == 256 and w.num_heads == 4 and w.head_dim == 128
    assert w.lengths.min() >= 16 and w.lengths.max() <= 4000
    assert 600 <= np.median(w.lengths) <= 1050               # log-normal around a median of 800
    assert abs(np.std(np.log(w.lengths)) - 1.0) < 0.2        # sigma 1 in log space (before clipping)
    assert w.q_rows == 256 and w.o_rows == 256 * 256


def test_fixed_shapes():
    t = W.tiny()
    assert t.lengths.tolist() == [17, 64, 129, 256] and (t.num_heads, t.head_dim) == (2, 64)
    blk = W.block(128)
    assert blk.batch == 1152 and set(blk.lengths.tolist()) == {4032} and blk.num_heads == 4
    d, g = W.dense(False), W.dense(True)
    assert d.lengths.tolist() == [8192] * 8 and d.num_heads == 16 and d.num_kv_heads == 16
    assert g.num_kv_heads == 4 and not g.bwd


def test_tensors_are_seeded_bf16_normal():
    w = W.custom([300, 77, 5], 4, 64, num_kv_heads=2, seed_base=123)
    q, k, v, do = w.tensors("cpu")
    assert q.shape == (382, 4, 64) and k.shape == v.shape == (382, 2, 64) and do.shape == (382, 4, 64)
    assert all(t.dtype == torch.bfloat16 for t in (q, k, v, do))
    again = w.tensors("cpu")
    assert all(torch.equal(x, y) for x, y in zip((q, k, v, do), again))
    assert not torch.equal(k, v)                              # each tensor has its own seed
    x = torch.cat([t.float().reshape(-1) for t in (q, k, v, do)])
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1.0) < 0.02
    b = W.custom([10, 0, 3], 2, 64, nq=7, seed_base=5)
    qb, kb, _, dob = b.tensors("cpu")
    assert qb.shape == (7, 2, 64) and kb.shape == (13, 2, 64) and dob.shape == (21, 2, 64)


def _pairs_brute(w):
    n = 0
    for L in w.lengths.tolist():
        if w.mode == "broadcast":
            n += sum(1 for _ in range(w.nq) for _ in range(L))
        elif w.mode == "block":
            for i in range(L):
                start = (i // 64) * 64
                n += min(start + 64, L) - start
        else:
            n += sum((i + 1) if w.causal else L for i in range(L))
    return n * w.num_heads


@pytest.mark.parametrize("w", [W.custom([1, 17, 64, 129, 300], 3, 64),
                               W.custom([1, 17, 64, 129, 300], 3, 64, causal=True),
                               W.custom([5, 0, 130, 70], 2, 128, nq=33),
                               W.custom([64, 65, 127, 200, 3], 4, 64, mode="block")],
                         ids=["jagged", "causal", "broadcast", "block"])
def test_flop_count_matches_enumeration(w):
    pairs = _pairs_brute(w)
    assert W.valid_pairs(w) == pairs
    f, b = W.flops(w)
    assert f == 4 * w.head_dim * pairs and b == int(2.5 * f)
