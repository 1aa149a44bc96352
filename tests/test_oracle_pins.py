"""Pins for the fp64 oracle: it is checked against things other than itself.

- the offsets worked example printed on the pages (tests/golden/),
- textbook dense attention in matrix form (scipy softmax / logsumexp),
- closed forms (zero queries, equal values, single tokens),
- structural equalities (packed == per-piece, broadcast dQ == sum over pieces,
  block mode == jagged attention over 64-token pieces),
- central finite differences of the forward for every gradient,
- invariants (softmax rows sum to 1, keys' gradients sum to zero).
Each check is chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from tests.dense_ref import packed_dense
from variable_length_attention_gb300.workloads import offsets_from_lengths

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [int(x) for x in rest]
    return vals


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _problem(rng, lengths, H, Hkv, D, nq=0):
    offs = offsets_from_lengths(lengths)
    T = int(offs[-1])
    q = _rand(rng, nq if nq else T, H, D)
    k = _rand(rng, T, Hkv, D)
    v = _rand(rng, T, Hkv, D)
    rows = len(lengths) * nq if nq else T
    do = _rand(rng, rows, H, D)
    return offs, q, k, v, do


# --------------------------------------------------------------------------- offsets
@pytest.mark.parametrize("name", ["offsets_worked_example.txt", "offsets_tiny_workload.txt"])
def test_offsets_golden(name):
    g = _read_golden(name)
    offs = offsets_from_lengths(g["lengths"])
    assert offs.tolist() == g["offsets"]
    if "padded_slots" in g:
        assert len(g["lengths"]) * max(g["lengths"]) == g["padded_slots"][0]
        assert int(offs[-1]) == g["valid_tokens"][0]


# --------------------------------------------------------------------------- dense brute force
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv,D", [(2, 2, 4), (4, 2, 8), (4, 1, 8)])
def test_forward_matches_textbook_dense(causal, H, Hkv, D):
    rng = np.random.default_rng(11 + H + 7 * Hkv + D + int(causal))
    lengths = [3, 1, 9, 0, 6]
    offs, q, k, v, _ = _problem(rng, lengths, H, Hkv, D)
    scale = 1.0 / math.sqrt(D)
    o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=scale, causal=causal)
    o_ref, lse_ref = packed_dense(q, k, v, offs, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_broadcast_forward_matches_textbook_dense():
    rng = np.random.default_rng(5)
    lengths = [4, 0, 7, 1]
    offs, q, k, v, _ = _problem(rng, lengths, 2, 2, 8, nq=5)
    o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.3, nq=5)
    o_ref, lse_ref = packed_dense(q, k, v, offs, 0.3, nq=5)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)
    # empty sequence: zero output rows, log-sum-exp of nothing is -inf
    assert np.all(o[5:10] == 0.0) and np.all(lse[:, 5:10] == -np.inf)


# --------------------------------------------------------------------------- invariants / closed forms
def test_softmax_rows_sum_to_one():
    # With V = identity (D >= L) the output row is the softmax row itself.
    rng = np.random.default_rng(3)
    L, D = 7, 8
    offs = offsets_from_lengths([L])
    q = _rand(rng, L, 1, D) * 3
    k = _rand(rng, L, 1, D) * 3
    v = np.zeros((L, 1, D))
    v[np.arange(L), 0, np.arange(L)] = 1.0
    for causal in (False, True):
        o, _, _ = oracle.attn_fwd(q, k, v, offs, scale=0.5, causal=causal)
        p = o[:, 0, :L]
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        if causal:
            assert np.all(np.triu(p, 1) == 0.0)


def test_zero_queries_average_values():
    rng = np.random.default_rng(4)
    lengths = [5, 3]
    offs, q, k, v, _ = _problem(rng, lengths, 2, 2, 4)
    q[:] = 0.0
    o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=1.0)
    for b, (a, e) in enumerate(zip(offs[:-1], offs[1:])):
        np.testing.assert_allclose(o[a:e], np.broadcast_to(v[a:e].mean(axis=0), o[a:e].shape), atol=1e-14)
        np.testing.assert_allclose(lse[:, a:e], math.log(e - a), atol=1e-14)
    oc, lsec, _ = oracle.attn_fwd(q, k, v, offs, scale=1.0, causal=True)
    for a, e in zip(offs[:-1], offs[1:]):
        for i in range(e - a):
            np.testing.assert_allclose(oc[a + i], v[a:a + i + 1].mean(axis=0), atol=1e-14)
            np.testing.assert_allclose(lsec[:, a + i], math.log(i + 1), atol=1e-14)


def test_single_token_sequences():
    rng = np.random.default_rng(6)
    offs, q, k, v, do = _problem(rng, [1, 1, 1], 2, 2, 8)
    o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.7)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, 0.7 * np.einsum("thd,thd->ht", q, k), atol=1e-14)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.7)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_array_equal(dv, do)


def test_equal_values_rows():
    # All V rows equal c: O = c whatever P is, so dQ = dK = 0 and sum_j dV_j = sum_i dO_i.
    rng = np.random.default_rng(7)
    offs, q, k, v, do = _problem(rng, [6, 4], 2, 2, 4)
    c = rng.standard_normal(4)
    v[:] = c
    o, _, _ = oracle.attn_fwd(q, k, v, offs, scale=0.5)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), atol=1e-14)
    for causal in (False, True):
        dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.5, causal=causal)
        np.testing.assert_allclose(dq, 0, atol=1e-13)
        np.testing.assert_allclose(dk, 0, atol=1e-13)
        for a, e in zip(offs[:-1], offs[1:]):
            np.testing.assert_allclose(dv[a:e].sum(axis=0), do[a:e].sum(axis=0), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_keys_give_uniform_weights(causal):
    # All keys of a (sequence, kv head) equal: every score of a row is the same,
    # so P is uniform over the visible keys (O = mean of those V rows, LSE =
    # scale q.k + log(count)), and dQ_i = scale * (sum_j dS_ij) k = 0 because
    # each row of dS sums to zero (which needs Di = sum_j P_ij dP_ij exactly).
    rng = np.random.default_rng(12)
    offs, q, k, v, do = _problem(rng, [6, 1, 4], 4, 2, 8)
    for a, e in zip(offs[:-1], offs[1:]):
        k[a:e] = k[a]
    o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.6, causal=causal)
    dq, _, _, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.6, causal=causal)
    for a, e in zip(offs[:-1], offs[1:]):
        for i in range(e - a):
            n = i + 1 if causal else e - a
            for h in range(4):
                g = h // 2
                np.testing.assert_allclose(o[a + i, h], v[a:a + n, g].mean(axis=0), atol=1e-13)
                np.testing.assert_allclose(lse[h, a + i], 0.6 * q[a + i, h] @ k[a, g] + math.log(n), atol=1e-13)
    np.testing.assert_allclose(dq, 0, atol=1e-13)


def test_causal_boundary_rows():
    # Causal: the first query of a sequence sees only key 0, so its P is 1, its
    # dS is 0 and dQ_0 = 0; the last key is seen only by the last query, so
    # dV_last = P_last,last dO_last with P_last,last = exp(scale q.k - LSE) from
    # the forward's log-sum-exp.
    rng = np.random.default_rng(13)
    offs, q, k, v, do = _problem(rng, [5, 3, 7], 4, 2, 8)
    _, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.7, causal=True)
    dq, _, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.7, causal=True)
    for a, e in zip(offs[:-1], offs[1:]):
        np.testing.assert_allclose(dq[a], 0, atol=1e-14)
        last = e - 1
        for g in range(2):
            want = sum(math.exp(0.7 * q[last, h] @ k[last, g] - lse[h, last]) * do[last, h] for h in (2 * g, 2 * g + 1))
            np.testing.assert_allclose(dv[last, g], want, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_backward_equals_repeated_kv(causal):
    # Grouped-query attention is attention with each K/V head shared by its G
    # query heads: the grouped gradients equal those of the ungrouped problem on
    # K/V repeated per query head, with dK/dV summed over each group.
    rng = np.random.default_rng(14)
    offs, q, k, v, do = _problem(rng, [6, 2, 9], 6, 2, 4)
    g = oracle.attn_bwd(q, k, v, do, offs, scale=0.5, causal=causal)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    r = oracle.attn_bwd(q, kr, vr, do, offs, scale=0.5, causal=causal)
    np.testing.assert_allclose(g[0], r[0], atol=1e-13)
    for grouped, repeated in ((g[1], r[1]), (g[2], r[2])):
        np.testing.assert_allclose(grouped, repeated.reshape(-1, 2, 3, 4).sum(axis=2), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_gradients_sum_to_zero(causal):
    # Shifting every key of a sequence by the same vector leaves the softmax
    # unchanged, so the key gradients of each (sequence, kv head) sum to zero.
    rng = np.random.default_rng(8)
    offs, q, k, v, do = _problem(rng, [5, 9, 2], 4, 2, 8)
    _, dk, _, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.4, causal=causal)
    for a, e in zip(offs[:-1], offs[1:]):
        np.testing.assert_allclose(dk[a:e].sum(axis=0), 0, atol=1e-12)


# --------------------------------------------------------------------------- structure
def test_packed_equals_pieces():
    rng = np.random.default_rng(9)
    lengths = [3, 8, 5]
    offs, q, k, v, do = _problem(rng, lengths, 2, 1, 8)
    for causal in (False, True):
        o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.3, causal=causal)
        dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.3, causal=causal)
        for a, e in zip(offs[:-1], offs[1:]):
            one = np.array([0, e - a], dtype=np.int32)
            o1, l1, _ = oracle.attn_fwd(q[a:e], k[a:e], v[a:e], one, scale=0.3, causal=causal)
            g1 = oracle.attn_bwd(q[a:e], k[a:e], v[a:e], do[a:e], one, scale=0.3, causal=causal)
            np.testing.assert_array_equal(o[a:e], o1)
            np.testing.assert_array_equal(lse[:, a:e], l1)
            for full, piece in zip((dq, dk, dv), g1[:3]):
                np.testing.assert_array_equal(full[a:e], piece)


def test_broadcast_dq_is_sum_over_sequences():
    rng = np.random.default_rng(10)
    lengths = [6, 0, 3, 11]
    nq = 4
    offs, q, k, v, do = _problem(rng, lengths, 2, 2, 8, nq=nq)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.35, nq=nq)
    dq_sum = np.zeros_like(dq)
    for b, (a, e) in enumerate(zip(offs[:-1], offs[1:])):
        one = np.array([0, e - a], dtype=np.int32)
        g = oracle.attn_bwd(q, k[a:e], v[a:e], do[b * nq:(b + 1) * nq], one, scale=0.35, nq=nq)
        dq_sum += g[0]
        np.testing.assert_allclose(dk[a:e], g[1], atol=1e-14)
        np.testing.assert_allclose(dv[a:e], g[2], atol=1e-14)
    np.testing.assert_allclose(dq, dq_sum, rtol=0, atol=1e-12)


@pytest.mark.parametrize("lengths", [[64, 128, 192], [130, 64, 7]])
def test_block_mode_equals_jagged_over_blocks(lengths):
    rng = np.random.default_rng(12)
    offs, q, k, v, do = _problem(rng, lengths, 2, 2, 4)
    pieces = []
    for L in lengths:
        pieces += [64] * (L // 64) + ([L % 64] if L % 64 else [])
    offs64 = offsets_from_lengths(pieces)
    o_b, _ = oracle.block_fwd(q, k, v, offs, scale=0.5)
    o_j, _, _ = oracle.attn_fwd(q, k, v, offs64, scale=0.5)
    np.testing.assert_array_equal(o_b, o_j)
    g_b = oracle.block_bwd(q, k, v, do, offs, scale=0.5)
    g_j = oracle.attn_bwd(q, k, v, do, offs64, scale=0.5)
    for a, b in zip(g_b[:3], g_j[:3]):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    # and against the textbook form over the same pieces
    o_ref, _ = packed_dense(q, k, v, offs64, 0.5)
    np.testing.assert_allclose(o_b, o_ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- sliding window
WINDOWS = [(0, 0), (2, 0), (1, 3), (5, None), (None, 2), (3, 1)]


@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("H,Hkv", [(2, 2), (4, 2)])
def test_window_forward_matches_textbook_dense(window, H, Hkv):
    # query i sees keys i-left .. i+right of its own sequence: the textbook form
    # with that mask, on sequences shorter and longer than the window
    rng = np.random.default_rng(50 + H + Hkv)
    lengths = [3, 1, 9, 0, 7]
    offs, q, k, v, _ = _problem(rng, lengths, H, Hkv, 8)
    o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.45, window=window)
    o_ref, lse_ref = packed_dense(q, k, v, offs, 0.45, window=window)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_window_of_one_key_is_the_identity():
    # left = right = 0: every query sees only its own key, so P = 1, O = V,
    # LSE = scale q.k, dS = 0 (dQ = dK = 0) and dV = dO summed over the group
    rng = np.random.default_rng(51)
    offs, q, k, v, do = _problem(rng, [4, 1, 6], 4, 2, 8)
    o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.8, window=(0, 0))
    g = np.arange(4) // 2
    np.testing.assert_array_equal(o, v[:, g])
    np.testing.assert_allclose(lse, 0.8 * np.einsum("thd,thd->ht", q, k[:, g]), atol=1e-14)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.8, window=(0, 0))
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv, do.reshape(-1, 2, 2, 8).sum(axis=2), atol=1e-14)


def test_wide_window_is_full_and_causal_window_is_causal():
    rng = np.random.default_rng(52)
    offs, q, k, v, do = _problem(rng, [5, 9, 2], 2, 1, 4)
    for causal, window in ((False, (9, 9)), (True, (9, None)), (False, (9, 0))):
        want_causal = causal or window[1] == 0
        o, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.5, causal=causal, window=window)
        o0, lse0, _ = oracle.attn_fwd(q, k, v, offs, scale=0.5, causal=want_causal)
        np.testing.assert_array_equal(o, o0)
        np.testing.assert_array_equal(lse, lse0)
        g = oracle.attn_bwd(q, k, v, do, offs, scale=0.5, causal=causal, window=window)
        g0 = oracle.attn_bwd(q, k, v, do, offs, scale=0.5, causal=want_causal)
        for a, b in zip(g[:3], g0[:3]):
            np.testing.assert_array_equal(a, b)


def test_window_edge_rows():
    # With a window of `left` keys to the left and none to the right, the key
    # gradient of key j collects queries j .. j+left only, so for a sequence
    # longer than the window the first key's dV is the sum over queries
    # 0 .. left of P_i0 dO_i, with P from the forward's log-sum-exp.
    rng = np.random.default_rng(53)
    left = 2
    offs, q, k, v, do = _problem(rng, [8], 1, 1, 4)
    _, lse, _ = oracle.attn_fwd(q, k, v, offs, scale=0.7, window=(left, 0))
    _, _, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.7, window=(left, 0))
    want = sum(math.exp(0.7 * q[i, 0] @ k[0, 0] - lse[0, i]) * do[i, 0] for i in range(left + 1))
    np.testing.assert_allclose(dv[0, 0], want, atol=1e-13)


# --------------------------------------------------------------------------- finite differences
def _loss(fwd, x_name, x, base, h_idx, eps, dout):
    args = dict(base)
    xp = x.copy()
    xp[h_idx] += eps
    args[x_name] = xp
    op = fwd(**args)
    xm = x.copy()
    xm[h_idx] -= eps
    args[x_name] = xm
    om = fwd(**args)
    return float(np.sum((op - om) * dout)) / (2 * eps)


def _check_fd(fwd, bwd_grads, base, dout, rng, n_probe=12, eps=1e-5):
    for name, g in zip(("q", "k", "v"), bwd_grads):
        x = base[name]
        for _ in range(n_probe):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            fd = _loss(fwd, name, x, base, idx, eps, dout)
            assert abs(fd - g[idx]) <= 1e-7 + 1e-6 * abs(fd), (name, idx, fd, g[idx])


@pytest.mark.parametrize("causal,H,Hkv", [(False, 2, 2), (True, 2, 2), (False, 4, 2), (True, 4, 1)])
def test_gradients_finite_differences(causal, H, Hkv):
    rng = np.random.default_rng(20 + H + Hkv + int(causal))
    offs, q, k, v, do = _problem(rng, [4, 7, 1], H, Hkv, 4)
    scale = 0.6

    def fwd(q, k, v):
        return oracle.attn_fwd(q, k, v, offs, scale=scale, causal=causal)[0]

    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=scale, causal=causal)
    _check_fd(fwd, (dq, dk, dv), dict(q=q, k=k, v=v), do, rng)


@pytest.mark.parametrize("window,H,Hkv", [((1, 0), 2, 2), ((2, 1), 4, 2), ((None, 1), 2, 1), ((3, None), 2, 2)])
def test_window_gradients_finite_differences(window, H, Hkv):
    rng = np.random.default_rng(60 + H + Hkv)
    offs, q, k, v, do = _problem(rng, [5, 7, 1], H, Hkv, 4)

    def fwd(q, k, v):
        return oracle.attn_fwd(q, k, v, offs, scale=0.6, window=window)[0]

    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.6, window=window)
    _check_fd(fwd, (dq, dk, dv), dict(q=q, k=k, v=v), do, rng)


@pytest.mark.parametrize("H,Hkv,lengths", [(2, 2, [4, 2, 5]), (4, 2, [4, 0, 5]), (4, 1, [3, 6])])
def test_broadcast_gradients_finite_differences(H, Hkv, lengths):
    # grouped heads: dK/dV of a key/value head collect every query head of its
    # group and every query row; dQ of the shared Q every sequence
    rng = np.random.default_rng(30 + H + Hkv)
    nq = 3
    offs, q, k, v, do = _problem(rng, lengths, H, Hkv, 4, nq=nq)

    def fwd(q, k, v):
        return oracle.attn_fwd(q, k, v, offs, scale=0.5, nq=nq)[0]

    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, offs, scale=0.5, nq=nq)
    _check_fd(fwd, (dq, dk, dv), dict(q=q, k=k, v=v), do, rng)


def test_block_gradients_finite_differences():
    rng = np.random.default_rng(31)
    offs, q, k, v, do = _problem(rng, [70, 5], 1, 1, 4)

    def fwd(q, k, v):
        return oracle.block_fwd(q, k, v, offs, scale=0.5)[0]

    dq, dk, dv, _ = oracle.block_bwd(q, k, v, do, offs, scale=0.5)
    _check_fd(fwd, (dq, dk, dv), dict(q=q, k=k, v=v), do, rng, n_probe=20)


def test_unit_selection_and_threads():
    rng = np.random.default_rng(40)
    offs, q, k, v, do = _problem(rng, [9, 4, 12], 2, 2, 8)
    sel = np.zeros((3, 2), dtype=bool)
    sel[1, 0] = sel[2, 1] = True
    o_all, lse_all, _ = oracle.attn_fwd(q, k, v, offs, scale=0.4, nthreads=1)
    o_sel, lse_sel, _ = oracle.attn_fwd(q, k, v, offs, scale=0.4, sel=sel, nthreads=3)
    for b in range(3):
        a, e = offs[b], offs[b + 1]
        for h in range(2):
            if sel[b, h]:
                np.testing.assert_array_equal(o_sel[a:e, h], o_all[a:e, h])
            else:
                assert np.all(np.isnan(o_sel[a:e, h]))


# --------------------------------------------------------------------------- rotary embedding (block attention)
def _rope_pins(rope_fn):
    """The rotary pins, parameterised by the rotation so that planted mistakes
    in it can be shown to fail them (tests/test_oracle_mutants.py)."""
    rng = np.random.default_rng(70)
    # closed form, D = 4: the pair (x0, x2) turns by pos, (x1, x3) by pos * base^(-1/2)
    base = 100.0
    offs = offsets_from_lengths([3, 5])
    x = rng.standard_normal((8, 1, 4))
    y = rope_fn(x, offs, base)
    for r in range(8):
        pos = r if r < 3 else r - 3
        for i, ang in ((0, pos * 1.0), (1, pos * base ** -0.5)):
            c, s = math.cos(ang), math.sin(ang)
            a, b = x[r, 0, i], x[r, 0, i + 2]
            assert abs(y[r, 0, i] - (a * c - b * s)) < 1e-14
            assert abs(y[r, 0, i + 2] - (b * c + a * s)) < 1e-14
    # the transposed rotation undoes it; every pair keeps its length
    x = rng.standard_normal((20, 3, 8))
    offs = offsets_from_lengths([7, 13])
    y = rope_fn(x, offs, 10000.0)
    np.testing.assert_allclose(rope_fn(y, offs, 10000.0, transpose=True), x, atol=1e-13)
    np.testing.assert_allclose(y[..., :4] ** 2 + y[..., 4:] ** 2, x[..., :4] ** 2 + x[..., 4:] ** 2, atol=1e-13)
    # scores of rotated rows depend on the positions only through their
    # difference: equal raw rows give a Toeplitz score matrix in every sequence
    L, D = 9, 8
    offs = offsets_from_lengths([L, L])
    a, b = rng.standard_normal(D), rng.standard_normal(D)
    q = np.broadcast_to(a, (2 * L, 1, D)).copy()
    k = np.broadcast_to(b, (2 * L, 1, D)).copy()
    sc = rope_fn(q, offs, 50.0)[:, 0] @ rope_fn(k, offs, 50.0)[:, 0].T
    for m in range(1, L):
        for n in range(1, L):
            assert abs(sc[m, n] - sc[m - 1, n - 1]) < 1e-12
    # positions restart in every sequence
    np.testing.assert_allclose(sc[:L, :L], sc[L:, L:], atol=1e-13)
    np.testing.assert_allclose(sc[0, 0], a @ b, atol=1e-13)


def test_rope_pins():
    _rope_pins(oracle.rope)


def test_rope_block_attention_finite_differences():
    # gradients of rotary block attention with respect to the unrotated Q, K
    # (the rotation's transpose carries them back) and V
    rng = np.random.default_rng(71)
    offs, q, k, v, do = _problem(rng, [70, 5], 1, 1, 4)

    def fwd(q, k, v):
        return oracle.block_fwd(q, k, v, offs, scale=0.5, rope_base=30.0)[0]

    dq, dk, dv, _ = oracle.block_bwd(q, k, v, do, offs, scale=0.5, rope_base=30.0)
    _check_fd(fwd, (dq, dk, dv), dict(q=q, k=k, v=v), do, rng, n_probe=20)


def test_rope_block_attention_is_attention_of_rotated_rows():
    # sequences of at most one 64-token block: rotary block attention is the
    # textbook attention of the rotated Q and K rows of each sequence
    rng = np.random.default_rng(72)
    offs, q, k, v, _ = _problem(rng, [64, 30], 2, 2, 8)
    o, _ = oracle.block_fwd(q, k, v, offs, scale=0.4, rope_base=1e4)
    o_ref, _ = packed_dense(oracle.rope(q, offs, 1e4), oracle.rope(k, offs, 1e4), v, offs, 0.4)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)


# --------------------------------------------------------------------------- two-stage block-sparse forward
def _topk_pins(ns):
    """The top-k pins, parameterised by the three stage functions (``ns`` has
    topk_scores, topk_select, attn_fwd_topk) so that planted mistakes in them
    can be shown to fail them (tests/test_oracle_mutants.py)."""
    rng = np.random.default_rng(80)
    # closed form of the scores: every row of query block m equal to a_m, every
    # key of key block n (the short tail block too) equal to c_n; grouped heads
    L, H, Hkv, D = 300, 4, 2, 8
    offs = offsets_from_lengths([L, 129])
    a = rng.standard_normal((2, H, D))
    c = rng.standard_normal((3, Hkv, D))
    q = np.zeros((L + 129, H, D))
    k = np.zeros((L + 129, Hkv, D))
    for r in range(L):
        q[r] = a[r // 256]
        k[r] = c[r // 128]
    q[L:] = rng.standard_normal((129, H, D))
    k[L:] = rng.standard_normal((129, Hkv, D))
    sc = ns.topk_scores(q, k, offs)
    # order b, h, m: sequence 0 has 2 query blocks per head, sequence 1 has 1
    assert len(sc) == H * 2 + H * 1
    for h in range(H):
        for m in range(2):
            want = [a[m, h] @ c[n, h // 2] for n in range(3)]
            np.testing.assert_allclose(sc[h * 2 + m], want, atol=1e-12)
    # selection: the k highest, ties to the lower index, ascending
    sel = ns.topk_select([np.array([0.1, 0.9, -0.5, 0.9, 0.3])], 2)
    assert sel == [[1, 3]]
    assert ns.topk_select([np.array([0.5, 0.2, 0.5, 0.5])], 2) == [[0, 2]]
    assert ns.topk_select([np.array([3.0, 1.0])], 5) == [[0, 1]]
    # every block chosen: exact attention
    offs = offsets_from_lengths([300, 40, 513])
    q = rng.standard_normal((853, 2, 8))
    k = rng.standard_normal((853, 2, 8))
    v = rng.standard_normal((853, 2, 8))
    sel = ns.topk_select(ns.topk_scores(q, k, offs), 99)
    o, lse = ns.attn_fwd_topk(q, k, v, offs, sel, scale=0.4)
    o_ref, lse_ref, _ = oracle.attn_fwd(q, k, v, offs, scale=0.4)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)
    # one chosen block: textbook attention over that block's keys, per query
    # block of 256 rows (rows 0..255 and 256..299 of sequence 0 choose
    # different blocks here)
    # units of sequence 0: (h0, m0), (h0, m1), (h1, m0), (h1, m1); then sequence 1
    # (one query block per head) and sequence 2 (three per head)
    sel1 = [[2], [0], [2], [0]] + [[0]] * 2 + [[1], [3], [4], [1], [3], [4]]
    assert len(sel1) == len(sel)
    o1, _ = ns.attn_fwd_topk(q, k, v, offs, sel1, scale=0.4)
    for h in range(2):
        s = 0.4 * q[0:256, h] @ k[256:300, h].T
        p = np.exp(s - s.max(axis=1, keepdims=True))
        np.testing.assert_allclose(o1[0:256, h], (p / p.sum(axis=1, keepdims=True)) @ v[256:300, h], atol=1e-12)
        s = 0.4 * q[256:300, h] @ k[0:128, h].T
        p = np.exp(s - s.max(axis=1, keepdims=True))
        np.testing.assert_allclose(o1[256:300, h], (p / p.sum(axis=1, keepdims=True)) @ v[0:128, h], atol=1e-12)
    # broadcast-Q: query blocks of the shared Q against each sequence, an empty
    # sequence has none; every block chosen is exact broadcast attention
    offs = offsets_from_lengths([200, 0, 390])
    qs = rng.standard_normal((300, 2, 8))
    k = rng.standard_normal((590, 2, 8))
    v = rng.standard_normal((590, 2, 8))
    sel = ns.topk_select(ns.topk_scores(qs, k, offs, nq=300), 99)
    assert len(sel) == 2 * 2 * 2  # 2 sequences with keys x 2 heads x 2 query blocks
    o, lse = ns.attn_fwd_topk(qs, k, v, offs, sel, scale=0.3, nq=300)
    o_ref, lse_ref, _ = oracle.attn_fwd(qs, k, v, offs, scale=0.3, nq=300)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    assert np.array_equal(np.isinf(lse), np.isinf(lse_ref))


def test_topk_pins():
    _topk_pins(oracle)
