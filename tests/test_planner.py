"""Host planners of libjfa, bit for bit against the naive restatement in
oracle/plan.py, plus structural invariants (every valid unit exactly once,
snake order, closed-form ranges).  CPU only: the planners are host code."""
import numpy as np
import pytest

import variable_length_attention_gb300 as V
from oracle import plan as P
from variable_length_attention_gb300 import workloads as W
from variable_length_attention_gb300.workloads import offsets_from_lengths


def _cases():
    rng = np.random.default_rng(0)
    cases = [("tiny", W.tiny()), ("jagged", W.jagged(False)), ("jagged_causal", W.jagged(True)),
             ("broadcast", W.broadcast()), ("dense", W.dense())]
    for i in range(4):
        L = rng.integers(0, 1500, size=int(rng.integers(1, 40)))
        L[rng.random(len(L)) < 0.2] = 0
        cases.append((f"random{i}", W.custom(L, int(rng.integers(1, 6)), 64, causal=bool(i % 2))))
    cases.append(("random_bcast", W.custom(rng.integers(0, 900, size=30), 3, 64, nq=300)))
    return cases


CASES = _cases()


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("n_cta", [1, 7, 148, 152])
def test_fwd_plan_bit_exact(name, w, n_cta):
    offs = w.offsets.tolist()
    u, s = V.jfa_plan_fwd(offs, w.num_heads, n_cta, nq=w.nq, causal=w.causal)
    fu, fs = P.plan_fwd(offs, w.num_heads, n_cta, causal=w.causal, nq=w.nq)
    assert u.tolist() == fu and s.tolist() == fs


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("n_cta", [1, 7, 148, 152])
def test_bwd_plan_bit_exact(name, w, n_cta):
    offs = w.offsets.tolist()
    u, s = V.jfa_plan_bwd(offs, w.num_heads, n_cta, nq=w.nq, causal=w.causal)
    fu, fs = P.plan_bwd(offs, w.num_heads, n_cta, causal=w.causal, nq=w.nq)
    assert u.tolist() == fu and s.tolist() == fs


WINDOW_CASES = [(w, win) for w in (W.tiny(), W.jagged(False), CASES[5][1], CASES[6][1])
                for win in ((0, 0), (127, 0), (255, 0), (300, 40), (None, 129), (1000, None), (None, 0))]


@pytest.mark.parametrize("w,window", WINDOW_CASES, ids=[f"{w.name}-{win}" for w, win in WINDOW_CASES])
def test_window_plans_bit_exact(w, window):
    # under a window the costs count the blocks / tiles the unit's rows or keys
    # see; the entries and their order follow the same rules as without one
    if w.nq:
        pytest.skip("windows are for self-attention")
    offs = w.offsets.tolist()
    for which, n_cta in ((0, 152), (0, 7), (1, 152), (1, 1)):
        u, s = V.jfa_plan_window(which, offs, w.num_heads, n_cta, window)
        fn = P.plan_fwd if which == 0 else P.plan_bwd
        fu, fs = fn(offs, w.num_heads, n_cta, window=window)
        assert u.tolist() == fu and s.tolist() == fs
    if window == (None, 0):  # the causal window is causal attention
        assert V.jfa_plan_window(0, offs, w.num_heads, 152, window)[0].tolist() == \
            V.jfa_plan_fwd(offs, w.num_heads, 152, causal=True)[0].tolist()
        assert V.jfa_plan_window(1, offs, w.num_heads, 152, window)[0].tolist() == \
            V.jfa_plan_bwd(offs, w.num_heads, 152, causal=True)[0].tolist()


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_fwd_plan_covers_every_query_row_once(name, w):
    offs = w.offsets
    u, s = V.jfa_plan_fwd(offs, w.num_heads, 148, nq=w.nq, causal=w.causal)
    units = u.reshape(-1, 4)
    seen = set()
    for b, h, m, cost in units:
        assert (b, h, m) not in seen
        seen.add((b, h, m))
        L = offs[b + 1] - offs[b]
        rows = w.nq or L
        assert L > 0 and 0 <= 256 * m < rows
        n_kv = -(-min(256 * (m + 1), rows, L) // 128) if w.causal else -(-L // 128)
        assert cost == n_kv
    expected = sum(w.num_heads * -(-(w.nq or (offs[b + 1] - offs[b])) // 256)
                   for b in range(w.batch) if offs[b + 1] > offs[b])
    assert len(seen) == expected
    # snake deal: costs, read in sorted order, are non-increasing
    assert np.all(np.diff(s) >= 0) and s[0] == 0 and s[-1] == len(units)


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_bwd_plan_lists_only_valid_blocks(name, w):
    offs = w.offsets
    u, s = V.jfa_plan_bwd(offs, w.num_heads, 148, nq=w.nq, causal=w.causal)
    units = u.reshape(-1, 4)
    keys = {(b, h, n) for b, h, n, _ in units}
    assert len(keys) == len(units)
    expected = {(b, h, n) for b in range(w.batch) for h in range(w.num_heads)
                for n in range(-(-(offs[b + 1] - offs[b]) // 128))}
    assert keys == expected


def test_snake_deal_formula():
    # 10 equal-cost units over 4 CTAs: passes 0..2, CTA order 0123 3210 01
    offs = [0, 1280]
    u, s = V.jfa_plan_bwd(offs, 1, 4)
    units = u.reshape(-1, 4)
    per_cta = [units[s[c]:s[c + 1], 2].tolist() for c in range(4)]
    assert per_cta == [[0, 7, 8], [1, 6, 9], [2, 5], [3, 4]]


@pytest.mark.parametrize("lengths,H,n_sm", [([4032] * 1152, 4, 148), ([64, 1, 130, 0, 7], 3, 4),
                                            ([100] * 3, 2, 152), ([0, 0], 2, 8)])
def test_block_plan(lengths, H, n_sm):
    offs = offsets_from_lengths(lengths)
    bpb, ps = V.block_plan(offs, H, n_sm)
    fb, fs = P.plan_block(offs.tolist(), H, n_sm)
    assert bpb.tolist() == fb and ps.tolist() == fs
    tiles = -(-bpb[-1] // 2) * H
    assert ps[-1] == tiles
    if tiles:
        sizes = np.diff(ps)
        assert sizes.max() - sizes.min() <= 1   # balanced contiguous ranges


def test_worked_example_block_prefix():
    # 1152 sequences of 4032 tokens = 63 blocks of 64 each
    offs = offsets_from_lengths([4032] * 1152)
    bpb, ps = V.block_plan(offs, 4, 148)
    assert bpb[1] == 63 and bpb[-1] == 1152 * 63
    assert ps[-1] == (1152 * 63 + 1) // 2 * 4


def _balance(per_cta):
    per_cta = np.asarray(per_cta, dtype=np.float64)
    return per_cta.mean() / per_cta.max()


@pytest.mark.parametrize("w,fwd_min,bwd_min", [(W.jagged(False), 0.90, 0.95), (W.jagged(True), 0.90, 0.95),
                                               (W.broadcast(), 0.85, 0.99), (W.dense(), 0.99, 0.99)],
                         ids=["jagged", "jagged_causal", "broadcast", "dense"])
def test_static_plans_balance_cost(w, fwd_min, bwd_min):
    # per-CTA summed unit cost over 152 CTAs (mean / max; 1 = perfect), and the
    # backward's sorted snake deal against plain round-robin in enumeration order
    for fn, lo in ((V.jfa_plan_fwd, fwd_min), (V.jfa_plan_bwd, bwd_min)):
        u, s = fn(w.offsets, w.num_heads, 152, nq=w.nq, causal=w.causal)
        units = u.reshape(-1, 4)
        cost = units[:, 3].astype(np.int64)
        snake = _balance([cost[s[c]:s[c + 1]].sum() for c in range(len(s) - 1)])
        assert snake >= lo, (fn.__name__, snake)
        if fn is V.jfa_plan_bwd:
            order = np.lexsort((units[:, 2], units[:, 1], units[:, 0]))  # enumeration order b, h, n
            rr = np.zeros(152, dtype=np.int64)
            np.add.at(rr, np.arange(len(order)) % 152, cost[order])
            assert snake >= _balance(rr) - 1e-12
