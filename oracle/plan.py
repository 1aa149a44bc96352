"""Naive restatement of the host tile planners -- TEST INFRASTRUCTURE ONLY.

The CUDA library plans its persistent kernels on the host (C++).  This module
states the same rules the slow, obvious way so that tests can compare the two
bit for bit.  Sources: the aixai.ru summary of "Optimizing Jagged Flash
Attention with TLX" (section on tile balancing and Cluster Launch Control) and
"TLX Block Attention" section 5 (scheduling variable-length sequences).

Forward (jagged): a unit is (b, h, m): 256 query rows [256m, 256m+256) of
sequence b and head h (two 128-row tiles sharing each K/V load).  Its cost is
the number of 128-key blocks it visits.  Units are sorted by cost, largest
first, keeping enumeration order (b, h, m ascending) among equal costs, and
dealt in snake order: pass p = t // P, slot r = t % P, CTA r on even passes and
P-1-r on odd passes.

Backward (jagged): a unit is (b, h, n), the n-th block of 128 keys of sequence b,
head h; only blocks that hold at least one key exist.  They are enumerated b
outer, h middle, n inner (units of one (b, h) run side by side and share the
same Q and dO in L2); their cost is the number of 128-row query tiles they
visit.  They are stably sorted by cost, largest first, and dealt in the same
snake order as the forward (with equal costs this is the enumeration order
dealt back and forth).

Block-diagonal: each sequence has ceil(L/64) blocks; BLOCK_PER_BATCH is their
exclusive prefix sum.  A tile is a pair of consecutive global blocks (2p, 2p+1)
for one head, tile id = pair * H + h.  P = min(n_sm, tiles) programs get
contiguous ranges by closed-form divmod: q, r = divmod(U, P), program p starts
at p*q + min(p, r).

Entries are int32 quadruples (b, h, m_or_n, cost); lists are CTA-major with a
[P+1] start array.
"""
from __future__ import annotations

FWD_ROWS = 256   # query rows per forward unit (two 128-row tiles)
KV_BLOCK = 128   # keys per K/V block
BLK = 64         # block-diagonal block size


def _cdiv(a, b):
    return -(-a // b)


def _visible(i, L, window):
    """Keys [lo, hi) that query i sees under window (left, right); None = open."""
    left, right = window
    lo = 0 if left is None else max(0, i - left)
    hi = L if right is None else min(L, i + right + 1)
    return lo, hi


def _window_fwd_cost(m, rows, L, window):
    # blocks from the first one any row of the unit sees to the last one
    first = min(_visible(r, L, window)[0] // KV_BLOCK for r in range(FWD_ROWS * m, min(FWD_ROWS * (m + 1), rows)))
    last = max((_visible(r, L, window)[1] - 1) // KV_BLOCK
               for r in range(FWD_ROWS * m, min(FWD_ROWS * (m + 1), rows)))
    return last - first + 1


def _window_bwd_cost(n, rows, L, window):
    # query tiles from the first one holding a row that sees some key of block n
    # to the last one; key k is seen by rows k-right .. k+left
    left, right = window
    keys = range(KV_BLOCK * n, min(KV_BLOCK * (n + 1), L))
    first = min((0 if right is None else max(0, k - right)) // KV_BLOCK for k in keys)
    last = max(((rows if left is None else min(rows, k + left + 1)) - 1) // KV_BLOCK for k in keys)
    return last - first + 1


def plan_fwd(offsets, num_heads, n_cta, *, causal=False, nq=0, window=None):
    """``window`` = (left, right), self-attention only: the unit's cost counts
    the K/V blocks its rows see inside the window."""
    B = len(offsets) - 1
    units = []
    for b in range(B):
        L = offsets[b + 1] - offsets[b]
        if L == 0:
            continue
        rows = nq if nq > 0 else L
        for h in range(num_heads):
            for m in range(_cdiv(rows, FWD_ROWS)):
                if window is not None:
                    cost = _window_fwd_cost(m, rows, L, window)
                elif causal:
                    last_row = min(FWD_ROWS * (m + 1), rows)
                    cost = _cdiv(min(last_row, L), KV_BLOCK)
                else:
                    cost = _cdiv(L, KV_BLOCK)
                units.append((b, h, m, cost))
    order = sorted(range(len(units)), key=lambda i: -units[i][3])  # Python sort is stable
    per_cta = [[] for _ in range(n_cta)]
    for t, i in enumerate(order):
        p, r = divmod(t, n_cta)
        cta = r if p % 2 == 0 else n_cta - 1 - r
        per_cta[cta].append(units[i])
    return _flatten(per_cta)


def plan_bwd(offsets, num_heads, n_cta, *, causal=False, nq=0, window=None):
    B = len(offsets) - 1
    units = []
    for b in range(B):
        L = offsets[b + 1] - offsets[b]
        rows = nq if nq > 0 else L
        for h in range(num_heads):
            for n in range(_cdiv(L, KV_BLOCK)):
                if window is not None:
                    cost = _window_bwd_cost(n, rows, L, window)
                elif causal:
                    cost = _cdiv(rows, FWD_ROWS // 2) - (KV_BLOCK * n) // (FWD_ROWS // 2)
                else:
                    cost = _cdiv(rows, FWD_ROWS // 2)
                units.append((b, h, n, cost))
    # stable sort by cost, largest first (a no-op when all costs are equal, as in
    # broadcast-Q), then the same snake deal as the forward
    order = sorted(range(len(units)), key=lambda i: -units[i][3])
    per_cta = [[] for _ in range(n_cta)]
    for t, i in enumerate(order):
        p, r = divmod(t, n_cta)
        cta = r if p % 2 == 0 else n_cta - 1 - r
        per_cta[cta].append(units[i])
    return _flatten(per_cta)


def plan_block(offsets, num_heads, n_sm):
    B = len(offsets) - 1
    bpb = [0]
    for b in range(B):
        L = offsets[b + 1] - offsets[b]
        bpb.append(bpb[-1] + _cdiv(L, BLK))
    n_blocks = bpb[-1]
    U = _cdiv(n_blocks, 2) * num_heads
    P = min(n_sm, U)
    starts = []
    if P > 0:
        q, r = divmod(U, P)
        starts = [p * q + min(p, r) for p in range(P + 1)]
    else:
        starts = [0]
    return bpb, starts


def _flatten(per_cta):
    starts = [0]
    flat = []
    for lst in per_cta:
        for e in lst:
            flat.extend(e)
        starts.append(starts[-1] + len(lst))
    return flat, starts
