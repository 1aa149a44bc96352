"""Helpers shared by the GPU parity tests: run a workload through the CUDA
library and the fp64 oracle on the same seeded bf16 inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import variable_length_attention_gb300 as V

# Tolerances (bf16 inputs, fp32 accumulation, bf16 outputs):
O_MAX_ABS = 1e-2       # output, max |gpu - oracle|
O_REL_L2 = 5e-3        # output, ||gpu - oracle|| / ||oracle||
LSE_MAX_ABS = 2e-3     # log-sum-exp, max abs
GRAD_REL_L2 = 2e-2     # dQ, dK, dV relative L2


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))


def to64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def sample_units(batch, H, n, seed=0):
    """A [batch, H] selection of at least n (sequence, head) units drawn from a
    seed, always including the first sequence's head 0 and the last sequence's
    last head (the two ends of the packed tensors)."""
    rng = np.random.default_rng(seed)
    sel = np.zeros((batch, H), dtype=bool)
    flat = rng.choice(batch * H, size=min(n, batch * H), replace=False)
    sel.reshape(-1)[flat] = True
    if batch > 0:
        sel[0, 0] = True
        sel[batch - 1, H - 1] = True
    return sel


def rows_of(offsets, sel, H, nq=0):
    """Boolean [rows, H] mask of output rows covered by a unit selection."""
    B = len(offsets) - 1
    rows = B * nq if nq else int(offsets[-1])
    mask = np.zeros((rows, H), dtype=bool)
    for b in range(B):
        a, e = (b * nq, (b + 1) * nq) if nq else (int(offsets[b]), int(offsets[b + 1]))
        mask[a:e] = sel[b][None, :]
    return mask


def gpu_inputs(w, device="cuda"):
    q, k, v, do = w.tensors("cpu")
    offs = torch.from_numpy(w.offsets).to(device)
    return [t.to(device) for t in (q, k, v, do)], offs, (q, k, v, do)


def check_fwd(w, sel=None, nthreads=0, window=None):
    """Runs jfa_fwd (jfa_fwd_window if ``window`` is given) and compares O and
    LSE with the oracle.  Returns a dict of errors."""
    (q, k, v, do), offs, cpu = gpu_inputs(w)
    o, lse = V.jfa_fwd(q, k, v, offs, w.offsets, causal=w.causal, nq_broadcast=w.nq, scale=w.scale, window=window)
    torch.cuda.synchronize()
    o_ref, lse_ref, _ = oracle.attn_fwd(to64(cpu[0]), to64(cpu[1]), to64(cpu[2]), w.offsets, scale=w.scale,
                                        causal=w.causal, nq=w.nq, sel=sel, nthreads=nthreads, window=window)
    o_g, lse_g = to64(o), to64(lse)
    if sel is not None:
        m = rows_of(w.offsets, sel, w.num_heads, w.nq)
        o_g, o_ref = o_g[m], o_ref[m]
        lse_g, lse_ref = lse_g.T[m], lse_ref.T[m]
    fin = np.isfinite(lse_ref)
    res = {
        "o_max_abs": float(np.max(np.abs(o_g - o_ref))) if o_g.size else 0.0,
        "o_rel_l2": rel_l2(o_g, o_ref),
        "lse_max_abs": float(np.max(np.abs(lse_g[fin] - lse_ref[fin]))) if fin.any() else 0.0,
        "lse_inf_match": bool(np.all(np.isneginf(lse_g[~fin]))) if (~fin).any() else True,
        "finite": bool(np.all(np.isfinite(o_g))),
    }
    return res, (o, lse)


def assert_fwd_ok(res):
    assert res["finite"], res
    assert res["o_max_abs"] <= O_MAX_ABS, res
    assert res["o_rel_l2"] <= O_REL_L2, res
    assert res["lse_max_abs"] <= LSE_MAX_ABS, res
    assert res["lse_inf_match"], res


def kv_rows_of(offsets, sel, H):
    """Boolean [kv_rows, H] mask of key rows covered by a unit selection."""
    B = len(offsets) - 1
    mask = np.zeros((int(offsets[-1]), H), dtype=bool)
    for b in range(B):
        mask[int(offsets[b]):int(offsets[b + 1])] = sel[b][None, :]
    return mask


def check_bwd(w, sel=None, nthreads=0, window=None):
    """Runs jfa_fwd then jfa_bwd on the GPU (the window entry points if ``window``
    is given) and compares dQ, dK, dV with the oracle."""
    (q, k, v, do), offs, cpu = gpu_inputs(w)
    o, lse = V.jfa_fwd(q, k, v, offs, w.offsets, causal=w.causal, nq_broadcast=w.nq, scale=w.scale, window=window)
    dq, dk, dv = V.jfa_bwd(q, k, v, o, do, lse, offs, w.offsets, causal=w.causal, nq_broadcast=w.nq,
                           scale=w.scale, window=window)
    torch.cuda.synchronize()
    ref = oracle.attn_bwd(to64(cpu[0]), to64(cpu[1]), to64(cpu[2]), to64(cpu[3]), w.offsets, scale=w.scale,
                          causal=w.causal, nq=w.nq, sel=sel, nthreads=nthreads, window=window)
    got = [to64(dq), to64(dk), to64(dv)]
    want = list(ref[:3])
    if sel is not None:
        mq = rows_of(w.offsets, sel, w.num_heads) if not w.nq else np.ones(got[0].shape[:2], bool)
        mk = kv_rows_of(w.offsets, sel, w.num_heads)
        got = [got[0][mq], got[1][mk], got[2][mk]]
        want = [want[0][mq], want[1][mk], want[2][mk]]
    res = {name: rel_l2(g, r) for name, g, r in zip(("dq", "dk", "dv"), got, want)}
    res["finite"] = bool(all(np.all(np.isfinite(g)) for g in got))
    return res


def assert_bwd_ok(res):
    assert res["finite"], res
    for name in ("dq", "dk", "dv"):
        assert res[name] <= GRAD_REL_L2, res
