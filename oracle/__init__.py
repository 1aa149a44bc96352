"""fp64 CPU oracle for jagged attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and it
never calls the CUDA library: the two share no code.

The arithmetic lives in ``jfa_oracle.c`` (plain C, fp64, one thread per
(sequence, head) unit); this module compiles it with gcc on first use and wraps
it with ctypes.  Arrays are float64 numpy arrays in [rows, heads, dim] layout;
offsets are int32 with offsets[0] == 0 (the packed-sequence convention of the
jagged-attention pages: sequence b is rows offsets[b] .. offsets[b+1]-1).

Functions
---------
attn_fwd   exact softmax(scale Q K^T) V per sequence and head, plus the natural-log
           log-sum-exp per row; self-attention or broadcast-Q (nq > 0).
attn_bwd   dQ, dK, dV for the loss sum(O * dO); broadcast-Q sums the shared-Q
           gradient over all sequences.
block_fwd  / block_bwd: the same inside fixed blocks of ``block`` tokens;
           with ``rope_base`` the rotary embedding is applied to Q and K first
           (and the gradients are taken with respect to the unrotated Q, K).
rope       the rotary embedding itself (and its transpose).
topk_scores / topk_select / attn_fwd_topk: the two-stage block-sparse
           forward (block means, top-k key blocks per query block, attention
           over the selected blocks only).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jfa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libjfa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -ffast-math: IEEE fp64 throughout)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib_path() -> str:
    """The compiled oracle.  tests/test_oracle_mutants.py alone sets
    JFA_ORACLE_MUTANT_LIB, to run the pins against copies of the oracle with a
    deliberate mistake planted in them and check that the pins fail."""
    return os.environ.get("JFA_ORACLE_MUTANT_LIB") or build()


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_lib_path())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            bp = ctypes.c_void_p
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_attn_fwd.argtypes = [dp, dp, dp, ip, i, i, i, i, i, d, i, bp, dp, dp, i]
            lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, ip, i, i, i, i, i, d, i, bp, dp, dp, dp, i]
            lib.oracle_attn_fwd_window.argtypes = [dp, dp, dp, ip, i, i, i, i, i, d, i, i, bp, dp, dp, i]
            lib.oracle_attn_bwd_window.argtypes = [dp, dp, dp, dp, ip, i, i, i, i, i, d, i, i, bp, dp, dp, dp, i]
            lib.oracle_block_fwd.argtypes = [dp, dp, dp, ip, i, i, i, d, i, bp, dp, i]
            lib.oracle_block_bwd.argtypes = [dp, dp, dp, dp, ip, i, i, i, d, i, bp, dp, dp, dp, i]
            for f in (lib.oracle_attn_fwd, lib.oracle_attn_bwd, lib.oracle_block_fwd, lib.oracle_block_bwd,
                      lib.oracle_attn_fwd_window, lib.oracle_attn_bwd_window):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _offs(offsets) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(offsets, dtype=np.int32))


def _sel(sel, batch, H):
    if sel is None:
        return None, None
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.uint8).reshape(batch * H))
    return s, s.ctypes.data_as(ctypes.c_void_p)


def _window(causal, window):
    """(left, right) of the visible window: key j is visible to query i iff
    i - left <= j <= i + right (a side given as None or a negative number is
    open); causal closes the right side at 0."""
    left, right = window if window is not None else (None, None)
    left = -1 if left is None or left < 0 else int(left)
    right = -1 if right is None or right < 0 else int(right)
    if causal:
        right = 0 if right < 0 else min(right, 0)
    return left, right


def attn_fwd(q, k, v, offsets, *, scale: float, causal: bool = False, nq: int = 0,
             sel=None, nthreads: int = 0, out=None, window=None):
    """Returns (o, lse, threads_used).

    Self mode (nq == 0): q [T,H,D], k/v [T,Hkv,D] -> o [T,H,D], lse [H,T].
    Broadcast (nq > 0): q [nq,H,D] -> o [B*nq,H,D], lse [H,B*nq].
    ``window`` = (left, right) restricts query i to keys i-left .. i+right of
    its sequence (self mode only).
    Units not selected by ``sel`` ([B,H] bool) are left as NaN.
    """
    lib = _load()
    q, k, v, offsets = _f64(q), _f64(k), _f64(v), _offs(offsets)
    B = offsets.shape[0] - 1
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    rows = B * nq if nq > 0 else int(offsets[-1])
    o = np.full((rows, H, D), np.nan)
    lse = np.full((H, rows), np.nan)
    s_arr, s_ptr = _sel(sel, B, H)
    left, right = _window(causal, window)
    used = lib.oracle_attn_fwd_window(_ptr(q), _ptr(k), _ptr(v),
                                      offsets.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, nq, H, Hkv, D,
                                      float(scale), left, right, s_ptr, _ptr(o), _ptr(lse), int(nthreads))
    if used < 0:
        raise ValueError(f"oracle_attn_fwd rejected its arguments ({used})")
    return o, lse, used


def attn_bwd(q, k, v, dout, offsets, *, scale: float, causal: bool = False, nq: int = 0,
             sel=None, nthreads: int = 0, window=None):
    """Returns (dq, dk, dv, threads_used) for the loss sum(O * dout); ``window``
    as in attn_fwd."""
    lib = _load()
    q, k, v, dout, offsets = _f64(q), _f64(k), _f64(v), _f64(dout), _offs(offsets)
    B = offsets.shape[0] - 1
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    s_arr, s_ptr = _sel(sel, B, H)
    left, right = _window(causal, window)
    used = lib.oracle_attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                      offsets.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, nq, H, Hkv, D,
                                      float(scale), left, right, s_ptr, _ptr(dq), _ptr(dk), _ptr(dv),
                                      int(nthreads))
    if used < 0:
        raise ValueError(f"oracle_attn_bwd rejected its arguments ({used})")
    return dq, dk, dv, used


def rope(x, offsets, base: float, *, transpose: bool = False):
    """Rotary position embedding of the rows of a packed [rows, heads, D] array,
    in fp64.  "TLX Block Attention" fuses a rotary embedding into the block
    kernel (introduction: 2.3x kernel, 3.5x with rotary fused) without giving
    its convention; the reading here is the rotate-half form: the position of a
    row is its index inside its sequence, and for i < D/2 the pair
    (x_i, x_{i+D/2}) is turned by the angle pos * base^(-2i/D):
        (x_i, x_{i+D/2}) -> (x_i cos - x_{i+D/2} sin, x_{i+D/2} cos + x_i sin).
    transpose=True applies the inverse (transposed) rotation, which carries a
    gradient with respect to rotated rows back to the unrotated rows."""
    x = _f64(x)
    offsets = _offs(offsets)
    D = x.shape[2]
    half = D // 2
    pos = np.zeros(x.shape[0])
    for b in range(len(offsets) - 1):
        a, e = int(offsets[b]), int(offsets[b + 1])
        pos[a:e] = np.arange(e - a)
    theta = base ** (-2.0 * np.arange(half) / D)
    ang = pos[:, None] * theta[None, :]          # [rows, D/2]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    if transpose:
        s = -s
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def block_fwd(q, k, v, offsets, *, scale: float, block: int = 64, sel=None, nthreads: int = 0, rope_base=None):
    """Block-diagonal forward; returns (o, threads_used).  With ``rope_base``,
    Q and K are rotated by rope() first."""
    lib = _load()
    if rope_base is not None:
        q, k = rope(q, offsets, rope_base), rope(k, offsets, rope_base)
    q, k, v, offsets = _f64(q), _f64(k), _f64(v), _offs(offsets)
    B = offsets.shape[0] - 1
    H, D = q.shape[1], q.shape[2]
    o = np.full_like(q, np.nan)
    s_arr, s_ptr = _sel(sel, B, H)
    used = lib.oracle_block_fwd(_ptr(q), _ptr(k), _ptr(v), offsets.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                B, H, D, float(scale), int(block), s_ptr, _ptr(o), int(nthreads))
    if used < 0:
        raise ValueError(f"oracle_block_fwd rejected its arguments ({used})")
    return o, used


def block_bwd(q, k, v, dout, offsets, *, scale: float, block: int = 64, sel=None, nthreads: int = 0,
              rope_base=None):
    """Block-diagonal backward; returns (dq, dk, dv, threads_used).  With
    ``rope_base``: the backward of the rotated problem, its dQ and dK carried
    back through the transposed rotation to the unrotated Q and K."""
    if rope_base is not None:
        qr, kr = rope(q, offsets, rope_base), rope(k, offsets, rope_base)
        dq, dk, dv, used = block_bwd(qr, kr, v, dout, offsets, scale=scale, block=block, sel=sel, nthreads=nthreads)
        return (rope(dq, offsets, rope_base, transpose=True), rope(dk, offsets, rope_base, transpose=True), dv,
                used)
    lib = _load()
    q, k, v, dout, offsets = _f64(q), _f64(k), _f64(v), _f64(dout), _offs(offsets)
    B = offsets.shape[0] - 1
    H, D = q.shape[1], q.shape[2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    s_arr, s_ptr = _sel(sel, B, H)
    used = lib.oracle_block_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                offsets.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, H, D, float(scale),
                                int(block), s_ptr, _ptr(dq), _ptr(dk), _ptr(dv), int(nthreads))
    if used < 0:
        raise ValueError(f"oracle_block_bwd rejected its arguments ({used})")
    return dq, dk, dv, used


# --------------------------------------------------------------------------- block-sparse top-k forward
# The aixai.ru summary ("MXFP8 and sparsity") describes a two-stage variant for
# long histories: a cheap first stage averages blocks of Q and of K and picks
# the top-k most relevant key blocks, and the attention kernel then attends
# over those blocks only.  The block sizes, the score and the tie rule are not
# given; the readings here: query blocks of 256 rows (the forward kernel's
# unit) and key blocks of 128 keys, each block's mean over the rows it really
# has; score = mean query . mean key (key/value head h // (H/Hkv)); the k
# highest scores, ties to the lower block index; attention is exact softmax
# attention over every key of the chosen blocks.
TOPK_Q_BLOCK = 256
TOPK_K_BLOCK = 128


def _topk_units(offsets, H, nq):
    """(b, h, m, query row range, key range) of every query block, in the
    order b, h, m (a sequence without keys has none)."""
    offsets = _offs(offsets)
    out = []
    for b in range(len(offsets) - 1):
        a, e = int(offsets[b]), int(offsets[b + 1])
        if e == a:
            continue
        rows = nq if nq > 0 else e - a
        for h in range(H):
            for m in range(-(-rows // TOPK_Q_BLOCK)):
                r0 = m * TOPK_Q_BLOCK
                r1 = min(rows, r0 + TOPK_Q_BLOCK)
                out.append((b, h, m, (r0, r1), (a, e)))
    return out


def topk_scores(q, k, offsets, *, nq: int = 0):
    """Stage one, fp64: for every query block (order b, h, m) the scores of the
    key blocks of its sequence, mean query row . mean key row."""
    q, k = _f64(q), _f64(k)
    H, Hkv = q.shape[1], k.shape[1]
    G = H // Hkv
    scores = []
    for b, h, m, (r0, r1), (a, e) in _topk_units(offsets, H, nq):
        qb = q[r0:r1, h] if nq > 0 else q[a + r0:a + r1, h]
        qm = qb.mean(axis=0)
        ks = k[a:e, h // G]
        sc = [qm @ ks[j:j + TOPK_K_BLOCK].mean(axis=0) for j in range(0, e - a, TOPK_K_BLOCK)]
        scores.append(np.array(sc))
    return scores


def topk_select(scores, topk: int):
    """The chosen key blocks of every query block: the topk highest scores
    (all blocks if there are fewer), ties to the lower index, ascending."""
    sel = []
    for sc in scores:
        order = sorted(range(len(sc)), key=lambda j: (-sc[j], j))
        sel.append(sorted(order[:topk]))
    return sel


def attn_fwd_topk(q, k, v, offsets, selection, *, scale: float, nq: int = 0):
    """Stage two, fp64: every query row attends over the keys of its query
    block's chosen key blocks (``selection`` as topk_select returns it, in the
    order b, h, m).  Returns (o, lse) shaped like attn_fwd's."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    offsets = _offs(offsets)
    H, Hkv, D = q.shape[1], k.shape[1], q.shape[2]
    G = H // Hkv
    B = len(offsets) - 1
    rows_out = B * nq if nq > 0 else int(offsets[-1])
    o = np.zeros((rows_out, H, D))
    lse = np.full((H, rows_out), -np.inf)
    units = _topk_units(offsets, H, nq)
    assert len(units) == len(selection)
    for (b, h, m, (r0, r1), (a, e)), blocks in zip(units, selection):
        keys = np.concatenate([np.arange(a + j * TOPK_K_BLOCK, min(e, a + (j + 1) * TOPK_K_BLOCK)) for j in blocks])
        qb = q[r0:r1, h] if nq > 0 else q[a + r0:a + r1, h]
        s = scale * (qb @ k[keys, h // G].T)
        mx = s.max(axis=1, keepdims=True)
        p = np.exp(s - mx)
        l = p.sum(axis=1, keepdims=True)
        out_rows = slice(b * nq + r0, b * nq + r1) if nq > 0 else slice(a + r0, a + r1)
        o[out_rows, h] = (p / l) @ v[keys, h // G]
        lse[h, out_rows] = (mx + np.log(l))[:, 0]
    return o, lse
