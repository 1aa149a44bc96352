"""Planted mistakes in the oracle: each must make the oracle's pins fail.

Every case copies oracle/jfa_oracle.c, plants one plausible mistake in the copy
(a dropped term, a wrong sign, a wrong index or operand, a lost sum), compiles
it, and runs tests/test_oracle_pins.py against it in a subprocess; the pins
must report a failure.  The unmodified source goes through the same steps as a
control and must pass.  Only value mistakes are planted: none of them can move
an array index out of its buffer, so a mutant fails by its numbers, not by
crashing.  CPU only.
"""
import concurrent.futures
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "jfa_oracle.c")

# name -> (text in the oracle, replacement, which occurrence (0-based); None = the text is unique)
MUTANTS = {
    "control": None,
    "scale dropped from the forward scores": (
        "p[j] = scale * dot(q + (long)i * qs, k + (long)j * ks, D);",
        "p[j] = dot(q + (long)i * qs, k + (long)j * ks, D);", None),
    "causal mask one key short": (
        "if (right >= 0 && i + right + 1 < e) e = i + right + 1;", "if (right >= 0 && i + right < e) e = i + right;",
        None),
    "causal mask one key long": (
        "if (right >= 0 && i + right + 1 < e) e = i + right + 1;",
        "if (right >= 0 && i + right + 2 < e) e = i + right + 2;", None),
    "window start one key early": (
        "if (left >= 0 && i - left > a) a = i - left;", "if (left >= 0 && i - left - 1 > a) a = i - left - 1;", None),
    "window start one key late": (
        "if (left >= 0 && i - left > a) a = i - left;", "if (left >= 0 && i - left + 1 > a) a = i - left + 1;", None),
    "row maximum not subtracted (LSE loses m)": ("p[j] = exp(p[j] - m);", "p[j] = exp(p[j]);", 0),
    "LSE without the maximum": ("lse[(long)i * lse_stride] = m + log(l);", "lse[(long)i * lse_stride] = log(l);",
                                None),
    "LSE in base 2": ("lse[(long)i * lse_stride] = m + log(l);", "lse[(long)i * lse_stride] = m + log2(l);",
                      None),
    "output not normalised": ("const double pij = p[j] / l;", "const double pij = p[j];", None),
    "backward P not normalised": ("for (int j = j0; j < n; ++j) p[j] /= l;", "", None),
    "Di dropped from dS": ("const double ds = p[j] * (dp[j] - di);", "const double ds = p[j] * dp[j];", None),
    "Di with the wrong sign": ("const double ds = p[j] * (dp[j] - di);", "const double ds = p[j] * (dp[j] + di);",
                               None),
    "dP against K instead of V": ("dp[j] = dot(doi, v + (long)j * ks, D);", "dp[j] = dot(doi, k + (long)j * ks, D);",
                                  None),
    "dQ without the scale": ("dqi[d] += scale * ds * kj[d];", "dqi[d] += ds * kj[d];", None),
    "dQ from Q instead of K": ("dqi[d] += scale * ds * kj[d];", "dqi[d] += scale * ds * qi[d];", None),
    "dK without the scale": ("dkj[d] += scale * ds * qi[d];", "dkj[d] += ds * qi[d];", None),
    "dK with the wrong sign": ("dkj[d] += scale * ds * qi[d];", "dkj[d] -= scale * ds * qi[d];", None),
    "dV from dP instead of P": ("dvj[d] += p[j] * doi[d];", "dvj[d] += dp[j] * doi[d];", None),
    "GQA: query head read the wrong K/V head": (
        "const int b = (int)(u / H), h = (int)(u % H), g = h / G;",
        "const int b = (int)(u / H), h = (int)(u % H), g = h % Hkv;", None),
    "GQA backward: only the group's first query head": (
        "for (int h = g * G; h < (g + 1) * G; ++h) {\n      if (!unit_selected(J, b, h)) continue;\n      const int step",
        "for (int h = g * G; h < g * G + 1; ++h) {\n      if (!unit_selected(J, b, h)) continue;\n      const int step",
        None),
    "backward ignores the causal mask": ("J->kind == 1 ? J->right : -1", "-1", None),
    "backward ignores the window start": ("J->kind == 1 ? J->left : -1", "-1", None),
    "broadcast: every sequence writes the first output rows": ("const long r0 = (long)b * J->nq;",
                                                               "const long r0 = 0;", None),
    "broadcast backward: dO of the first sequence for all": ("J->dout + (long)b * nq * qs", "J->dout", None),
    "broadcast dQ keeps one chunk instead of the sum": (
        "s += J.dq_part[((size_t)c * H + h) * part + (size_t)i * D + d];",
        "s = J.dq_part[((size_t)c * H + h) * part + (size_t)i * D + d];", None),
    "block forward: keys of the rest of the sequence visible": (
        "n, n, D, J->scale, -1, -1, J->o + (t0 + s) * qs", "n, L - s, D, J->scale, -1, -1, J->o + (t0 + s) * qs",
        None),
    "block backward: whole sequence as one block": (
        "const int step = (J->kind == 4) ? J->block : (L > 0 ? L : 1);", "const int step = (L > 0 ? L : 1);", None),
}


def _plant(text, mutation):
    if mutation is None:
        return text
    old, new, which = mutation
    n = text.count(old)
    if which is None:
        assert n == 1, f"{old!r} occurs {n} times in the oracle"
        return text.replace(old, new)
    assert n > which, f"{old!r} occurs {n} times in the oracle"
    at = -1
    for _ in range(which + 1):
        at = text.index(old, at + 1)
    return text[:at] + new + text[at + len(old):]


def _run(name, mutation, workdir, src):
    tag = "m%02d" % list(MUTANTS).index(name)
    c_path = os.path.join(workdir, tag + ".c")
    so_path = os.path.join(workdir, tag + ".so")
    with open(c_path, "w") as f:
        f.write(_plant(src, mutation))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", c_path, "-o", so_path, "-lm"])
    env = dict(os.environ, JFA_ORACLE_MUTANT_LIB=so_path, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x",
                        "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    last = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else ""
    return r.returncode, last


@pytest.fixture(scope="module")
def outcomes():
    with open(SRC) as f:
        src = f.read()
    with tempfile.TemporaryDirectory() as workdir:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            futs = {name: ex.submit(_run, name, m, workdir, src) for name, m in MUTANTS.items()}
            return {name: f.result() for name, f in futs.items()}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(outcomes, name):
    rc, last = outcomes[name]
    if MUTANTS[name] is None:
        assert rc == 0, last  # the unmodified oracle passes its pins
    else:
        assert rc == 1, f"{name}: pins exit {rc} ({last})"  # 1: a pin failed (not a crash, not a usage error)


# Planted mistakes in the rotary embedding (Python, fp64): each variant of the
# rotation must fail the rotary pins.
def _rope_variant(kind):
    import numpy as np
    import oracle

    def rope(x, offsets, base, *, transpose=False):
        x = np.asarray(x, dtype=np.float64)
        D = x.shape[2]
        half = D // 2
        pos = np.zeros(x.shape[0])
        for b in range(len(offsets) - 1):
            a, e = int(offsets[b]), int(offsets[b + 1])
            pos[a:e] = np.arange(e - a) if kind != "global positions" else np.arange(a, e)
        expo = -1.0 if kind == "angle exponent halved" else -2.0
        theta = base ** (expo * np.arange(half) / D)
        ang = pos[:, None] * theta[None, :]
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        if transpose and kind != "transpose not inverted":
            s = -s
        if kind == "sine with the wrong sign":
            s = -s
        if kind == "adjacent pairs instead of halves":
            x1, x2 = x[..., 0::2], x[..., 1::2]
            y = np.empty_like(x)
            y[..., 0::2], y[..., 1::2] = x1 * c - x2 * s, x2 * c + x1 * s
            return y
        x1, x2 = x[..., :half], x[..., half:]
        return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
    return rope


ROPE_MUTANTS = ["sine with the wrong sign", "angle exponent halved", "global positions", "transpose not inverted",
                "adjacent pairs instead of halves"]


@pytest.mark.parametrize("kind", ROPE_MUTANTS)
def test_rope_pins_catch_planted_mistake(kind):
    from tests.test_oracle_pins import _rope_pins
    with pytest.raises(AssertionError):
        _rope_pins(_rope_variant(kind))


def test_rope_variant_control_passes():
    from tests.test_oracle_pins import _rope_pins
    _rope_pins(_rope_variant("control"))


# Planted mistakes in the two-stage block-sparse forward (Python, fp64): each
# must fail the top-k pins.
def _topk_variant(kind):
    import types

    import numpy as np
    import oracle

    ns = types.SimpleNamespace(topk_scores=oracle.topk_scores, topk_select=oracle.topk_select,
                               attn_fwd_topk=oracle.attn_fwd_topk)
    if kind == "lowest scores chosen":
        ns.topk_select = lambda scores, topk: [sorted(sorted(range(len(sc)), key=lambda j: (sc[j], j))[:topk])
                                               for sc in scores]
    elif kind == "ties to the higher index":
        ns.topk_select = lambda scores, topk: [sorted(sorted(range(len(sc)), key=lambda j: (-sc[j], -j))[:topk])
                                               for sc in scores]
    elif kind == "tail block mean over the full block size":
        def scores_fn(q, k, offsets, nq=0):
            q, k = np.asarray(q, float), np.asarray(k, float)
            H, Hkv = q.shape[1], k.shape[1]
            out = []
            for b, h, m, (r0, r1), (a, e) in oracle._topk_units(offsets, H, nq):
                qm = (q[r0:r1, h] if nq > 0 else q[a + r0:a + r1, h]).mean(axis=0)
                ks = k[a:e, h // (H // Hkv)]
                out.append(np.array([qm @ (ks[j:j + 128].sum(axis=0) / 128) for j in range(0, e - a, 128)]))
            return out
        ns.topk_scores = scores_fn
    elif kind == "unchosen keys attended":
        def attn_all(q, k, v, offsets, selection, *, scale, nq=0):
            full = [list(range(-(-(int(e) - int(a)) // 128))) for (_, _, _, _, (a, e)) in
                    oracle._topk_units(offsets, q.shape[1], nq)]
            return oracle.attn_fwd_topk(q, k, v, offsets, full, scale=scale, nq=nq)
        ns.attn_fwd_topk = attn_all
    elif kind == "query blocks of 128 rows":
        saved = oracle.TOPK_Q_BLOCK

        def scores_fn(*args, **kw):
            oracle.TOPK_Q_BLOCK = 128
            try:
                return oracle.topk_scores(*args, **kw)
            finally:
                oracle.TOPK_Q_BLOCK = saved
        ns.topk_scores = scores_fn
    return ns


TOPK_MUTANTS = ["lowest scores chosen", "ties to the higher index", "tail block mean over the full block size",
                "unchosen keys attended", "query blocks of 128 rows"]


@pytest.mark.parametrize("kind", TOPK_MUTANTS)
def test_topk_pins_catch_planted_mistake(kind):
    from tests.test_oracle_pins import _topk_pins
    with pytest.raises((AssertionError, ValueError)):
        _topk_pins(_topk_variant(kind))


def test_topk_variant_control_passes():
    from tests.test_oracle_pins import _topk_pins
    _topk_pins(_topk_variant("control"))
