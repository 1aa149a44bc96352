"""The jagged forward under Cluster Launch Control scheduling: same results as
the static plan (parity with the oracle, and bit-identical outputs, since each
unit is computed by one CTA in the same way whichever CTA takes it)."""
import pytest
import torch

import variable_length_attention_gb300 as V
from variable_length_attention_gb300 import workloads as W
from tests.parity import assert_fwd_ok, check_fwd, gpu_inputs, sample_units

pytestmark = pytest.mark.gpu


@pytest.fixture
def clc_mode():
    old = V.jfa_get_schedule()
    V.jfa_set_schedule("clc")
    yield
    V.jfa_set_schedule(old)


@pytest.mark.parametrize("w", [W.tiny(), W.custom([1, 63, 129, 257, 513, 1000], 2, 128, causal=True, seed_base=40),
                               W.custom([5, 0, 130, 700], 2, 64, nq=300, seed_base=41)],
                         ids=["tiny", "causal_edges", "broadcast"])
def test_clc_parity(clc_mode, w):
    res, _ = check_fwd(w)
    assert_fwd_ok(res)


def test_clc_full_size_matches_static(clc_mode):
    w = W.jagged(False)
    (q, k, v, _), offs, _ = gpu_inputs(w)
    o_clc, l_clc = V.jfa_fwd(q, k, v, offs, w.offsets)
    V.jfa_set_schedule("static")
    o_st, l_st = V.jfa_fwd(q, k, v, offs, w.offsets)
    torch.cuda.synchronize()
    assert torch.equal(o_clc, o_st) and torch.equal(l_clc, l_st)
    V.jfa_set_schedule("clc")
    res, _ = check_fwd(w, sel=sample_units(w.batch, w.num_heads, 8, seed=5))
    assert_fwd_ok(res)
