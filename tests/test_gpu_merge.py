"""GPU parity of the standalone LSE merge against the oracle's fp64 merge, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_merge_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,hd,dtype", [(1, 128, "bf16"), (1000, 128, "bf16"), (777, 64, "bf16"),
                                           (513, 64, "f32"), (300, 128, "f32"), (64, 256, "f32"),
                                           (50, 24, "bf16")])
@pytest.mark.parametrize("neg_inf_frac", [0.0, 0.3])
def test_merge_matches_oracle(rows, hd, dtype, neg_inf_frac):
    o1, l1, o2, l2 = make_merge_inputs(rows, hd, dtype, seed=rows + hd, neg_inf_frac=neg_inf_frac)
    o_ref, l_ref = oracle.lse_merge(o1.double().numpy(), l1.double().numpy(), o2.double().numpy(),
                                    l2.double().numpy())
    oa, la = o1.cuda(), l1.cuda()
    usp.usp_lse_merge(oa, la, o2.cuda(), l2.cuda())
    usp.usp_check()
    o = oa.float().cpu().numpy()
    lse = la.cpu().numpy()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isneginf(lse), ~fin)
    np.testing.assert_allclose(lse[fin], l_ref[fin], rtol=1e-6, atol=1e-6)
    # fp32 arithmetic; a bf16 output is rounded once to nearest (at most 2^-8 of its magnitude)
    rel = 1e-6 if dtype == "f32" else 2.0 ** -8
    assert np.all(np.abs(o - o_ref) <= rel * np.abs(o_ref) + 1e-5)
    assert np.all(o[~fin] == 0)


def test_merge_chain_equals_single_pass():
    """Folding k partials one at a time is the same as the oracle folding them."""
    rows, hd = 256, 128
    parts = [make_merge_inputs(rows, hd, "f32", seed=s) for s in range(4)]
    oa, la = parts[0][0].cuda(), parts[0][1].cuda()
    o_ref, l_ref = parts[0][0].double().numpy(), parts[0][1].double().numpy()
    for o2, l2, _, _ in parts[1:]:
        usp.usp_lse_merge(oa, la, o2.cuda(), l2.cuda())
        o_ref, l_ref = oracle.lse_merge(o_ref, l_ref, o2.double().numpy(), l2.double().numpy())
    usp.usp_check()
    np.testing.assert_allclose(la.cpu().numpy(), l_ref, rtol=1e-6, atol=1e-6)
    assert np.abs(oa.cpu().numpy() - o_ref).max() <= 1e-5
