"""Host logic of the GPU parity checks (no GPU): which kernel routing choices
the checks accept, and the routing they then give the oracle."""
import numpy as np
import pytest

import oracle

import _gpu


def _case():
    """E = 4, k = 2, one token per row of the logit table: token 0 decided,
    token 1 with a near-tie between experts 1 and 2 for the second slot."""
    logits = np.array([[3.0, 1.0, 0.5, 0.0],
                       [3.0, 1.0, 1.0 + 5e-6, 0.0]])
    # x = the identity (d = 2) and W_r = the table transposed give these logits
    return dict(x=np.eye(2), w_router=logits.T.copy(), bias=None)


def test_forced_routing_keeps_the_oracles_choice_where_it_is_decided():
    inp = _case()
    idx, _, _, flagged, _ = oracle.route_ref(inp["x"], inp["w_router"], None, 2)
    assert list(flagged) == [False, True]
    use, p, fl = _gpu.forced_routing(inp, 2, idx)
    assert np.array_equal(use, idx)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-15)


def test_forced_routing_takes_a_valid_choice_on_a_near_tie():
    inp = _case()
    gpu = np.array([[0, 1], [0, 1]], dtype=np.int32)   # oracle: [0, 2] for token 1
    use, p, _ = _gpu.forced_routing(inp, 2, gpu)
    assert np.array_equal(use, gpu)
    l = np.array([3.0, 1.0])
    np.testing.assert_allclose(p[1], np.exp(l - 3) / np.exp(l - 3).sum(), rtol=1e-15)


@pytest.mark.parametrize("gpu", [
    [[0, 2], [0, 2]],   # token 0 is decided: its second expert is 1
    [[0, 1], [0, 3]],   # token 1: expert 3 is far below the tie
    [[0, 1], [2, 2]],   # an expert twice
])
def test_forced_routing_rejects_invalid_choices(gpu):
    with pytest.raises(AssertionError):
        _gpu.forced_routing(_case(), 2, np.array(gpu, dtype=np.int32))
