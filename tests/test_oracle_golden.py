"""The pages' own worked examples, re-run on the oracle (fixtures in tests/golden/)."""
import json
import os

import numpy as np

from oracle_pins import phi_np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_mlblogg_pairwise_example(orc):
    g = _load("mlblogg_pairwise_check.json")
    rng = np.random.default_rng(g["seed"])
    q, k = rng.normal(size=(2, g["N"], g["dk"]))
    v = rng.normal(size=(g["N"], g["dv"]))
    out = orc.noncausal(q, k, v, 1e-6)
    assert list(out.shape) == g["printed_shape"]
    pairwise = phi_np(q) @ phi_np(k).T
    reference = (pairwise @ v) / pairwise.sum(-1, keepdims=True)
    np.testing.assert_allclose(out, reference, atol=g["atol"], rtol=0)


def test_problems_doctest_shape(orc):
    g = _load("problems_doctest_shape.json")
    rng = np.random.default_rng(0)
    q = rng.standard_normal(g["q_shape"])
    k = rng.standard_normal(g["k_shape"])
    v = rng.standard_normal(g["v_shape"])
    out = orc.causal_recurrent(q, k, v, 1e-6)
    assert list(out.shape) == g["printed_shape"]
    # the same page's sanity check: output 0 equals v_0
    np.testing.assert_allclose(out[:, 0], v[:, 0], rtol=1e-14, atol=1e-15)
