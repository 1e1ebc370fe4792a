"""The oracle against worked values the pages print (fixtures under
tests/golden/, each citing its page and section)."""
import json
import os

import numpy as np

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ops(names):
    t = np.zeros(O.N_OPS, bool)
    for name in names:
        t[0 if name == "add" else 1 + int(name.split()[1])] = True
    return t


def test_frontier_explorer_eight_token_slot():
    """GraceKV "02 Progressively refinable representation": one 8-token slot
    stores 0, 1, 3 or 8 entries; the 1-entry root covers all eight tokens and
    the 8-entry frontier holds the original tokens' K/V."""
    g = json.load(open(os.path.join(GOLDEN, "frontier_explorer_8_tokens.json")))
    x0, y0 = g["slot"]
    n = y0
    rng = np.random.default_rng(0)
    d = 16
    K = O.rope_rotate(rng.standard_normal((n, d)), np.arange(n), 10000.0)
    V = rng.standard_normal((n, d))
    r = rng.uniform(0.1, 1.0, n)
    nodes = O.tree_nodes(x0, y0)
    for case in g["cases"]:
        t = _ops(case["ops_taken"])
        front = O.frontier(t, x0, y0)
        assert len(front) == case["entries"], case
        Kp, Vp, lm, ps = O.pack_head(K, V, r, np.asarray([x0, y0]), t[None], n, 0, 10000.0, 0.1)
        assert len(Kp) == case["entries"]
        if "covers" in case:
            assert [list(nodes[j]) for _, j in front] == case["covers"]
            np.testing.assert_allclose(ps, [(a + b - 1) / 2 for a, b in case["covers"]])
        if case.get("original_tokens"):
            # eight one-token leaves: each stored entry is its token's K/V
            np.testing.assert_allclose(Kp, K, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(Vp, V, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lm, 0.0, atol=1e-12)
            np.testing.assert_array_equal(ps, np.arange(n))
