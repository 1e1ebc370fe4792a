"""Pins for the oracle's prototype trees, merge math, distortion and op utilities."""
import math

import numpy as np
import pytest

import oracle as O


def _rot(x, p, base=10000.0):
    return O.rope_rotate(x, p, base)


# ------------------------------------------------------------------ tree shape
def test_midpoint_tree_shape():
    nodes = O.tree_nodes(0, 64)
    assert nodes[0] == (0, 64) and nodes[1] == (0, 32) and nodes[2] == (32, 64)
    assert [n for n in nodes[7:]] == [(8 * k, 8 * k + 8) for k in range(8)]
    odd = O.tree_nodes(100, 117)                    # 17 tokens: leaves of 2 or 3 tokens
    leaves = odd[7:]
    assert leaves[0][0] == 100 and leaves[-1][1] == 117
    assert all(leaves[k][1] == leaves[k + 1][0] for k in range(7))
    assert sorted(b - a for a, b in leaves) == [2] * 7 + [3]
    for j in range(7):                               # children partition the parent
        a, b = odd[j]
        assert odd[2 * j + 1][0] == a and odd[2 * j + 2][1] == b
        assert odd[2 * j + 1][1] == odd[2 * j + 2][0] == (a + b) // 2


# ------------------------------------------------------------------ prototypes
def test_one_token_prototype_is_the_token():
    rng = np.random.default_rng(0)
    k = rng.standard_normal((1, 64)); v = rng.standard_normal((1, 64))
    pr = O.prototype(k, v, np.array([0.3]), 37, 38, 10000.0, 0.1)
    np.testing.assert_allclose(pr.k_hat, k[0], atol=1e-12)
    np.testing.assert_allclose(pr.v_hat, v[0], atol=1e-15)
    assert pr.m == 1.0 and pr.log_m == 0.0 and pr.p_bar == 37.0


def test_identical_unrotated_keys_give_full_multiplicity():
    """Keys R(i) k for one k: kappa = 1, m = c, k_hat = R(p_bar) k (p_bar = (x+y-1)/2)."""
    rng = np.random.default_rng(1)
    k = rng.standard_normal(128)
    x, y = 200, 213
    K = _rot(np.tile(k, (y - x, 1)), np.arange(x, y))
    pr = O.prototype(K, rng.standard_normal((y - x, 128)), np.ones(y - x), x, y, 10000.0, 0.1)
    assert abs(pr.kappa - 1.0) < 1e-12 and abs(pr.m - 13.0) < 1e-10
    assert pr.p_bar == 206.0
    np.testing.assert_allclose(pr.k_hat, _rot(k, 206.0), atol=1e-11)
    pr2 = O.prototype(K[:12], K[:12], np.ones(12), x, x + 12, 10000.0, 0.1)
    assert pr2.p_bar == 205.5
    np.testing.assert_allclose(pr2.k_hat, _rot(k, 205.5), atol=1e-11)


def test_incoherent_keys_clamp_multiplicity_to_one():
    """Two opposite unrotated keys: mean is 0, kappa = 0 -> m = c * clamp(0, 1/c, 1) = 1."""
    k = np.random.default_rng(2).standard_normal(16)
    K = _rot(np.stack([k, -k]), np.array([5, 6]))
    pr = O.prototype(K, K, np.ones(2), 5, 7, 10000.0, 0.1)
    assert pr.m == 1.0


def test_value_merge_weights():
    rng = np.random.default_rng(3)
    V = rng.standard_normal((8, 32))
    K = rng.standard_normal((8, 32))
    # zero relevance -> uniform mean
    pr = O.prototype(K, V, np.zeros(8), 0, 8, 10000.0, 0.1)
    np.testing.assert_allclose(pr.v_hat, V.mean(0), atol=1e-14)
    # all relevance on token 3 -> 0.9 v_3 + 0.1 * mean(v)
    r = np.zeros(8); r[3] = 2.5
    pr = O.prototype(K, V, r, 0, 8, 10000.0, 0.1)
    np.testing.assert_allclose(pr.v_hat, 0.9 * V[3] + 0.1 * V.mean(0), atol=1e-14)
    # weights sum to one: constant values are reproduced
    c = np.tile(rng.standard_normal(32), (8, 1))
    pr = O.prototype(K, c, rng.uniform(size=8), 0, 8, 10000.0, 0.1)
    np.testing.assert_allclose(pr.v_hat, c[0], atol=1e-14)


def test_multiplicity_entry_equals_copies_in_attention():
    """One entry (k_hat, v_hat) with bias +ln c attends exactly like c copies of it."""
    rng = np.random.default_rng(4)
    d, c = 64, 9
    k = rng.standard_normal(d)
    K = _rot(np.tile(k, (c, 1)), np.arange(40, 40 + c))
    V = rng.standard_normal((c, d))
    pr = O.prototype(K, V, rng.uniform(size=c), 40, 40 + c, 10000.0, 0.1)
    assert abs(pr.m - c) < 1e-9
    others_k = rng.standard_normal((20, d)); others_v = rng.standard_normal((20, d))
    q = rng.standard_normal((4, d))
    merged = O.decode_head(q, np.vstack([others_k, pr.k_hat]), np.vstack([others_v, pr.v_hat]),
                           np.r_[np.zeros(20), pr.log_m])
    copies = O.decode_head(q, np.vstack([others_k] + [pr.k_hat[None]] * c),
                           np.vstack([others_v] + [pr.v_hat[None]] * c), np.zeros(20 + c))
    np.testing.assert_allclose(merged, copies, atol=1e-12)


# ------------------------------------------------------------------ distortion
def test_distortion_hand_worked_example():
    """Worked by hand: d = 2 (theta_0 = 1), n = 4, one probe row with q = 0 (uniform
    attention 1/4), node [0, 2) with unrotated keys e1, e2, values e1, e2, relevance
    (1, 0), value floor 0.1, all |v| = 1.
      A = 1/2, U = (1/4, 1/4); kappa = cos(e1, (e1+e2)/2) = 1/sqrt2, m = sqrt2;
      A_hat = exp(0 + ln m - ln 4) = sqrt2/4; v_hat = (0.95, 0.05); U_hat = A_hat v_hat.
      D = 0.25 |A - A_hat| + 0.75 |U - U_hat|;  D_drop = 0.25 A + 0.75 |U|."""
    e1, e2 = np.array([1.0, 0.0]), np.array([0.0, 1.0])
    Kpost = np.stack([e1, _rot(e2, 1.0), _rot(e1, 2.0), _rot(e2, 3.0)])
    V = np.stack([e1, e2, e1, e2])
    q = np.zeros((1, 2))
    sc = O.score_head(Kpost, V, q.reshape(1, 1, 2), 4, 1)
    pr = O.prototype(Kpost[0:2], V[0:2], np.array([1.0, 0.0]), 0, 2, 10000.0, 0.1)
    nu = float(sc.feats[:, 1].mean())
    D, Dd = O.node_distortion(sc.a[:, 0:2], V[0:2], q, sc.lse, pr, nu, 0.25, 0.75)
    Ah = math.sqrt(2) / 4
    A = 0.5
    U = np.array([0.25, 0.25])
    Uh = Ah * np.array([0.95, 0.05])
    D_exp = 0.25 * abs(A - Ah) + 0.75 * math.hypot(*(U - Uh))
    Dd_exp = 0.25 * A + 0.75 * math.hypot(0.25, 0.25)
    assert nu == 1.0
    assert abs(pr.m - math.sqrt(2)) < 1e-14
    assert abs(D - D_exp) < 1e-14 and abs(Dd - Dd_exp) < 1e-14


def test_exact_prototype_has_zero_distortion():
    """Uniform attention (q = 0), identical unrotated keys and identical values: the
    prototype with m = c reproduces both the partition mass and the value aggregate."""
    rng = np.random.default_rng(5)
    d, n = 32, 50
    k = rng.standard_normal(d); v = rng.standard_normal(d)
    K = _rot(np.tile(k, (n, 1)), np.arange(n))
    V = np.tile(v, (n, 1))
    Q = np.zeros((2, 3, d))
    sc = O.score_head(K, V, Q, n, 3)
    pr = O.prototype(K[10:26], V[10:26], rng.uniform(size=16), 10, 26, 10000.0, 0.1)
    D, Dd = O.node_distortion(sc.a[:, 10:26], V[10:26], Q.reshape(6, d), sc.lse, pr,
                              float(np.linalg.norm(v)), 0.25, 0.75)
    assert D < 1e-14 and Dd > 0.1


def test_one_token_node_add_gain_is_one():
    rng = np.random.default_rng(6)
    d, n = 32, 40
    K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d)); Q = rng.standard_normal((4, 2, d))
    sc = O.score_head(K, V, Q, n, 2)
    pr = O.prototype(K[7:8], V[7:8], np.array([1.0]), 7, 8, 10000.0, 0.1)
    D, Dd = O.node_distortion(sc.a[:, 7:8], V[7:8], Q.reshape(8, d), sc.lse, pr,
                              float(sc.feats[:, 1].mean()), 0.25, 0.75)
    assert D < 1e-13 * Dd
    assert abs(O.gain_fraction(Dd - D, Dd) - 1.0) < 1e-12


def test_slot_ops_gains_costs_and_value_flow():
    rng = np.random.default_rng(7)
    D = rng.uniform(0.1, 1.0, 15)
    Dd = D + rng.uniform(0.0, 1.0, 15)
    r = rng.uniform(size=64)
    nodes = O.tree_nodes(0, 64)
    Rv = np.array([r[a:b].sum() for a, b in nodes])
    for j in range(7):                                   # parent value = sum of child values
        assert abs(Rv[j] - Rv[2 * j + 1] - Rv[2 * j + 2]) < 1e-13
    sizes = np.array([b - a for a, b in nodes])
    u, c = O.slot_ops(D, Dd, Rv, sizes, 2.0)
    assert list(c) == [1] * 8 + [7] * 8
    assert abs(u[0] - Rv[0] * (1 - D[0] / Dd[0]) * 2.0) < 1e-12
    for j in range(7, 15):                               # split into exact tokens: D / D_drop
        g = min(D[j] / Dd[j], 1.0)
        assert abs(u[1 + j] - Rv[j] * g * 2.0 / 7) < 1e-12
    for j in range(7):
        g = min(max((D[j] - D[2 * j + 1] - D[2 * j + 2]) / Dd[j], 0.0), 1.0)
        assert abs(u[1 + j] - Rv[j] * g * 2.0) < 1e-12
    assert (u >= 0).all()


def test_head_utilities_gain_range():
    rng = np.random.default_rng(8)
    n, d, G, P = 300, 32, 2, 8
    K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d)); Q = rng.standard_normal((G, P, d))
    bounds = np.array([0, 64, 100, 180, 250])
    res = O.score_and_value_head(K, V, Q, n, P, bounds, 1.0)
    gains = res.util * res.cost
    for s in range(4):
        nodes = O.tree_nodes(int(bounds[s]), int(bounds[s + 1]))
        Rv = np.array([res.r[a:b].sum() for a, b in nodes])
        g = gains[s] / np.r_[Rv[0], Rv]
        assert (g >= -1e-15).all() and (g <= 1 + 1e-12).all()


def _scored(K, V, Q, n, P, bounds):
    # no hops: relevance is the probe attention alone, which involves no values
    return O.score_and_value_head(K, V, Q, n, P, bounds, 1.0, n_hops=0)


def test_distortion_and_utilities_invariant_to_value_scale():
    """The value term divides by the mean value norm (R4), so scaling every
    value by the same factor changes no distortion, gain or utility.  A
    missing or misplaced normalisation fails this."""
    rng = np.random.default_rng(21)
    n, d, G, P = 260, 32, 2, 8
    K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d)); Q = rng.standard_normal((G, P, d))
    bounds = np.array([0, 40, 100, 170, 230])
    a = _scored(K, V, Q, n, P, bounds)
    b = _scored(K, 3.5 * V, Q, n, P, bounds)
    np.testing.assert_allclose(b.D, a.D, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(b.Ddrop, a.Ddrop, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(b.util, a.util, rtol=1e-9, atol=1e-14)
    np.testing.assert_array_equal(b.cost, a.cost)


@pytest.mark.parametrize("shift", [1, 37, 1000])
def test_distortion_invariant_to_a_common_rope_shift(shift):
    """Rotating every key and every probe by the same RoPE shift leaves the
    probe attention unchanged (it depends on position differences) and rotates
    each prototype key with its tokens, so every distortion and utility is
    unchanged: the path sees keys and probes only through relative rotations.
    (A wrong sign of the merge's own rotations keeps this property; the
    one-token and identical-key prototype pins catch that.)"""
    rng = np.random.default_rng(22)
    n, d, G, P = 260, 32, 2, 8
    K = _rot(rng.standard_normal((n, d)), np.arange(n))
    V = rng.standard_normal((n, d))
    Q = rng.standard_normal((G, P, d))
    bounds = np.array([0, 40, 100, 170, 230])
    a = _scored(K, V, Q, n, P, bounds)
    b = _scored(_rot(K, float(shift)), V, _rot(Q, float(shift)), n, P, bounds)
    np.testing.assert_allclose(b.lse, a.lse, rtol=1e-10)
    np.testing.assert_allclose(b.D, a.D, rtol=1e-8, atol=1e-12)
    np.testing.assert_allclose(b.Ddrop, a.Ddrop, rtol=1e-8, atol=1e-12)
    np.testing.assert_allclose(b.util, a.util, rtol=1e-7, atol=1e-12)


def test_node_values_add_up_the_tree_and_feed_the_utilities():
    """[GK] "03 Bottom-up value flow": a node's value is the sum of its tokens'
    relevance, so a parent's value equals the sum of its children's, the
    root's the slot's total; and each op's utility is that value times its
    gain (times sens) per new entry."""
    rng = np.random.default_rng(23)
    n, d, G, P = 260, 32, 2, 8
    K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d)); Q = rng.standard_normal((G, P, d))
    bounds = np.array([0, 40, 100, 170, 230])
    res = O.score_and_value_head(K, V, Q, n, P, bounds, 0.7)
    for s in range(4):
        Rv = res.Rv[s]
        x0, y0 = int(bounds[s]), int(bounds[s + 1])
        np.testing.assert_allclose(Rv[0], res.r[x0:y0].sum(), rtol=1e-12)
        for j in range(7):
            np.testing.assert_allclose(Rv[j], Rv[2 * j + 1] + Rv[2 * j + 2], rtol=1e-12)
        for j in range(7, 15):
            a, b = O.tree_nodes(x0, y0)[j]
            np.testing.assert_allclose(Rv[j], res.r[a:b].sum(), rtol=1e-12)
        g_add = O.gain_fraction(res.Ddrop[s, 0] - res.D[s, 0], res.Ddrop[s, 0])
        np.testing.assert_allclose(res.util[s, 0], Rv[0] * g_add * 0.7, rtol=1e-12)
        for j in range(15):
            num = res.D[s, j] - res.D[s, 2 * j + 1] - res.D[s, 2 * j + 2] if j < 7 else res.D[s, j]
            g = O.gain_fraction(num, res.Ddrop[s, j])
            np.testing.assert_allclose(res.util[s, 1 + j], Rv[j] * g * 0.7 / res.cost[s, 1 + j],
                                       rtol=1e-12, atol=1e-300)


def test_coherence_is_the_mean_cosine_to_the_mean_hand_worked():
    """R7: kappa = mean over tokens of cos(unrotated key, unrotated mean).  Two
    tokens with unrotated keys (1, 0) and (0, 3): the mean is (0.5, 1.5), the
    cosines are 1/sqrt(10) and 3/sqrt(10), so kappa = 2/sqrt(10) and
    m = 2 * kappa = 4/sqrt(10) (|mean| / mean |k| would give 0.79 instead)."""
    u = np.array([[1.0, 0.0], [0.0, 3.0]])
    x = 5
    K = _rot(u, np.arange(x, x + 2))
    pr = O.prototype(K, np.zeros((2, 2)), np.ones(2), x, x + 2, 10000.0, 0.1)
    assert abs(pr.kappa - 2 / math.sqrt(10)) < 1e-12
    assert abs(pr.m - 4 / math.sqrt(10)) < 1e-12


def test_distortion_is_a_mean_over_probe_rows():
    """R4 averages over the probe rows: duplicating every probe row (same query,
    same attention, same LSE) leaves D and D_drop unchanged."""
    e1, e2 = np.array([1.0, 0.0]), np.array([0.0, 1.0])
    Kpost = np.stack([e1, _rot(e2, 1.0), _rot(e1, 2.0), _rot(e2, 3.0)])
    V = np.stack([e1, e2, e1, e2])
    q = np.array([[0.3, -0.2]])
    sc = O.score_head(Kpost, V, q.reshape(1, 1, 2), 4, 1)
    pr = O.prototype(Kpost[0:2], V[0:2], np.array([1.0, 0.5]), 0, 2, 10000.0, 0.1)
    nu = float(sc.feats[:, 1].mean())
    D1, Dd1 = O.node_distortion(sc.a[:, 0:2], V[0:2], q, sc.lse, pr, nu, 0.25, 0.75)
    D2, Dd2 = O.node_distortion(np.repeat(sc.a[:, 0:2], 2, axis=0), V[0:2], np.repeat(q, 2, axis=0),
                                np.repeat(sc.lse, 2), pr, nu, 0.25, 0.75)
    assert abs(D2 - D1) < 1e-14 and abs(Dd2 - Dd1) < 1e-14


def test_value_norm_scale_is_the_mean_over_the_head():
    """R4: the value term divides by nu_bar, the mean |v| over the (l, h)'s
    tokens.  Values of unequal norms (every fourth token 5x longer) make the
    mean differ from other summaries; the head's distortions equal the node
    distortions recomputed with that mean."""
    rng = np.random.default_rng(24)
    n, d, G, P = 200, 16, 2, 8
    K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d)); Q = rng.standard_normal((G, P, d))
    V[::4] *= 5.0
    bounds = np.array([0, 48, 100, 160])
    res = O.score_and_value_head(K, V, Q, n, P, bounds, 1.0, n_hops=0)
    nu = float(np.linalg.norm(V, axis=1).mean())
    sc = O.score_head(K, V, Q, n, P)
    q = Q.reshape(G * P, d)
    for s in range(3):
        for j, (x, y) in enumerate(O.tree_nodes(int(bounds[s]), int(bounds[s + 1]))):
            pr = O.prototype(K[x:y], V[x:y], res.r[x:y], x, y, 10000.0, 0.1)
            D, Dd = O.node_distortion(sc.a[:, x:y], V[x:y], q, sc.lse, pr, nu, 0.25, 0.75)
            assert abs(res.D[s, j] - D) <= 1e-12 * max(1.0, abs(D))
            assert abs(res.Ddrop[s, j] - Dd) <= 1e-12 * max(1.0, abs(Dd))


def test_default_hop_seed_count_is_the_probe_count():
    """R2: each hop seeds from the P tokens (the probe count) of largest relevance."""
    rng = np.random.default_rng(25)
    n, d, G, P = 120, 16, 2, 8
    K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d)); Q = rng.standard_normal((G, P, d))
    res = O.score_and_value_head(K, V, Q, n, P, np.array([0, 48, 96]), 1.0)
    assert [len(s) for s in res.seeds] == [P, P]
