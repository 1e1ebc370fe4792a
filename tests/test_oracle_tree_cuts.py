"""Pins for the oracle's curvature-chosen prototype trees (GraceKV "Technical
details and default settings": tree construction considers high-curvature split
candidates plus the midpoint; the curvature measure of "01 Curvature-guided
partition").  Reading R18: per-(layer, KV head) curvature of the unrotated key
trajectory; each internal node cut at the valid position maximising curvature
minus the partition's length-balance penalty."""
import numpy as np
import pytest

import oracle as O
from oracle import kvc_oracle as OK

BASE = 10000.0


def _great_circle_keys(n, d, phi, rng):
    """Keys whose RoPE-removed trajectory runs along a great circle at a constant
    angular step phi, each key scaled by a random positive factor."""
    e = np.linalg.qr(rng.standard_normal((d, 2)))[0]
    i = np.arange(n, dtype=np.float64)
    u = np.cos(i * phi)[:, None] * e[:, 0] + np.sin(i * phi)[:, None] * e[:, 1]
    u *= rng.uniform(0.5, 2.0, size=(n, 1))
    return O.rope_rotate(u, i, BASE)                 # post-RoPE keys


def test_key_curvature_great_circle_closed_form():
    """Chords of a great circle at step w*phi meet at the angle w*phi, so
    kappa_w = 1 - cos(w*phi) wherever every scale fits (t in [8, n - 8))."""
    rng = np.random.default_rng(0)
    n, phi = 96, 0.07
    kap = O.key_curvature(_great_circle_keys(n, 64, phi, rng), BASE)
    want = np.mean([1.0 - np.cos(w * phi) for w in (1, 2, 4, 8)])
    np.testing.assert_allclose(kap[8:n - 8], want, rtol=1e-9, atol=1e-12)
    # only scale 1 fits at t = 1
    np.testing.assert_allclose(kap[1], 1.0 - np.cos(phi), rtol=1e-9)
    assert kap[0] == 0.0 and kap[n - 1] == 0.0


def test_key_curvature_removes_rope_rotation():
    """The same great-circle keys measured without removing RoPE do not give the
    closed form: the per-pair rotation at different frequencies bends the
    trajectory, so a sign or angle error in the inverse rotation fails the
    closed-form test above."""
    rng = np.random.default_rng(1)
    n, phi = 96, 0.07
    K = _great_circle_keys(n, 64, phi, rng)
    want = np.mean([1.0 - np.cos(w * phi) for w in (1, 2, 4, 8)])
    assert np.abs(O.curvature(K)[8:n - 8] - want).max() > 1e-3
    twice = O.curvature(O.rope_rotate(K, np.arange(n), BASE))       # R(+i) instead of R(-i)
    assert np.abs(twice[8:n - 8] - want).max() > 1e-3


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_flat_curvature_gives_the_midpoint_tree(dtype):
    """Constant curvature: every score is kappa - kappa * r^2, largest at the
    midpoint, so the tree is the midpoint tree of reading R3."""
    for c in (16, 17, 31, 64, 100, 127, 128):
        for val in (0.0, 0.3):
            kap = np.full(300, val)
            cuts = O.tree_cuts(kap, 50, 50 + c, dtype)
            assert O.tree_nodes(50, 50 + c, cuts) == O.tree_nodes(50, 50 + c)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_single_turn_hand_worked(dtype):
    """Slot [0, 64) with one turn kappa[20] = 1: the root is cut at 20 (score
    1 - (1/64)(12/32)^2 > 0 at the midpoint); the turn sits at the start of the
    right child, where it is no valid cut, so everything below is cut at
    midpoints: [0,20) at 10, [20,64) at 42, then 5, 15, 31, 53."""
    kap = np.zeros(64)
    kap[20] = 1.0
    assert O.tree_cuts(kap, 0, 64, dtype) == [20, 10, 42, 5, 15, 31, 53]


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_turn_against_balance_hand_worked(dtype):
    """Background 0.5 and a turn of 0.6: lam = (63*0.5 + 0.6)/64 = 0.5015625.
    At t = 28 the score 0.6 - lam/64 = 0.592 beats the midpoint's 0.5; at t = 10
    the penalty lam*(22/32)^2 = 0.237 leaves 0.363 and the midpoint wins."""
    kap = np.full(64, 0.5)
    kap[28] = 0.6
    assert O.tree_cuts(kap, 0, 64, dtype)[0] == 28
    kap = np.full(64, 0.5)
    kap[10] = 0.6
    assert O.tree_cuts(kap, 0, 64, dtype)[0] == 32


def test_full_slot_leaves_no_freedom():
    """A 128-token slot with leaves of at most 16 tokens is the midpoint tree
    whatever the curvature."""
    rng = np.random.default_rng(2)
    for _ in range(5):
        kap = rng.uniform(0, 2, 200)
        assert O.tree_nodes(30, 158, O.tree_cuts(kap, 30, 158)) == O.tree_nodes(30, 158)


def _valid(leaves, size):
    return O.LEAF_MIN * leaves <= size <= O.LEAF_MAX * leaves


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_random_curvature_trees_are_valid_and_optimal(dtype):
    """Random spiky curvature: every tree partitions its slot, every node keeps
    LEAF_MIN..LEAF_MAX tokens per leaf below it, and each cut's
    score is at least that of every other valid cut of its node (brute force)."""
    rng = np.random.default_rng(3)
    f = np.dtype(dtype).type
    for _ in range(60):
        c = int(rng.integers(16, 129))
        x0 = int(rng.integers(0, 40))
        kap = rng.uniform(0, 0.2, x0 + c + 10) + (rng.uniform(size=x0 + c + 10) < 0.05) * 1.5
        cuts = O.tree_cuts(kap, x0, x0 + c, dtype)
        nodes = O.tree_nodes(x0, x0 + c, cuts)
        assert [b - a for a, b in nodes[7:]] and sum(b - a for a, b in nodes[7:]) == c
        for j, (a, b) in enumerate(nodes):
            depth = 0 if j == 0 else 1 if j < 3 else 2 if j < 7 else 3
            assert _valid(2 ** (3 - depth), b - a), (j, a, b)
        k32 = kap.astype(dtype)
        for j in range(7):
            a, b = nodes[j]
            lo = 2 ** (2 - (0 if j == 0 else 1 if j < 3 else 2))
            m = (a + b) // 2
            acc = f(0)
            for i in range(a, b):
                acc = f(acc + k32[i])
            lam = f(acc / f(b - a))
            sc = lambda t: f(k32[t] - f(lam * f(f(f(t - m) / f(f(b - a) * f(0.5))) ** 2)))  # noqa: E731
            best = sc(cuts[j])
            for t in range(a + 1, b):
                if _valid(lo, t - a) and _valid(lo, b - t):
                    assert sc(t) <= best
                    if t < cuts[j] and t != m:
                        assert sc(t) < best or cuts[j] == m   # ties: midpoint, then smaller t


def test_invalid_cuts_are_rejected():
    with pytest.raises(ValueError):
        O.tree_nodes(0, 64, [0, 16, 48, 8, 24, 40, 56])


def test_curvature_trees_keep_pack_and_floor_invariants():
    """With any valid cuts: all ops taken packs the slot's tokens in order; only
    Add taken packs one root prototype; a floor token's path ends at its leaf."""
    rng = np.random.default_rng(4)
    n, d, W = 160, 16, 16
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    r = rng.uniform(0.01, 1, n)
    bounds = np.asarray([0, 40, 96, 144])
    kap = O.key_curvature(K, BASE) + (rng.uniform(size=n) < 0.1)
    cuts = O.slot_cuts(kap, bounds)
    t_all = np.ones((3, O.N_OPS), bool)
    Kp, Vp, lm, ps = O.pack_head(K, V, r, bounds, t_all, n, W, BASE, 0.1, cuts)
    np.testing.assert_array_equal(Kp, K)
    np.testing.assert_array_equal(ps, np.arange(n))
    t_add = np.zeros((3, O.N_OPS), bool)
    t_add[:, 0] = True
    Kp, Vp, lm, ps = O.pack_head(K, V, r, bounds, t_add, n, W, BASE, 0.1, cuts)
    np.testing.assert_allclose(ps[:3], [(0 + 39) / 2, (40 + 95) / 2, (96 + 143) / 2])
    for s in range(3):
        x0, y0 = int(bounds[s]), int(bounds[s + 1])
        nodes = O.tree_nodes(x0, y0, cuts[s])
        for i in range(x0, y0):
            leaf, path = OK._leaf_of(i, x0, y0, cuts[s])
            assert nodes[leaf][0] <= i < nodes[leaf][1] and path[-1] == leaf
            assert all(nodes[a][0] <= nodes[b][0] and nodes[b][1] <= nodes[a][1]
                       for a, b in zip(path, path[1:]))


def test_sixteen_token_slot_is_always_the_midpoint_tree():
    """Leaves keep at least 2 tokens (R18), so a 16-token slot (8 leaves) has
    exactly one valid tree, the midpoint tree, whatever the curvature: a turn
    at token 5 that would win with 1-token leaves (root children of 5 and 11)
    cannot move the root cut from 8."""
    k = np.zeros(20)
    k[5] = 1.0
    for dtype in (np.float64, np.float32):
        assert O.tree_cuts(k, 0, 16, dtype) == [8, 4, 12, 2, 6, 10, 14]
