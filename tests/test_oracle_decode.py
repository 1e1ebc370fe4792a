"""Pins for the oracle's ragged decode and the curvature partition."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W


# ------------------------------------------------------------------ decode
def test_full_cache_decode_equals_torch_sdpa():
    """With every entry exact (log m = 0) decode is plain GQA attention
    (torch scaled_dot_product_attention, float64, CPU)."""
    rng = np.random.default_rng(0)
    G, d, n = 4, 64, 77
    q = rng.standard_normal((G, d)); K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d))
    out = O.decode_head(q, K, V, np.zeros(n))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None, :, None, :], torch.tensor(K)[None, None].expand(1, G, n, d),
        torch.tensor(V)[None, None].expand(1, G, n, d))[0, :, 0, :]
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-13)


@pytest.mark.parametrize("seed", range(5))
def test_drop_only_bound(seed):
    """DistillCache 3.1.4: dropping entries of attention mass eps moves the output by
    at most 2 max|v| eps."""
    rng = np.random.default_rng(seed)
    G, d, n = 4, 32, 200
    q = rng.standard_normal((G, d)) * 2
    K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d))
    keep = rng.uniform(size=n) > 0.6
    full = O.decode_head(q, K, V, np.zeros(n))
    part = O.decode_head(q, K[keep], V[keep], np.zeros(keep.sum()))
    s = q @ K.T / math.sqrt(d)
    a = np.exp(s - s.max(1, keepdims=True)); a /= a.sum(1, keepdims=True)
    eps = a[:, ~keep].sum(1)
    C = np.linalg.norm(V, axis=1).max()
    assert (np.linalg.norm(full - part, axis=1) <= 2 * C * eps + 1e-12).all()


def test_append_then_attend():
    """The appended token (multiplicity 1) is attended at the step that appends it."""
    rng = np.random.default_rng(1)
    d = 16
    K = rng.standard_normal((10, d)); V = rng.standard_normal((10, d))
    k_new = rng.standard_normal(d); v_new = rng.standard_normal(d)
    q = (50.0 * k_new / np.linalg.norm(k_new))[None]
    out, K2, V2, lm2 = O.decode_step_head(q, k_new, v_new, K, V, np.zeros(10))
    assert K2.shape[0] == 11 and lm2[-1] == 0.0
    s = q @ K2.T / 4.0
    a = np.exp(s - s.max()); a /= a.sum()
    np.testing.assert_allclose(out[0], (a @ V2)[0], atol=1e-13)
    assert a[0, -1] > 0.99


# ------------------------------------------------------------------ partition (a0)
def test_curvature_on_great_circle_closed_form():
    """Unit states moving at constant angle omega on a great circle: consecutive
    chords of span w meet at angle w*omega, so kappa_w = 1 - cos(w omega)."""
    dim, n, om = 12, 100, 0.02
    rng = np.random.default_rng(2)
    e1 = rng.standard_normal(dim); e1 /= np.linalg.norm(e1)
    e2 = rng.standard_normal(dim); e2 -= (e2 @ e1) * e1; e2 /= np.linalg.norm(e2)
    t = np.arange(n)
    h = np.cos(om * t)[:, None] * e1 + np.sin(om * t)[:, None] * e2
    k = O.curvature(h * 3.0)                           # scaling is removed by normalisation
    exp = np.mean([1 - math.cos(w * om) for w in (1, 2, 4, 8)])
    np.testing.assert_allclose(k[8:n - 8], exp, atol=1e-12)


def test_curvature_right_angle_turn():
    """A path that turns by 90 degrees at t0 has kappa_1(t0) = 1 (cos = 0); states are
    kept on the unit sphere by using tiny steps around a far-away unit point."""
    dim = 6
    base = np.zeros(dim); base[0] = 1.0
    n, t0, eps = 40, 20, 1e-7
    h = np.zeros((n, dim))
    for t in range(n):
        h[t] = base + eps * (np.eye(dim)[1] * min(t, t0) + np.eye(dim)[2] * max(t - t0, 0))
    k = O.curvature(h, scales=(1,))
    assert abs(k[t0] - 1.0) < 1e-6
    assert np.abs(k[1:t0]).max() < 1e-6 and np.abs(k[t0 + 1:n - 1]).max() < 1e-6


def _brute_partition(kappa, end, lmin, lmax, target, lam):
    best = None
    def rec(x, cuts, score):
        nonlocal best
        if x == end:
            if best is None or score > best[0] + 1e-12:
                best = (score, list(cuts))
            return
        for ln in range(lmin, lmax + 1):
            y = x + ln
            if y > end:
                break
            sc = score - lam * ((ln - target) / target) ** 2 + (kappa[y] if y < end else 0.0)
            rec(y, cuts + [y], sc)
    rec(0, [0], 0.0)
    return best


@pytest.mark.parametrize("seed", range(4))
def test_partition_dp_matches_exhaustive_search(seed):
    rng = np.random.default_rng(seed)
    end = 37
    kappa = rng.uniform(size=end + 5) ** 3
    cuts = O.partition_dp(kappa, end, lmin=4, lmax=11, target=7, lam=0.3)
    best = _brute_partition(kappa, end, 4, 11, 7, 0.3)
    score = sum(-0.3 * ((b - a - 7) / 7) ** 2 for a, b in zip(cuts[:-1], cuts[1:])) + \
        sum(kappa[c] for c in cuts[1:-1])
    assert abs(score - best[0]) < 1e-12
    assert list(cuts) == best[1]
    assert all(4 <= b - a <= 11 for a, b in zip(cuts[:-1], cuts[1:]))


def test_partition_recovers_planted_turns():
    """Cuts fall within +-2 tokens of the generator's planted turns."""
    cfg = W.get_config("long").replace(B=1, n=2200, n_min=2200, L=1, H=1, hidden_dim=256)
    planted = W.planted_bounds(cfg, 0, 2200)
    hs = W.hidden_states(cfg, 0, 2200, planted)
    kappa = O.curvature(hs)
    end = int(planted[-1])
    cuts = O.partition_dp(kappa, end)
    assert all(16 <= b - a <= 128 for a, b in zip(cuts[:-1], cuts[1:]))
    inner = planted[1:-1]
    hit = [np.abs(cuts - p).min() <= 2 for p in inner]
    assert np.mean(hit) >= 0.95


def test_partition_default_lambda_hand_worked():
    """kappa = 1 everywhere on [0, 64): the default lambda is the mean curvature,
    1.  Four 16-token slots gain 3 cuts and pay 4 * ((16 - 64)/64)^2 = 2.25:
    +0.75; two 32-token slots 1 - 2 * 0.25 = +0.5; one slot 0; three slots at
    most 2 - 1.33 = +0.67.  So the default gives four slots, while lambda = 2
    (four slots -1.5, two slots 0, one slot 0) keeps the single slot."""
    k = np.ones(80)
    np.testing.assert_array_equal(O.partition_dp(k, 64), [0, 16, 32, 48, 64])
    np.testing.assert_array_equal(O.partition_dp(k, 64, lam=2.0), [0, 64])


def test_curvature_zero_chord_convention():
    """R1: a zero chord (a repeated state) counts as no turn (cos = 1): a
    trajectory that stays put has kappa = 0 everywhere, and a single repeated
    state inside a great-circle walk adds nothing at scale 1 there."""
    h = np.tile(np.array([0.3, -1.2, 0.5]), (24, 1))
    np.testing.assert_array_equal(O.curvature(h), 0.0)
    ang = 0.2 * np.arange(24.0)
    g = np.stack([np.cos(ang), np.sin(ang), np.zeros(24)], axis=1)
    g[12] = g[11]                                       # repeat: chord 11 -> 12 is zero
    k1 = O.curvature(g, scales=(1,))
    assert k1[12] == 0.0 and k1[11] == 0.0             # both involve the zero chord
    np.testing.assert_allclose(k1[5], 1 - np.cos(0.2), rtol=1e-9)
