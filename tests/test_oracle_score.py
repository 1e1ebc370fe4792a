"""Pins for the oracle's RoPE, probe scoring / token features and relevance hops.

Each pin checks the oracle against something other than itself: a closed form,
an invariant the method fixes, an independent library routine (torch, float64,
CPU), an independent formulation, or a brute-force loop on a tiny case.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W


# ------------------------------------------------------------------ RoPE
def test_rope_unrotate_rerotate_identity():
    rng = np.random.default_rng(1)
    k = rng.standard_normal((50, 128))
    p = rng.uniform(0, 131072, size=50)
    p[::2] = np.floor(p[::2]) + 0.5          # half-integer representative positions
    back = O.rope_rotate(O.rope_rotate(k, p, 10000.0), -p, 10000.0)
    assert np.abs(back - k).max() <= 1e-12 * np.abs(k).max() * 10


def test_rope_matches_euler_form():
    """Rotate-half RoPE equals multiplying z_j = x_j + i x_{j+d/2} by exp(i p theta_j)
    with theta_j = exp(-(2j/d) ln base) (independent formulation)."""
    rng = np.random.default_rng(2)
    d = 64
    x = rng.standard_normal((7, d))
    p = np.array([0, 1, 2.5, 17, 1000, 4095.5, 65537])
    th = np.exp(-(2.0 * np.arange(d // 2) / d) * math.log(10000.0))
    z = (x[:, :d // 2] + 1j * x[:, d // 2:]) * np.exp(1j * p[:, None] * th[None, :])
    ref = np.concatenate([z.real, z.imag], axis=1)
    # angle conditioning: |d angle| ~ p * 1e-16, so allow 1e-15 * max(p) per unit of |x|
    np.testing.assert_allclose(O.rope_rotate(x, p, 10000.0), ref, rtol=0, atol=1e-15 * p.max() * 8)


def test_rope_closed_form_d2():
    # d = 2 -> theta_0 = 1: (1, 0) rotated by p is (cos p, sin p)
    out = O.rope_rotate(np.array([1.0, 0.0]), 0.7, 10000.0)
    np.testing.assert_allclose(out, [math.cos(0.7), math.sin(0.7)], atol=1e-15)


def test_rope_inverts_generator_keys():
    """Unrotating the generator's post-RoPE keys recovers its pre-RoPE walk
    (the generator rotates with its own complex-number code)."""
    cfg = W.small_config(d=64, dtype="f32", n=300, n_min=300, B=1, L=1, H=1, needles="none")
    bounds = W.planted_bounds(cfg, 0, 300)
    K, V, Q, _ = W.gen_head(cfg, 0, 0, 0, 300, bounds, 0)
    full = np.concatenate([bounds.astype(np.int64), [300]])
    pre = W._walk(W._rng(cfg, 0, 0, 0, W.TAG_K), 300, 64, full)
    back = O.rope_rotate(K, -np.arange(300), cfg.rope_base)
    assert np.abs(back - pre).max() < 1e-5


# ------------------------------------------------------------------ scoring
def _rand_head(n=40, d=16, G=2, P=4, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, d)), rng.standard_normal((n, d)) * 0.7,
            rng.standard_normal((G, P, d)))


def test_attention_rows_normalised_and_alpha_sums_to_one():
    K, V, Q = _rand_head()
    sc = O.score_head(K, V, Q, 40, 4)
    a = sc.a
    np.testing.assert_allclose(a.sum(axis=1), 1.0, atol=1e-13)
    np.testing.assert_allclose(sc.feats[:, 0].sum(), 1.0, atol=1e-13)
    H = sc.feats[:, 3]
    assert (H >= 0).all() and (H <= math.log(40) + 1e-12).all()


def test_causal_mask_uniform_closed_form():
    """Zero queries give uniform attention over exactly the n - P + p + 1 visible keys."""
    n, d, G, P = 30, 8, 3, 5
    K = np.random.default_rng(3).standard_normal((n, d))
    sc = O.score_head(K, K, np.zeros((G, P, d)), n, P)
    for g in range(G):
        for p in range(P):
            vis = n - P + p + 1
            row = sc.a[g * P + p]
            np.testing.assert_allclose(row[:vis], 1.0 / vis, atol=1e-15)
            assert (row[vis:] == 0).all()
            assert abs(sc.lse[g * P + p] - math.log(vis)) < 1e-13
            assert abs(sc.H_rows[g * P + p] - math.log(vis)) < 1e-13


def test_single_key_row_has_unit_mass_zero_entropy():
    K = np.ones((1, 4))
    sc = O.score_head(K, K, np.random.default_rng(0).standard_normal((2, 1, 4)), 1, 1)
    np.testing.assert_allclose(sc.a, 1.0)
    np.testing.assert_allclose(sc.H_rows, 0.0)
    np.testing.assert_allclose(sc.feats[0, 3], 0.0)


def test_alpha_matches_torch_softmax():
    """alpha = mean over rows of torch.softmax(Q K^T / sqrt(d), causal mask), float64."""
    K, V, Q = _rand_head(n=50, d=32, G=4, P=6, seed=5)
    sc = O.score_head(K, V, Q, 50, 6)
    q = torch.tensor(Q.reshape(-1, 32))
    s = q @ torch.tensor(K).T / math.sqrt(32)
    p_of_row = torch.arange(6).repeat(4)
    mask = torch.arange(50)[None, :] > (50 - 6 + p_of_row)[:, None]
    s = s.masked_fill(mask, float("-inf"))
    a = torch.softmax(s, dim=1)
    np.testing.assert_allclose(sc.feats[:, 0], a.mean(0).numpy(), atol=1e-15)
    np.testing.assert_allclose(sc.lse, torch.logsumexp(s, 1).numpy(), atol=1e-13)


def test_features_brute_force_loops():
    """Tiny case computed with explicit Python loops and math.exp / math.log."""
    n, d, G, P = 7, 3, 2, 2
    K, V, Q = _rand_head(n=n, d=d, G=G, P=P, seed=9)
    sc = O.score_head(K, V, Q, n, P)
    R = G * P
    a = [[0.0] * n for _ in range(R)]
    Hr = [0.0] * R
    for g in range(G):
        for p in range(P):
            rho = g * P + p
            vis = [i for i in range(n) if i <= n - P + p]
            ss = {i: sum(Q[g, p, t] * K[i, t] for t in range(d)) / math.sqrt(d) for i in vis}
            z = sum(math.exp(v) for v in ss.values())
            for i in vis:
                a[rho][i] = math.exp(ss[i]) / z
            Hr[rho] = -sum(a[rho][i] * math.log(a[rho][i]) for i in vis)
    for i in range(n):
        alpha = sum(a[r][i] for r in range(R)) / R
        mass = sum(a[r][i] for r in range(R))
        Hi = sum(a[r][i] * Hr[r] for r in range(R)) / mass
        means = [sum(a[g * P + p][i] for p in range(P)) / P for g in range(G)]
        mu = sum(means) / G
        var = sum((m - mu) ** 2 for m in means) / G
        vn = math.sqrt(sum(V[i, t] ** 2 for t in range(d)))
        np.testing.assert_allclose(sc.feats[i], [alpha, vn, var, Hi, i / (n - 1)], rtol=1e-12,
                                   atol=1e-15)


def test_sigma_zero_for_identical_query_heads():
    n, d, P = 20, 8, 3
    rng = np.random.default_rng(4)
    K = rng.standard_normal((n, d))
    q1 = rng.standard_normal((1, P, d))
    sc = O.score_head(K, K, np.repeat(q1, 4, axis=0), n, P)
    assert np.abs(sc.feats[:, 2]).max() < 1e-30


# ------------------------------------------------------------------ hops
def test_zero_hop_weight_gives_alpha():
    K, V, _ = _rand_head(n=60, d=16)
    alpha = np.random.default_rng(1).dirichlet(np.ones(60))
    r, _ = O.hop_relevance(alpha, K, V, 8, 0.0, 2)
    np.testing.assert_array_equal(r, alpha)


def test_all_seed_hop_equals_dense_attention_product():
    """With S_h = n each hop is r0 + w * r^T softmax(V K^T / sqrt d), so two hops
    are r0 + w T r0 + w^2 T T r0 (torch, float64)."""
    n, d = 40, 16
    K, V, _ = _rand_head(n=n, d=d, seed=11)
    alpha = np.random.default_rng(2).dirichlet(np.ones(n))
    A = torch.softmax(torch.tensor(V) @ torch.tensor(K).T / math.sqrt(d), dim=1)
    r0 = torch.tensor(alpha)
    T = lambda r: r @ A  # noqa: E731
    r1, _ = O.hop_relevance(alpha, K, V, n, 0.3, 1)
    np.testing.assert_allclose(r1, (r0 + 0.3 * T(r0)).numpy(), atol=1e-15)
    r2, _ = O.hop_relevance(alpha, K, V, n, 0.3, 2)
    np.testing.assert_allclose(r2, (r0 + 0.3 * T(r0) + 0.09 * T(T(r0))).numpy(), atol=1e-15)


def test_seed_ties_go_to_lower_index():
    x = np.array([0.5, 0.9, 0.9, 0.1, 0.9])
    assert list(O.top_indices(x, 3)) == [1, 2, 4]
    assert list(O.top_indices(x, 2)) == [1, 2]


def test_two_hop_chain_raises_bridge_relevance():
    """A planted B needle (key aligned to needle A's value) gains at least
    0.3 * r(A) * (softmax mass of B under A's value) over its direct alpha."""
    cfg = W.small_config(B=1, L=1, H=1, n=900, n_min=900, dtype="f32")
    wl = W.make_workload(cfg)
    s = wl.seqs[0]
    res = O.score_and_value_head(s.K[0, 0], s.V[0, 0], s.Qp[0, 0:4], s.n, cfg.P, s.slot_bounds, 1.0)
    alpha = res.feats[:, 0]
    d = cfg.d
    checked = 0
    for (_, _, i, kind, a) in s.needles:
        if kind != "B":
            continue
        sc = s.V[0, 0, a].astype(np.float64) @ s.K[0, 0].astype(np.float64).T / math.sqrt(d)
        mass = np.exp(sc - sc.max())
        mass /= mass.sum()
        if a in set(res.seeds[0].tolist()):
            assert res.r[i] - alpha[i] >= 0.3 * alpha[a] * mass[i] * (1 - 1e-9)
            checked += 1
    assert checked > 0


def test_second_hop_seeds_follow_the_first_hop():
    """Hand-built case (R2: hop k seeds from r^(k-1)): token 0 has the largest
    alpha and its value points at token 1's key, so hop 1 moves most of token
    0's relevance onto token 1 (r^1_1 = 0.35 + 0.3 * 0.40 > r^1_0 = 0.40 + ~0);
    with one seed per hop, hop 2 must seed from token 1, not token 0."""
    alpha = np.array([0.40, 0.35, 0.10, 0.10, 0.05])
    K = np.zeros((5, 2)); K[1] = [10.0, 0.0]
    V = np.zeros((5, 2)); V[0] = [10.0, 0.0]
    r, seeds = O.hop_relevance(alpha, K, V, 1, 0.3, 2)
    assert list(seeds[0]) == [0] and list(seeds[1]) == [1]
    # brute force: hop 1 from seed 0, hop 2 from seed 1 (v_1 = 0: uniform softmax)
    sm0 = np.exp(K @ V[0] / np.sqrt(2)); sm0 /= sm0.sum()
    r1 = alpha + 0.3 * alpha[0] * sm0
    assert r1[1] > r1[0]
    r2 = alpha + 0.3 * r1[1] * np.full(5, 0.2)
    np.testing.assert_allclose(r, r2, rtol=1e-12)
