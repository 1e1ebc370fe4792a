"""Pins for the oracle's per-step top-B eviction (DistillCache Algorithm 1 with the
heuristic score alpha, reading R17)."""
import math

import numpy as np
import pytest
import torch

import oracle as O


def test_budget_closed_forms():
    assert O.evict_budget(100, 0.25, 32) == 32            # the minimum budget binds
    assert O.evict_budget(16384, 0.25, 32) == 4096
    assert O.evict_budget(16385, 0.25, 32) == 4096        # floor
    assert O.evict_budget(131, 0.25, 32) == 32
    assert O.evict_budget(200, 0.25, 32) == 50


@pytest.mark.parametrize("seed", range(5))
def test_top_b_is_a_brute_force_sort_with_ties_to_the_lower_index(seed):
    rng = np.random.default_rng(seed)
    s = rng.choice([0.0, 0.1, 0.25, 0.5], size=57)          # many ties
    for B in (0, 1, 7, 20, 57, 80):
        want = sorted(sorted(range(len(s)), key=lambda i: (-s[i], i))[:B])
        np.testing.assert_array_equal(O.top_b(s, B), want)


def _cache(rng, L=2, H=2, c=50, d=16):
    K = rng.standard_normal((L, H, c, d))
    V = rng.standard_normal((L, H, c, d))
    return K, V


@pytest.mark.parametrize("seed", range(4))
def test_alpha_is_the_mean_attention_probability(seed):
    rng = np.random.default_rng(seed)
    L, H, G, c, d = 2, 2, 3, 40, 16
    K, V = _cache(rng, L, H, c, d)
    q = rng.standard_normal((L, H * G, d))
    kn, vn = rng.standard_normal((L, H, d)), rng.standard_normal((L, H, d))
    out, alpha, keep = O.evict_step(q, kn, vn, K, V, 200, 0.25, 8)
    assert alpha.shape == (c + 1,)
    assert abs(alpha.sum() - 1.0) < 1e-12
    acc = torch.zeros(c + 1, dtype=torch.float64)
    for l in range(L):
        for h in range(H):
            Kc = torch.from_numpy(np.concatenate([K[l, h], kn[l, h][None]]))
            qq = torch.from_numpy(q[l, h * G:(h + 1) * G])
            acc += torch.softmax(qq @ Kc.T / math.sqrt(d), dim=-1).sum(0)
    np.testing.assert_allclose(alpha, (acc / (L * H * G)).numpy(), rtol=1e-12, atol=1e-15)
    # the step's output is the a7 decode over the appended cache
    for l in range(L):
        for h in range(H):
            o4, *_ = O.decode_step_head(q[l, h * G:(h + 1) * G], kn[l, h], vn[l, h], K[l, h], V[l, h],
                                        np.zeros(c))
            np.testing.assert_allclose(out[l, h * G:(h + 1) * G], o4, rtol=1e-12, atol=1e-12)
    assert len(keep) == min(O.evict_budget(200, 0.25, 8), c + 1) and (np.diff(keep) > 0).all()


@pytest.mark.parametrize("seed", range(4))
def test_eviction_error_bound(seed):
    """[DC] 3.1.4: attention renormalised over the kept entries differs from the
    full attention by at most 2 C eps (C = max |v|, eps = evicted mass)."""
    rng = np.random.default_rng(seed)
    L, H, G, c, d = 1, 1, 1, 60, 8
    K, V = _cache(rng, L, H, c, d)
    q = rng.standard_normal((L, H * G, d)) * 2.0
    kn, vn = rng.standard_normal((L, H, d)), rng.standard_normal((L, H, d))
    out, alpha, keep = O.evict_step(q, kn, vn, K, V, 80, 0.25, 4)
    Kc = np.concatenate([K[0, 0], kn[0, 0][None]])
    Vc = np.concatenate([V[0, 0], vn[0, 0][None]])
    sub = O.decode_head(q[0], Kc[keep], Vc[keep], np.zeros(len(keep)))
    eps = 1.0 - alpha[keep].sum()                  # one query head: alpha = its probabilities
    C = np.linalg.norm(Vc, axis=1).max()
    assert np.linalg.norm(out[0, 0] - sub[0]) <= 2 * C * eps + 1e-12


def test_keep_everything_when_the_budget_covers_the_cache():
    rng = np.random.default_rng(0)
    K, V = _cache(rng, 1, 2, 10, 8)
    q = rng.standard_normal((1, 4, 8))
    kn, vn = rng.standard_normal((1, 2, 8)), rng.standard_normal((1, 2, 8))
    _, _, keep = O.evict_step(q, kn, vn, K, V, 40, 0.5, 32)
    np.testing.assert_array_equal(keep, np.arange(11))
