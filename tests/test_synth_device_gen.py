"""The torch generator of the synthetic workloads (run on the CPU here): the
recipe's structure holds — per-slot random walks with unit variance and steps
of sigma 0.1, RoPE at the integer positions, needles at cosine 0.9 to a probe
row (A) or to a needle's value (B) — and each sequence is reproducible."""
import math

import numpy as np
import torch

from synth import device_gen as DG
from synth import workloads as W


def _cfg(**kw):
    return W.small_config(B=2, L=2, H=2, n=900, n_min=700, d=128, P=16, W=32, needle_frac=0.02,
                          **kw)


def _unrope(x, base):
    n, d = x.shape[-2], x.shape[-1]
    half = d // 2
    inv = base ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = torch.arange(n, dtype=torch.float64)[:, None] * inv[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    a, b = x[..., :half].double(), x[..., half:].double()
    return torch.cat([a * c + b * s, -a * s + b * c], dim=-1)


def test_walk_structure_and_variance():
    cfg = _cfg()
    n = 900
    pb = W.planted_bounds(cfg, 0, n)
    K, V, Q = DG.gen_sequence(cfg, 0, n, pb, np.zeros(cfg.L * cfg.H, np.int64), "cpu",
                              dtype=torch.float32)
    assert K.shape == (4, n, 128) and V.shape == (4, n, 128) and Q.shape == (2, 8, 16, 128)
    full = np.r_[pb, n] if pb[-1] != n else pb
    for X in (V.double(), _unrope(K, cfg.rope_base)):
        assert abs(float(X.var()) - 1.0) < 0.05
        steps = []
        for a, b in zip(full[:-1], full[1:]):
            t = torch.arange(b - a, dtype=torch.float64)
            raw = X[:, a:b] * torch.sqrt(1.0 + 0.01 * t)[None, :, None]
            steps.append((raw[:, 1:] - raw[:, :-1]).reshape(-1))
        assert abs(float(torch.cat(steps).std()) - 0.1) < 0.005
    assert abs(float(Q.double().var()) - 1.0) < 0.05


def test_needles_sit_at_cosine_0_9():
    cfg = _cfg()
    n = 900
    pb = W.planted_bounds(cfg, 1, n)
    counts = np.array([6, 5, 1, 0])
    K, V, Q = DG.gen_sequence(cfg, 1, n, pb, counts, "cpu", dtype=torch.float32)
    q = Q.reshape(4, -1, 128).double()
    for lh, c in enumerate(counts):
        k = K[lh].double()
        kn = k / k.norm(dim=-1, keepdim=True)
        cq = (kn @ (q[lh] / q[lh].norm(dim=-1, keepdim=True)).T).max(dim=1).values
        va = V[lh].double()
        cv = (kn @ (va / va.norm(dim=-1, keepdim=True)).T).max(dim=1).values
        n_a = (c + 1) // 2
        a_hits = torch.nonzero(cq > 0.85).reshape(-1)
        b_hits = torch.nonzero(cv > 0.85).reshape(-1)
        assert len(a_hits) == n_a and len(b_hits) == c - n_a
        assert torch.allclose(cq[a_hits], torch.full_like(cq[a_hits], 0.9), atol=1e-5)
        # a B needle's partner value has neighbours in its slot walk that are
        # nearly parallel to it, so the best match is at least 0.9
        assert bool((cv[b_hits] >= 0.9 - 1e-5).all() and (cv[b_hits] < 0.95).all())
        assert all(int(i) < n - cfg.W for i in torch.cat([a_hits, b_hits]))


def test_fill_workload_is_reproducible_per_sequence():
    cfg = _cfg()
    ns = W.context_lengths(cfg)
    rows = int(ns.sum()) * cfg.L * cfg.H
    bufs = []
    for _ in range(2):
        K = torch.zeros((rows, 128), dtype=torch.bfloat16)
        V = torch.zeros_like(K)
        Qp = torch.zeros((cfg.B, cfg.L, cfg.H * cfg.G, cfg.P, 128), dtype=torch.bfloat16)
        ns2, bounds = DG.fill_workload(cfg, K, V, Qp)
        bufs.append((K, V, Qp))
    assert np.array_equal(ns, ns2) and len(bounds) == cfg.B
    for a, b in zip(*bufs):
        assert torch.equal(a, b)
    K = bufs[0][0]
    n0 = int(ns[0]) * cfg.L * cfg.H
    k1, _, _ = DG.gen_sequence(cfg, 1, int(ns[1]), bounds[1],
                               W._needle_counts(cfg, 1, int(ns[1])), "cpu")
    assert torch.equal(K[n0:n0 + k1.numel() // 128], k1.reshape(-1, 128))
    assert not torch.equal(K[:128], K[n0:n0 + 128])
    assert math.isfinite(float(K.float().abs().max()))


def test_hidden_states_turn_at_the_planted_boundaries():
    """The oracle's curvature (a0) is far larger at the planted turns than elsewhere."""
    import oracle as O
    cfg = W.get_config("long").replace(hidden_dim=256)
    n = 2000
    pb = W.planted_bounds(cfg, 0, n)
    h = DG.hidden_states(cfg, 0, n, pb, "cpu", dtype=torch.float32).double().numpy()
    assert h.shape == (n, 256)
    k = O.curvature(h)
    turns = pb[1:-1]
    assert k[turns].mean() > 5 * k.mean()
    others = np.setdiff1d(np.arange(16, n - 16), np.concatenate([turns + o for o in range(-9, 10)]))
    assert np.quantile(k[others], 0.99) < k[turns].min()
