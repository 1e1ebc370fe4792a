"""The synthetic workloads generated with torch, straight into device memory.

Same recipe as ``synth.workloads`` (per-slot Gaussian random walks with unit
per-element variance, rotate-half RoPE at the integer positions, N(0, I)
probe queries, needle keys aligned to a probe row at cosine 0.9 and two-hop
partners aligned to a needle's value), drawn from torch's counter-based
generator instead of numpy's PCG64, so the numbers differ from the numpy
generator's while the shapes, distributions and structure are the same.  It
exists for workloads too large to build as host arrays (the 64-sequence
serving batch holds 90 GB of bf16 K and V): every sequence is generated on the
target device, all (layer, KV head) pairs at once, and written into the
caller's token-layout tensors.  It runs on any torch device (the CPU for
tests).  Every sequence b draws from its own generator seeded from
(seed, b, tag), so any sequence can be regenerated alone.

Nothing here computes any part of the compression method.
"""
from __future__ import annotations

import math
from typing import Tuple

import numpy as np
import torch

from synth import workloads as W

_TAGS = {"K": 101, "V": 102, "Q": 103, "NEEDLE": 104}


def _gen(cfg, b: int, tag: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(((cfg.seed * 1_000_003 + b) * 1_009 + _TAGS[tag]) & 0x7FFFFFFFFFFFFFFF)
    return g


def _walk(gen, LH: int, n: int, d: int, bounds: torch.Tensor, device) -> torch.Tensor:
    """[LH, n, d] float32: per-segment random walks (unit-variance base, steps of
    sigma 0.1), divided by sqrt(1 + 0.01 t) for unit per-element variance."""
    starts = bounds[:-1]
    lens = bounds[1:] - bounds[:-1]
    seg = torch.repeat_interleave(torch.arange(len(starts), device=device), lens)
    t_in = (torch.arange(n, device=device) - starts[seg]).to(torch.float32)
    x = torch.randn((LH, n, d), generator=gen, device=device, dtype=torch.float32) * 0.1
    x[:, starts] = 0.0
    x = torch.cumsum(x, dim=1)
    x -= x[:, starts][:, seg]
    base = torch.randn((LH, len(starts), d), generator=gen, device=device, dtype=torch.float32)
    x += base[:, seg]
    x /= torch.sqrt(1.0 + 0.01 * t_in)[None, :, None]
    return x


def _rope(x: torch.Tensor, base: float) -> torch.Tensor:
    """Rotate-half RoPE at positions 0..n-1 (angles in float64)."""
    n, d = x.shape[-2], x.shape[-1]
    half = d // 2
    inv = base ** (-2.0 * torch.arange(half, dtype=torch.float64, device=x.device) / d)
    ang = torch.arange(n, dtype=torch.float64, device=x.device)[:, None] * inv[None, :]
    c, s = torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)
    a, b = x[..., :half], x[..., half:]
    return torch.cat([a * c - b * s, a * s + b * c], dim=-1)


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)


def _align(norm: torch.Tensor, target: torch.Tensor, noise: torch.Tensor) -> torch.Tensor:
    """norm * (0.9 t^ + sqrt(0.19) u), u the unit part of `noise` orthogonal to t^."""
    th = _unit(target)
    u = noise - (noise * th).sum(-1, keepdim=True) * th
    return norm * (0.9 * th + math.sqrt(0.19) * _unit(u))


def gen_sequence(cfg, b: int, n: int, bounds: np.ndarray, counts: np.ndarray, device,
                 dtype=torch.bfloat16) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """K, V [L*H, n, d] and Qp [L, H*G, P, d] of sequence b in `dtype` on `device`.
    ``bounds``: the slot boundaries over [0, n - W); ``counts`` [L*H]: needles per
    (l, h) (half aligned to a probe row, half to such a needle's value; as in
    ``synth.workloads.gen_head`` for 'pairs' and 'zipf', all probe-aligned for
    'tiny')."""
    LH, d, G, P = cfg.L * cfg.H, cfg.d, cfg.G, cfg.P
    full = np.asarray(bounds, np.int64)
    if full[-1] != n:
        full = np.concatenate([full, [n]])
    bd = torch.as_tensor(full, device=device)
    V = _walk(_gen(cfg, b, "V", device), LH, n, d, bd, device)
    K = _rope(_walk(_gen(cfg, b, "K", device), LH, n, d, bd, device), cfg.rope_base)
    Q = torch.randn((LH, G * P, d), generator=_gen(cfg, b, "Q", device), device=device)
    Q = Q.to(dtype).to(torch.float32)
    V = V.to(dtype).to(torch.float32)
    cnt = torch.as_tensor(np.asarray(counts, np.int64), device=device)
    c_max = int(cnt.max()) if LH else 0
    if c_max > 0:
        gn = _gen(cfg, b, "NEEDLE", device)
        end = n - cfg.W
        pos = torch.rand((LH, end), generator=gn, device=device).topk(c_max, dim=1).indices
        n_a = cnt if cfg.needles == "tiny" else (cnt + 1) // 2
        j = torch.arange(c_max, device=device)[None, :]
        is_a = j < n_a[:, None]
        valid = j < cnt[:, None]
        rows = torch.arange(LH, device=device)[:, None].expand(LH, c_max)
        # partner of B needle j: A needle (j - n_a) mod n_a
        a_idx = torch.remainder(j - n_a[:, None], torch.clamp(n_a, min=1)[:, None])
        a_pos = torch.gather(pos, 1, a_idx)
        qrow = torch.randint(0, G * P, (LH, c_max), generator=gn, device=device)
        noise = torch.randn((LH, c_max, d), generator=gn, device=device)
        knorm = torch.linalg.vector_norm(K[rows, pos], dim=-1, keepdim=True)
        target = torch.where(is_a[..., None], Q[rows, qrow], V[rows, a_pos])
        newk = _align(knorm, target, noise)
        sel = valid
        K[rows[sel], pos[sel]] = newk[sel]
    return (K.to(dtype), V.to(dtype), Q.reshape(cfg.L, cfg.H * G, P, d).to(dtype))


def fill_workload(cfg, K: torch.Tensor, V: torch.Tensor, Qp: torch.Tensor, dtype=torch.bfloat16):
    """Generates every sequence of ``cfg`` into the token-layout tensors K, V
    ([sum_b L*H*n_b, d]) and Qp ([B, L, H*G, P, d]) on their device.  Returns
    (context lengths [B], slot bounds per sequence)."""
    ns = W.context_lengths(cfg)
    bounds = []
    row = 0
    for b, n in enumerate(ns):
        n = int(n)
        pb = W.planted_bounds(cfg, b, n)
        k, v, q = gen_sequence(cfg, b, n, pb, W._needle_counts(cfg, b, n), K.device, dtype)
        m = cfg.L * cfg.H * n
        K[row:row + m] = k.reshape(m, cfg.d)
        V[row:row + m] = v.reshape(m, cfg.d)
        Qp[b] = q
        row += m
        bounds.append(pb)
        del k, v, q
    return ns, bounds


def decode_inputs(cfg, steps: int, device, dtype=torch.bfloat16, B=None):
    """Decode-step inputs of `steps` steps on `device`, N(0, 1) in `dtype`:
    q [steps, B, L, H*G, d], k_new and v_new [steps, B, L, H, d]."""
    B = cfg.B if B is None else B
    g = torch.Generator(device=device)
    g.manual_seed((cfg.seed * 1_000_003 + 7_919) & 0x7FFFFFFFFFFFFFFF)
    shp_q = (B, cfg.L, cfg.H * cfg.G, cfg.d)
    shp_kv = (B, cfg.L, cfg.H, cfg.d)
    q = torch.empty((steps,) + shp_q, device=device, dtype=dtype)
    k = torch.empty((steps,) + shp_kv, device=device, dtype=dtype)
    v = torch.empty((steps,) + shp_kv, device=device, dtype=dtype)
    for t in range(steps):                     # one step at a time: no float32 copy of all
        q[t] = torch.randn(shp_q, generator=g, device=device, dtype=torch.float32)
        k[t] = torch.randn(shp_kv, generator=g, device=device, dtype=torch.float32)
        v[t] = torch.randn(shp_kv, generator=g, device=device, dtype=torch.float32)
    return q, k, v


def hidden_states(cfg, b: int, n: int, planted: np.ndarray, device, dtype=torch.bfloat16,
                  noise: float = 0.002) -> torch.Tensor:
    """Piecewise-smooth hidden-state trajectory [n, hidden_dim] with turns at
    ``planted`` (the recipe of ``synth.workloads.hidden_states``): the state
    moves on the sphere of radius sqrt(dim) along a great circle at 0.02..0.06
    rad per token; each boundary starts a new great circle through the
    current state in a random direction.  Built in float64, rounded to `dtype`;
    the segments' start states are chained in a short loop."""
    dim = cfg.hidden_dim
    g = torch.Generator(device=device)
    g.manual_seed(((cfg.seed * 1_000_003 + b) * 1_009 + 105) & 0x7FFFFFFFFFFFFFFF)
    full = np.asarray(planted, np.int64)
    if full[-1] != n:
        full = np.concatenate([full, [n]])
    S = len(full) - 1
    rho = float(np.sqrt(dim))
    e2s = torch.randn((S, dim), generator=g, device=device, dtype=torch.float64)
    oms = 0.02 + 0.04 * torch.rand((S,), generator=g, device=device, dtype=torch.float64)
    cur = _unit(torch.randn((dim,), generator=g, device=device, dtype=torch.float64))
    lens = np.diff(full)
    starts = torch.empty((S, dim), device=device, dtype=torch.float64)
    dirs = torch.empty((S, dim), device=device, dtype=torch.float64)
    for s_ in range(S):
        e2 = _unit(e2s[s_] - (e2s[s_] @ cur) * cur)
        starts[s_], dirs[s_] = cur, e2
        ang = oms[s_] * float(lens[s_])
        cur = _unit(torch.cos(ang) * cur + torch.sin(ang) * e2)
    seg = torch.repeat_interleave(torch.arange(S, device=device),
                                  torch.as_tensor(lens, device=device))
    t_in = (torch.arange(n, device=device) -
            torch.as_tensor(full[:-1], device=device)[seg]).to(torch.float64)
    ang = oms[seg] * t_in
    h = rho * (torch.cos(ang)[:, None] * starts[seg] + torch.sin(ang)[:, None] * dirs[seg])
    h += noise * torch.randn((n, dim), generator=g, device=device, dtype=torch.float64)
    return h.to(torch.float32).to(dtype)
