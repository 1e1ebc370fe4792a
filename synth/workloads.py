"""Seeded synthetic workloads shaped like the pages' evaluation settings.

The pages evaluate on LongBench / RULER with Mistral-7B, Qwen2.5-7B and
Llama-3-8B.  Neither those datasets nor the weights are available, so these
generators stand in for them with caches of the same shapes:

* post-RoPE keys and values built as per-slot Gaussian random walks
  (unit-variance base, step sigma 0.1, renormalised to unit per-element
  variance), keys rotated with the rotate-half RoPE convention at their
  integer positions;
* probe queries N(0, I), already post-RoPE;
* planted "needle" keys: a key is replaced (keeping its norm) by
  0.9 * (unit probe query) + sqrt(0.19) * (unit vector orthogonal to it), and
  for two-hop chains a second key is aligned the same way to the first
  needle's value;
* seeded slot boundaries (fixed 64-token, U{16..112}, or planted turns of a
  piecewise-smooth hidden-state trajectory for the curvature partition).

Every (sequence, layer, KV head) triple draws from its own counter-derived
stream (numpy PCG64 seeded through SeedSequence([seed, b, l, h, tag])), so any
subset of heads can be regenerated without generating the rest.

Nothing here computes any part of the compression method.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

TAG_K, TAG_V, TAG_Q, TAG_NEEDLE, TAG_SLOTS, TAG_CTX, TAG_ZIPF, TAG_DEC, TAG_HID = range(1, 10)


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    L: int
    H: int            # KV heads
    G: int            # query heads per KV head
    d: int            # head dim
    n: int            # context length (maximum for ragged batches)
    n_min: int        # minimum context length (== n unless ragged)
    dtype: str        # 'f32' | 'bf16'
    P: int            # probe positions (last P queries)
    W: int            # exact recent window
    budget_ratio: float
    budget_entries_per_lh: int   # > 0 overrides budget_ratio
    floor_cap_frac: float
    floor_cap_tokens: int        # < 0: no token cap
    slots: str        # 'fixed64' | 'uniform' | 'curvature'
    needles: str      # 'tiny' | 'pairs' | 'zipf' | 'none'
    needle_frac: float
    n_decode: int
    rope_base: float = 10000.0
    hop_weight: float = 0.3
    n_hops: int = 2
    w_part: float = 0.25
    w_value: float = 0.75
    value_floor: float = 0.10
    seed: int = 0
    hidden_dim: int = 4096
    description: str = ""

    @property
    def R(self) -> int:
        return self.G * self.P

    @property
    def decode_reserve(self) -> int:
        return self.n_decode

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": Config(
        name="tiny", B=1, L=1, H=2, G=4, d=64, n=512, n_min=512, dtype="f32", P=32, W=32,
        budget_ratio=0.25, budget_entries_per_lh=0, floor_cap_frac=1.0, floor_cap_tokens=8,
        slots="fixed64", needles="tiny", needle_frac=0.0, n_decode=8,
        description="1 layer, 2 KV / 8 query heads, d 64, context 512, fp32, 32 probes, "
                    "fixed 64-token slots, 25% budget incl. 32-token window, singleton cap 8"),
    "mistral16k": Config(
        name="mistral16k", B=1, L=32, H=8, G=4, d=128, n=16384, n_min=16384, dtype="bf16",
        P=64, W=128, budget_ratio=0.25, budget_entries_per_lh=0, floor_cap_frac=0.01,
        floor_cap_tokens=-1, slots="uniform", needles="pairs", needle_frac=0.005, n_decode=256,
        description="Mistral-7B-shaped cache: 32 layers, 8 KV / 32 query heads, d 128, bf16, "
                    "batch 1, context 16384, 64 probes, slots U{16..112}, 25% budget with "
                    "128-token window, 1% singleton cap, 0.5% needles with two-hop chains, "
                    "256 decode steps"),
    "long": Config(
        name="long", B=4, L=32, H=8, G=4, d=128, n=32768, n_min=32768, dtype="bf16",
        P=64, W=128, budget_ratio=0.10, budget_entries_per_lh=0, floor_cap_frac=0.6,
        floor_cap_tokens=-1, slots="curvature", needles="pairs", needle_frac=0.005,
        n_decode=1024,
        description="long context: batch 4 x 32768, 10% budget, curvature-chosen slots from "
                    "d=4096 hidden-state trajectories with turns every 64+-16 tokens"),
    "aggressive": Config(
        name="aggressive", B=1, L=32, H=8, G=4, d=128, n=131072, n_min=131072, dtype="bf16",
        P=64, W=256, budget_ratio=0.0, budget_entries_per_lh=1024, floor_cap_frac=0.6,
        floor_cap_tokens=-1, slots="uniform", needles="zipf", needle_frac=0.005, n_decode=512,
        description="aggressive: context 131072 compressed 128x (1024 entries per layer-head "
                    "incl. a 256-token window), Zipf(1.1) needle placement across heads"),
    "serving": Config(
        name="serving", B=64, L=32, H=8, G=4, d=128, n=16384, n_min=4096, dtype="bf16",
        P=64, W=128, budget_ratio=0.25, budget_entries_per_lh=0, floor_cap_frac=0.01,
        floor_cap_tokens=-1, slots="uniform", needles="pairs", needle_frac=0.005, n_decode=512,
        description="serving batch: 64 sequences with contexts U{4096..16384}, 25% budget"),
}


def get_config(name: str) -> Config:
    return CONFIGS[name]


def small_config(**kw) -> Config:
    """A multi-tile, ragged bf16 case that the CPU oracle finishes in seconds."""
    base = Config(
        name="small", B=2, L=2, H=2, G=4, d=128, n=1500, n_min=1100, dtype="bf16", P=64, W=128,
        budget_ratio=0.25, budget_entries_per_lh=0, floor_cap_frac=0.05, floor_cap_tokens=-1,
        slots="uniform", needles="pairs", needle_frac=0.01, n_decode=4,
        description="small ragged bf16 parity case")
    return base.replace(**kw)


# --------------------------------------------------------------------------- helpers

def _rng(cfg: Config, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg.seed, *key])))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _to_dtype(cfg: Config, x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float32)
    return round_bf16(x) if cfg.dtype == "bf16" else x


def _post_rope(x_pre: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Apply rotary position embedding (rotate-half pairing j <-> j + d/2).

    Written as complex multiplication: z_j = x_j + i x_{j+d/2} is multiplied
    by exp(i * pos * base^(-2j/d)).
    """
    d = x_pre.shape[-1]
    half = d // 2
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    phase = np.exp(1j * (pos.astype(np.float64)[:, None] * inv[None, :]))
    z = (x_pre[..., :half].astype(np.float64) + 1j * x_pre[..., half:].astype(np.float64)) * phase
    return np.concatenate([z.real, z.imag], axis=-1).astype(np.float32)


def _walk(rng: np.random.Generator, n: int, d: int, seg_bounds: np.ndarray) -> np.ndarray:
    """Per-segment Gaussian random walk with unit per-element variance."""
    starts = seg_bounds[:-1].astype(np.int64)
    lens = np.diff(seg_bounds).astype(np.int64)
    steps = rng.standard_normal((n, d), dtype=np.float32) * np.float32(0.1)
    base = rng.standard_normal((len(starts), d), dtype=np.float32)
    steps[starts] = 0.0
    cs = np.cumsum(steps, axis=0, dtype=np.float32)
    seg_id = np.repeat(np.arange(len(starts)), lens)
    cs -= cs[starts][seg_id]
    t_in = (np.arange(n) - starts[seg_id]).astype(np.float32)
    x = base[seg_id] + cs
    x /= np.sqrt(np.float32(1.0) + np.float32(0.01) * t_in)[:, None]
    return x


def _unit_orth(rng: np.random.Generator, u: np.ndarray) -> np.ndarray:
    g = rng.standard_normal(u.shape[0]).astype(np.float64)
    g -= (g @ u) * u
    return g / np.linalg.norm(g)


# --------------------------------------------------------------------------- structure

def context_lengths(cfg: Config) -> np.ndarray:
    if cfg.n_min == cfg.n:
        return np.full(cfg.B, cfg.n, dtype=np.int64)
    r = _rng(cfg, TAG_CTX)
    return r.integers(cfg.n_min, cfg.n + 1, size=cfg.B).astype(np.int64)


def planted_bounds(cfg: Config, b: int, n: int) -> np.ndarray:
    """Slot boundaries over the compressible region [0, n - W)."""
    end = n - cfg.W
    if cfg.slots == "fixed64":
        b_ = list(range(0, end, 64)) + [end]
        if len(b_) > 2 and b_[-1] - b_[-2] < 16:
            del b_[-2]
        return np.asarray(b_, dtype=np.int32)
    r = _rng(cfg, b, TAG_SLOTS)
    lo, hi = (16, 112) if cfg.slots == "uniform" else (48, 80)
    out = [0]
    pos = 0
    while pos < end:
        ln = int(r.integers(lo, hi + 1))
        pos = min(end, pos + ln)
        out.append(pos)
    if len(out) > 2 and out[-1] - out[-2] < 16:
        del out[-2]
    return np.asarray(out, dtype=np.int32)


@dataclass
class SeqInputs:
    n: int
    K: np.ndarray            # [L, H, n, d] float32, values exact in cfg.dtype (post-RoPE)
    V: np.ndarray            # [L, H, n, d]
    Qp: np.ndarray           # [L, H*G, P, d] post-RoPE probe queries
    slot_bounds: np.ndarray  # int32 [S+1] over [0, n - W)
    planted: np.ndarray      # generator's segment boundaries (== slot_bounds unless curvature)
    needles: List[Tuple[int, int, int, str, int]] = field(default_factory=list)
    # (l, h, position, 'A' | 'B', partner position or -1)


@dataclass
class Workload:
    cfg: Config
    seqs: List[SeqInputs]
    head_sens: np.ndarray    # [L, H] float32

    @property
    def ctx_len(self) -> np.ndarray:
        return np.asarray([s.n for s in self.seqs], dtype=np.int64)


def _needle_counts(cfg: Config, b: int, n: int) -> np.ndarray:
    LH = cfg.L * cfg.H
    if cfg.needles == "none":
        return np.zeros(LH, dtype=np.int64)
    if cfg.needles == "tiny":
        return np.full(LH, 4, dtype=np.int64)
    total = int(round(cfg.needle_frac * n))
    if cfg.needles == "pairs":
        return np.full(LH, total, dtype=np.int64)
    # zipf: total needles over all pairs, weight rank^-1.1 over a random permutation
    r = _rng(cfg, b, TAG_ZIPF)
    perm = r.permutation(LH)
    w = 1.0 / np.arange(1, LH + 1, dtype=np.float64) ** 1.1
    share = total * w / w.sum()
    cnt = np.floor(share).astype(np.int64)
    rem = total - int(cnt.sum())
    order = np.argsort(-(share - cnt), kind="stable")
    cnt[order[:rem]] += 1
    out = np.zeros(LH, dtype=np.int64)
    out[perm] = cnt
    return out


def gen_head(cfg: Config, b: int, l: int, h: int, n: int, seg_bounds: np.ndarray,
             n_needles: int):
    """K [n,d], V [n,d], Qp [G,P,d] for one (sequence, layer, KV head) and its needles."""
    d = cfg.d
    full = np.concatenate([seg_bounds.astype(np.int64), [n]]) if seg_bounds[-1] != n else \
        seg_bounds.astype(np.int64)
    V = _walk(_rng(cfg, b, l, h, TAG_V), n, d, full)
    Kpre = _walk(_rng(cfg, b, l, h, TAG_K), n, d, full)
    K = _post_rope(Kpre, np.arange(n), cfg.rope_base)
    Q = _rng(cfg, b, l, h, TAG_Q).standard_normal((cfg.G, cfg.P, d), dtype=np.float32)
    Q = _to_dtype(cfg, Q)
    V = _to_dtype(cfg, V)
    needles = []
    if n_needles > 0:
        r = _rng(cfg, b, l, h, TAG_NEEDLE)
        end = n - cfg.W
        pos = r.choice(end, size=min(n_needles, end), replace=False)
        n_a = n_needles if cfg.needles == "tiny" else (n_needles + 1) // 2
        a_pos = pos[:n_a]
        b_pos = pos[n_a:]
        for i in a_pos:
            g = int(r.integers(cfg.G)); p = int(r.integers(cfg.P))
            q = Q[g, p].astype(np.float64)
            qh = q / np.linalg.norm(q)
            u = _unit_orth(r, qh)
            nk = np.linalg.norm(K[i].astype(np.float64))
            K[i] = (nk * (0.9 * qh + np.sqrt(0.19) * u)).astype(np.float32)
            needles.append((l, h, int(i), "A", -1))
        for j, i in enumerate(b_pos):
            a = int(a_pos[j % len(a_pos)])
            va = V[a].astype(np.float64)
            vh = va / np.linalg.norm(va)
            u = _unit_orth(r, vh)
            nk = np.linalg.norm(K[i].astype(np.float64))
            K[i] = (nk * (0.9 * vh + np.sqrt(0.19) * u)).astype(np.float32)
            needles.append((l, h, int(i), "B", a))
    K = _to_dtype(cfg, K)
    return K, V, Q, needles


def make_workload(cfg: Config, heads: Optional[Sequence[Tuple[int, int]]] = None) -> Workload:
    """Generate every sequence of ``cfg``.  ``heads`` restricts generation to the
    listed (layer, KV head) pairs; the others stay zero."""
    seqs = []
    ns = context_lengths(cfg)
    want = None if heads is None else set(heads)
    for b in range(cfg.B):
        n = int(ns[b])
        planted = planted_bounds(cfg, b, n)
        counts = _needle_counts(cfg, b, n)
        K = np.zeros((cfg.L, cfg.H, n, cfg.d), dtype=np.float32)
        V = np.zeros_like(K)
        Qp = np.zeros((cfg.L, cfg.H * cfg.G, cfg.P, cfg.d), dtype=np.float32)
        needles = []
        for l in range(cfg.L):
            for h in range(cfg.H):
                if want is not None and (l, h) not in want:
                    continue
                k, v, q, nd = gen_head(cfg, b, l, h, n, planted, int(counts[l * cfg.H + h]))
                K[l, h] = k
                V[l, h] = v
                Qp[l, h * cfg.G:(h + 1) * cfg.G] = q
                needles += nd
        seqs.append(SeqInputs(n=n, K=K, V=V, Qp=Qp, slot_bounds=planted.copy(),
                              planted=planted, needles=needles))
    return Workload(cfg=cfg, seqs=seqs, head_sens=np.ones((cfg.L, cfg.H), dtype=np.float32))


def _gen_job(job):
    cfg, b, l, h, n, planted, count = job
    return b, l, h, gen_head(cfg, b, l, h, n, planted, count)


def make_workload_parallel(cfg: Config, processes: int) -> Workload:
    """``make_workload(cfg)`` with the (b, l, h) heads generated by a spawn
    process pool (each head has its own seeded stream, so the result is the
    same array for array)."""
    import multiprocessing as mp
    ns = context_lengths(cfg)
    planted = [planted_bounds(cfg, b, int(ns[b])) for b in range(cfg.B)]
    counts = [_needle_counts(cfg, b, int(ns[b])) for b in range(cfg.B)]
    seqs = []
    for b in range(cfg.B):
        n = int(ns[b])
        seqs.append(SeqInputs(n=n, K=np.zeros((cfg.L, cfg.H, n, cfg.d), dtype=np.float32),
                              V=np.zeros((cfg.L, cfg.H, n, cfg.d), dtype=np.float32),
                              Qp=np.zeros((cfg.L, cfg.H * cfg.G, cfg.P, cfg.d), dtype=np.float32),
                              slot_bounds=planted[b].copy(), planted=planted[b], needles=[]))
    jobs = [(cfg, b, l, h, int(ns[b]), planted[b], int(counts[b][l * cfg.H + h]))
            for b in range(cfg.B) for l in range(cfg.L) for h in range(cfg.H)]
    nd_all = {}
    with mp.get_context("spawn").Pool(max(1, processes)) as pool:
        for b, l, h, (k, v, q, nd) in pool.imap_unordered(_gen_job, jobs, chunksize=2):
            s = seqs[b]
            s.K[l, h] = k
            s.V[l, h] = v
            s.Qp[l, h * cfg.G:(h + 1) * cfg.G] = q
            nd_all[(b, l, h)] = nd
    for (b, l, h) in sorted(nd_all):                      # the serial order of make_workload
        seqs[b].needles += nd_all[(b, l, h)]
    return Workload(cfg=cfg, seqs=seqs, head_sens=np.ones((cfg.L, cfg.H), dtype=np.float32))


def decode_inputs(cfg: Config, step: int, B: Optional[int] = None):
    """Decode-step inputs: q [B, L, H*G, d], k_new / v_new [B, L, H, d], N(0, 1)."""
    B = cfg.B if B is None else B
    r = _rng(cfg, TAG_DEC, step)
    q = r.standard_normal((B, cfg.L, cfg.H * cfg.G, cfg.d), dtype=np.float32)
    k = r.standard_normal((B, cfg.L, cfg.H, cfg.d), dtype=np.float32)
    v = r.standard_normal((B, cfg.L, cfg.H, cfg.d), dtype=np.float32)
    return _to_dtype(cfg, q), _to_dtype(cfg, k), _to_dtype(cfg, v)


def hidden_states(cfg: Config, b: int, n: int, planted: np.ndarray,
                  dim: Optional[int] = None, noise: float = 0.002) -> np.ndarray:
    """Piecewise-smooth hidden-state trajectory [n, dim] with turns at ``planted``.

    The state moves on the sphere of radius sqrt(dim) (components of order 1,
    so bf16 resolves the motion): inside a segment it travels along a great
    circle at 0.02-0.06 rad per token; each planted boundary starts a new
    great circle through the current state in a random direction, so the
    direction of motion turns there while the state stays continuous.
    """
    dim = cfg.hidden_dim if dim is None else dim
    r = _rng(cfg, b, TAG_HID)
    rho = np.sqrt(dim)
    h = np.empty((n, dim), dtype=np.float64)
    cur = r.standard_normal(dim)
    cur /= np.linalg.norm(cur)
    bounds = list(planted.astype(np.int64))
    if bounds[-1] != n:
        bounds.append(n)
    for s in range(len(bounds) - 1):
        x0, x1 = bounds[s], bounds[s + 1]
        e2 = r.standard_normal(dim)
        e2 -= (e2 @ cur) * cur
        e2 /= np.linalg.norm(e2)
        om = r.uniform(0.02, 0.06)
        ang = om * np.arange(x1 - x0 + 1, dtype=np.float64)
        path = np.cos(ang)[:, None] * cur[None, :] + np.sin(ang)[:, None] * e2[None, :]
        h[x0:x1] = rho * path[:-1]
        cur = path[-1] / np.linalg.norm(path[-1])
    h += r.standard_normal((n, dim)) * noise
    return _to_dtype(cfg, h.astype(np.float32))
