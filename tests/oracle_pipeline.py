"""Runs the CPU oracle over a whole synthetic workload (test infrastructure)."""
from dataclasses import dataclass
from typing import List

import numpy as np

import oracle as O


@dataclass
class OracleRun:
    cfg: object
    S_max: int
    lse: np.ndarray           # [B, L, H, R]
    feats: List[np.ndarray]   # per b: [L, H, n, 5]
    r: List[np.ndarray]       # per b: [L, H, n]
    util: np.ndarray          # [B, L, H, S_max, 16] float64
    cost: np.ndarray          # [B, L, H, S_max, 16]
    heads: dict               # (b, l, h) -> HeadResult


def score_all(wl, S_h=None, keep_protos=False) -> OracleRun:
    cfg = wl.cfg
    S_max = max(len(s.slot_bounds) - 1 for s in wl.seqs)
    B, L, H = cfg.B, cfg.L, cfg.H
    lse = np.zeros((B, L, H, cfg.R))
    util = np.zeros((B, L, H, S_max, 16))
    cost = np.zeros((B, L, H, S_max, 16), dtype=np.int64)
    feats, rr, heads = [], [], {}
    for b, s in enumerate(wl.seqs):
        f = np.zeros((L, H, s.n, 5)); r = np.zeros((L, H, s.n))
        S = len(s.slot_bounds) - 1
        for l in range(L):
            for h in range(H):
                res = O.score_and_value_head(
                    s.K[l, h], s.V[l, h], s.Qp[l, h * cfg.G:(h + 1) * cfg.G], s.n, cfg.P,
                    s.slot_bounds, float(wl.head_sens[l, h]), base=cfg.rope_base,
                    hop_weight=cfg.hop_weight, n_hops=cfg.n_hops, w_part=cfg.w_part,
                    w_value=cfg.w_value, value_floor=cfg.value_floor, S_h=S_h,
                    keep_protos=keep_protos)
                lse[b, l, h] = res.lse
                f[l, h] = res.feats
                r[l, h] = res.r
                util[b, l, h, :S] = res.util
                cost[b, l, h, :S] = res.cost
                heads[(b, l, h)] = res
        feats.append(f)
        rr.append(r)
    return OracleRun(cfg=cfg, S_max=S_max, lse=lse, feats=feats, r=rr, util=util, cost=cost,
                     heads=heads)


def select_all(wl, util, cost, r_list, cfg=None):
    """Per-sequence selection; util/cost [B, L, H, S_max, 16], r_list per b [L, H, n]."""
    cfg = cfg or wl.cfg
    sels = []
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        sels.append(O.select_sequence(util[b, :, :, :S], cost[b, :, :, :S], r_list[b],
                                      wl.head_sens, s.slot_bounds, s.n, cfg.W, cfg.budget_ratio,
                                      cfg.budget_entries_per_lh, cfg.floor_cap_frac,
                                      cfg.floor_cap_tokens))
    return sels


def pack_all(wl, taken_list, r_list, cfg=None):
    """Oracle packing of every (b, l, h); returns per-(b,l,h) arrays and len/cap/off."""
    cfg = cfg or wl.cfg
    B, L, H = cfg.B, cfg.L, cfg.H
    ent = {}
    lens = np.zeros((B, L, H), dtype=np.int64)
    for b, s in enumerate(wl.seqs):
        for l in range(L):
            for h in range(H):
                K, V, lm, ps = O.pack_head(s.K[l, h], s.V[l, h], r_list[b][l, h], s.slot_bounds,
                                           taken_list[b][l, h], s.n, cfg.W, cfg.rope_base,
                                           cfg.value_floor)
                ent[(b, l, h)] = (K, V, lm, ps)
                lens[b, l, h] = len(K)
    caps, offs = O.offsets(lens, cfg.decode_reserve)
    return ent, lens, caps, offs


def _score_job(job):
    """One (layer, KV head) of the oracle's scoring, in a worker process."""
    l, h, K, V, Q, n, P, bounds, sens, kw = job
    res = O.score_and_value_head(K, V, Q, n, P, bounds, sens, **kw)
    return l, h, res.util, res.cost, res.r


_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def score_sequence_parallel(wl, b, processes):
    """The oracle's float64 scoring of every (layer, KV head) of sequence b, spread
    over a spawn process pool with one BLAS thread per worker.  Returns
    (util [L, H, S, 16] float64, cost [L, H, S, 16], r [L, H, n])."""
    import multiprocessing as mp
    import os
    cfg = wl.cfg
    s = wl.seqs[b]
    S = len(s.slot_bounds) - 1
    kw = dict(base=cfg.rope_base, hop_weight=cfg.hop_weight, n_hops=cfg.n_hops,
              w_part=cfg.w_part, w_value=cfg.w_value, value_floor=cfg.value_floor)
    jobs = [(l, h, s.K[l, h], s.V[l, h], s.Qp[l, h * cfg.G:(h + 1) * cfg.G], s.n, cfg.P,
             s.slot_bounds, float(wl.head_sens[l, h]), kw)
            for l in range(cfg.L) for h in range(cfg.H)]
    util = np.zeros((cfg.L, cfg.H, S, 16))
    cost = np.zeros((cfg.L, cfg.H, S, 16), dtype=np.int64)
    r = np.zeros((cfg.L, cfg.H, s.n))
    saved = {k: os.environ.get(k) for k in _BLAS_VARS}
    os.environ.update({k: "1" for k in _BLAS_VARS})
    try:
        pool = mp.get_context("spawn").Pool(max(1, processes))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    with pool:
        for l, h, u, c, rr in pool.imap_unordered(_score_job, jobs):
            util[l, h], cost[l, h], r[l, h] = u, c, rr
    return util, cost, r
