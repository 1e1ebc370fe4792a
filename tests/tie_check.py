"""End-to-end selection parity with near-ties (test infrastructure).

The device chain's selection is compared with the oracle chain's own (float64
keys).  Selected sets must be identical except where two keys lie within a
relative band (1e-6) of each other: such near-ties may be resolved either way,
and every selection difference they cause is counted and reported.

Method.  Sort the oracle's keys (descending, index ascending, the order of
GraceKV "04 Top-down budget flow" with reading R13).  Group adjacent keys into
runs whose neighbours lie within the band of each other.  Inside a run the
device's keys decide the order (descending, index ascending); between runs the
oracle's order stands.  The oracle's floor and auction are then re-run on
these tie-resolved orders.  The device's taken set must equal that result bit
for bit: a difference from the oracle chain is then caused only by how
near-ties fell.  The same is done for the singleton floor's candidate keys
r * sens.

Only the oracle's own selection runs here; nothing of the device path.
"""
from dataclasses import dataclass

import numpy as np

import oracle as O

TIE_REL = 1e-6


def tie_resolved_rank(key64: np.ndarray, key_dev: np.ndarray, rel: float = TIE_REL):
    """Rank keys (float64, larger = earlier) following key64's total order
    (descending, flat index ascending) except inside runs of near-equal key64
    values (adjacent within `rel` relative), which follow key_dev's order
    (descending, flat index ascending).  Returns (rank, runs moved) where the
    second counts the runs whose order the device keys changed."""
    k64 = np.asarray(key64, np.float64).reshape(-1)
    kd = np.asarray(key_dev, np.float64).reshape(-1)
    n = k64.size
    idx = np.arange(n)
    order = np.lexsort((idx, -k64))
    ks = k64[order]
    if n > 1:
        gap = np.abs(np.diff(ks)) > rel * np.maximum(np.abs(ks[1:]), np.abs(ks[:-1]))
        run = np.concatenate([[0], np.cumsum(gap)])
    else:
        run = np.zeros(n, np.int64)
    order2 = order[np.lexsort((order, -kd[order], run))]
    moved = np.unique(run[order2 != order]).size
    rank = np.empty(n)
    rank[order2] = np.arange(n, 0, -1, dtype=np.float64)
    return rank.reshape(np.shape(key64)), int(moved)


@dataclass
class TieReport:
    diff_ops: int          # ops whose taken bit differs between the device and the oracle chain
    runs_moved_util: int   # near-tie runs of op keys that the device ordered differently
    runs_moved_floor: int  # the same for floor candidate keys
    max_abs_err: float     # over every op key: |device - oracle|
    max_rel_err: float     # |device - oracle| / |oracle| over ops with a non-zero oracle key


def check_sequence(util64, util_dev, cost, r64, r_dev, sens, taken_dev, bounds, n, cfg,
                   rel: float = TIE_REL) -> TieReport:
    """One sequence.  util64 / util_dev [L, H, S, 16] (oracle float64 keys, device
    fp32 keys), cost [L, H, S, 16] (identical on both sides), r64 / r_dev [L, H, n]
    relevance, sens [L, H], taken_dev [L, H, S, 16] bool.  Raises AssertionError
    if the device's taken set is not the oracle's selection under some
    resolution of the near-ties; returns the report otherwise."""
    L, H, S, _ = util64.shape
    end = int(bounds[-1])
    sel64 = O.select_sequence(util64, cost, r64, sens, bounds, n, cfg.W, cfg.budget_ratio,
                              cfg.budget_entries_per_lh, cfg.floor_cap_frac, cfg.floor_cap_tokens)
    u_rank, mu = tie_resolved_rank(util64, util_dev, rel)
    # floor keys r * sens: float64 on the oracle side, one rounded fp32 multiply on the device
    f64 = np.asarray(r64, np.float64)[:, :, :end] * np.asarray(sens, np.float64)[:, :, None]
    fdev = (np.asarray(r_dev, np.float32)[:, :, :end] *
            np.asarray(sens, np.float32)[:, :, None]).astype(np.float32)
    pos64 = np.asarray(r64)[:, :, :end] > 0
    posd = np.asarray(r_dev)[:, :, :end] > 0
    assert np.array_equal(pos64, posd), "floor candidates (r > 0) differ"
    f_rank, mf = tie_resolved_rank(f64, fdev, rel)
    r_mix = np.zeros((L, H, n))
    r_mix[:, :, :end] = np.where(pos64, f_rank, 0.0)
    selx = O.select_sequence(u_rank, cost, r_mix, np.ones((L, H)), bounds, n, cfg.W,
                             cfg.budget_ratio, cfg.budget_entries_per_lh, cfg.floor_cap_frac,
                             cfg.floor_cap_tokens)
    bad = np.argwhere(selx.taken != taken_dev)
    if bad.size:
        l, h, s, o = (int(x) for x in bad[0])
        raise AssertionError(
            f"{len(bad)} taken bits differ from the oracle under every {rel:g} tie resolution; "
            f"first at (l={l}, h={h}, slot={s}, op={o}): device {bool(taken_dev[l, h, s, o])}, "
            f"oracle key {util64[l, h, s, o]!r}, device key {float(util_dev[l, h, s, o])!r}")
    d64 = np.asarray(util_dev, np.float64)
    err = np.abs(d64 - util64)
    nz = util64 != 0
    return TieReport(diff_ops=int((sel64.taken != taken_dev).sum()), runs_moved_util=mu,
                     runs_moved_floor=mf, max_abs_err=float(err.max()) if err.size else 0.0,
                     max_rel_err=float((err[nz] / np.abs(util64[nz])).max()) if nz.any() else 0.0)


def band_needed(util64, util_dev, cost, r64, r_dev, sens, taken_dev, bounds, n, cfg):
    """Smallest power-of-ten band (1e-7 .. 1e-1) under which the device's taken set
    is explained by near-ties, or None (a diagnostic for failure messages)."""
    for e in range(7, 0, -1):
        try:
            check_sequence(util64, util_dev, cost, r64, r_dev, sens, taken_dev, bounds, n, cfg,
                           rel=10.0 ** -e)
            return 10.0 ** -e
        except AssertionError:
            continue
    return None


def utility_slack(u64, u_dev, cost, r64, sens, bounds):
    """Every utility of one sequence against the utility tolerance of the
    tests: |g - o| <= 1e-5 * max(|o|, 3 * scale), scale = R(N) * sens / cost
    per op (R(N) the node's oracle relevance mass; the Add op uses the root's).
    A utility is scale times a clamped difference of normalised distortions,
    so fp32 reaches it to an accuracy relative to the scale, not to |u|.
    Returns (ops, ops within 1e-5 * |o|, ops that pass only through the scale
    term, worst err / bound); asserts that every op passes."""
    from oracle import kvc_oracle as O
    L, H, S, _ = u64.shape
    scale = np.empty_like(u64)
    for l in range(L):
        for h in range(H):
            cs = np.r_[0.0, np.cumsum(r64[l, h])]
            for k in range(S):
                nodes = O.tree_nodes(int(bounds[k]), int(bounds[k + 1]))
                Rv = np.array([cs[y] - cs[x] for x, y in nodes])
                scale[l, h, k] = np.r_[Rv[0], Rv] * float(sens[l, h]) / cost[l, h, k]
    err = np.abs(u_dev.astype(np.float64) - u64)
    bound = 1e-5 * np.maximum(np.abs(u64), 3 * scale)
    worst = float((err / np.maximum(bound, 1e-300)).max())
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"utility outside tolerance at (l, h, slot, op) {tuple(i)}: "
                             f"device {u_dev[tuple(i)]!r}, oracle {u64[tuple(i)]!r}, "
                             f"bound {bound[tuple(i)]!r}")
    rel_ok = err <= 1e-5 * np.abs(u64)
    return int(u64.size), int(rel_ok.sum()), int((~rel_ok).sum()), worst
