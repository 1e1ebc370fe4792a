"""The near-tie checker of the end-to-end selection parity (CPU only).

It must accept a device selection that differs from the oracle chain only
through keys within 1e-6 relative of each other, and reject one that differs
through any larger key error.  The instances are random selection problems
with the tree shape and costs of reading R3 (GraceKV "02 Progressively
refinable representation"), selected by the oracle's own floor and auction."""
import numpy as np
import pytest

import oracle as O
from synth import workloads as W
from tests.tie_check import band_needed, check_sequence, tie_resolved_rank


def _instance(seed, L=2, H=3, n=1400):
    rng = np.random.default_rng(seed)
    cfg = W.small_config(L=L, H=H, n=n, W=128, budget_ratio=0.25, floor_cap_frac=0.05)
    end = n - cfg.W
    cuts = [0]
    while cuts[-1] < end:
        cuts.append(min(end, cuts[-1] + int(rng.integers(16, 113))))
    if cuts[-1] - cuts[-2] < 16:
        cuts.pop(-2)
    bounds = np.asarray(cuts)
    S = len(bounds) - 1
    cost = np.zeros((L, H, S, 16), np.int64)
    for s in range(S):
        c = np.r_[1, [y - x for x, y in O.tree_nodes(int(bounds[s]), int(bounds[s + 1]))]]
        cost[:, :, s] = np.r_[1, np.ones(7), c[8:] - 1][None, None]
    util = np.exp(rng.normal(0, 2, size=(L, H, S, 16)))
    r = np.exp(rng.normal(-8, 1.5, size=(L, H, n)))
    return cfg, bounds, cost, util, r, np.ones((L, H))


def _select(cfg, bounds, n, util, cost, r, sens):
    return O.select_sequence(util, cost, r, sens, bounds, n, cfg.W, cfg.budget_ratio,
                             cfg.budget_entries_per_lh, cfg.floor_cap_frac,
                             cfg.floor_cap_tokens).taken


def test_rank_follows_the_oracle_order_outside_near_ties():
    k64 = np.array([5.0, 3.0, 3.0 * (1 + 5e-7), 1.0, 3.0 * (1 - 5e-7), 0.0, 0.0])
    kd = np.array([5.0, 3.1, 2.9, 1.0, 3.0, 0.1, 0.0])      # reorders the 3.0 run and the zeros
    rank, moved = tie_resolved_rank(k64, kd)
    order = list(np.argsort(-rank))
    assert order == [0, 1, 4, 2, 3, 5, 6]
    assert moved == 1                                       # zeros already in index order
    kd2 = kd.copy(); kd2[6] = 0.2
    rank2, moved2 = tie_resolved_rank(k64, kd2)
    assert list(np.argsort(-rank2))[-2:] == [6, 5] and moved2 == 2
    far = np.array([2.0, 1.0]); rank3, m3 = tie_resolved_rank(far, np.array([1.0, 2.0]))
    assert list(np.argsort(-rank3)) == [0, 1] and m3 == 0  # not a near-tie: oracle order


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fp32_rounded_keys_are_explained(seed):
    cfg, bounds, cost, util, r, sens = _instance(seed)
    n = cfg.n
    u32, r32 = util.astype(np.float32), r.astype(np.float32)
    taken = _select(cfg, bounds, n, u32.astype(np.float64), cost, r32.astype(np.float64), sens)
    rep = check_sequence(util, u32, cost, r, r32, sens, taken, bounds, n, cfg)
    assert rep.max_rel_err <= 2 ** -24


def test_planted_near_ties_resolved_the_other_way_are_explained_and_counted():
    cfg, bounds, cost, util, r, sens = _instance(3)
    n = cfg.n
    sel = _select(cfg, bounds, n, util, cost, r, sens)
    # exact ties between each op and a random other op, device order flipped
    rng = np.random.default_rng(5)
    flat = util.reshape(-1).copy()
    a = rng.choice(flat.size, 200, replace=False)
    flat[a[100:]] = flat[a[:100]]
    util_t = flat.reshape(util.shape)
    dev = util_t.copy().reshape(-1)
    hi = np.maximum(a[:100], a[100:])
    dev[hi] *= 1 + 3e-7                                     # the later op now ranks first
    dev = dev.reshape(util.shape)
    taken = _select(cfg, bounds, n, dev, cost, r, sens)
    rep = check_sequence(util_t, dev, cost, r, r, sens, taken, bounds, n, cfg)
    assert rep.runs_moved_util >= 1
    assert rep.diff_ops == int((_select(cfg, bounds, n, util_t, cost, r, sens) != taken).sum())
    del sel


def test_a_key_error_beyond_the_band_that_changes_the_selection_is_rejected():
    cfg, bounds, cost, util, r, sens = _instance(4)
    n = cfg.n
    sel = _select(cfg, bounds, n, util, cost, r, sens)
    # walk the ops from the lowest key up and scale one key by 1.05 until the
    # selection changes: that op sits at the cut and its key error is 5%
    for flat in np.argsort(util.reshape(-1)):
        dev = util.copy().reshape(-1)
        dev[flat] *= 1.05
        dev = dev.reshape(util.shape)
        taken = _select(cfg, bounds, n, dev, cost, r, sens)
        if (taken != sel).any():
            break
    else:
        pytest.fail("no single key change moved the selection")
    with pytest.raises(AssertionError, match="taken bits differ"):
        check_sequence(util, dev, cost, r, r, sens, taken, bounds, n, cfg)
    assert band_needed(util, dev, cost, r, r, sens, taken, bounds, n, cfg) == 1e-1


def test_a_relevance_error_that_changes_the_floor_is_rejected():
    cfg, bounds, cost, util, r, sens = _instance(6)
    n = cfg.n
    cfg = cfg.replace(floor_cap_frac=0.02)
    sel = _select(cfg, bounds, n, util, cost, r, sens)
    end = int(bounds[-1])
    order = np.argsort(-r[:, :, :end].reshape(-1))
    for k in order[:400]:
        rd = r.copy()
        l, h, i = np.unravel_index(k, (cfg.L, cfg.H, end))
        rd[l, h, i] *= 0.5
        taken = _select(cfg, bounds, n, util, cost, rd, sens)
        if (taken != sel).any():
            break
    else:
        pytest.fail("no single relevance change moved the floor")
    with pytest.raises(AssertionError):
        check_sequence(util, util, cost, r, rd, sens, taken, bounds, n, cfg)


def test_utility_slack_counts_and_rejects():
    from tests.tie_check import utility_slack
    rng = np.random.default_rng(9)
    bounds = np.array([0, 40, 104], np.int64)
    r = rng.random((1, 1, 104))
    cost = np.ones((1, 1, 2, 16), np.int64)
    sens = np.ones((1, 1))
    u = rng.random((1, 1, 2, 16)) * 1e-3
    u[0, 0, 1, 3] = 0.0                       # a utility that cancelled to zero
    got = u.astype(np.float32)
    got[0, 0, 1, 3] = 1e-7                    # within the scale term only
    n, n_rel, n_scale, worst = utility_slack(u, got, cost, r, sens, bounds)
    assert n == 32 and n_scale >= 1 and n_rel + n_scale == 32 and worst <= 1.0
    got[0, 0, 0, 5] = u[0, 0, 0, 5] + 1.0     # far outside any bound
    with pytest.raises(AssertionError):
        utility_slack(u, got, cost, r, sens, bounds)
