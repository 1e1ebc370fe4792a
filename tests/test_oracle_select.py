"""Pins for the oracle's budget, singleton floor, greedy auction and packing.

The greedy is checked against two independent implementations written here:
a repeated linear scan for the best exposed op (brute force), and the
"effective key" formulation (sort ops by the running minimum of their key along
the tree path, then one scan) that the GPU selection is built on.  The floor is
checked against its prefix formulation (a candidate's path cost depends only on
whether an earlier candidate shares its tree / subtree / leaf).
"""
import math

import numpy as np
import pytest

import oracle as O
from synth import workloads as W


# ------------------------------------------------------------------ budget arithmetic
def test_budget_numbers_of_the_configs():
    assert O.budget(512, 1, 2, 32, 0.25, 0, 1.0) == (256, 192, 192)
    assert O.budget(16384, 32, 8, 128, 0.25, 0, 0.01) == (1048576, 1015808, 10158)
    assert O.budget(131072, 32, 8, 256, 0.0, 1024, 0.6)[:2] == (262144, 196608)
    assert O.budget(32768, 32, 8, 128, 0.10, 0, 0.6)[0] == 3276 * 256
    with pytest.raises(ValueError):
        O.budget(100, 1, 1, 64, 0.25, 0, 0.6)


# ------------------------------------------------------------------ random instances
def _instance(seed, L=2, H=2, bounds=(0, 16, 40, 64, 100), levels=(0.0, 0.1, 0.2, 0.5)):
    rng = np.random.default_rng(seed)
    bounds = np.asarray(bounds)
    S = len(bounds) - 1
    util = rng.choice(np.asarray(levels, np.float32), size=(L, H, S, 16))
    cost = np.zeros((L, H, S, 16), dtype=np.int64)
    for s in range(S):
        nodes = O.tree_nodes(int(bounds[s]), int(bounds[s + 1]))
        cost[:, :, s, :8] = 1
        for j in range(7, 15):
            cost[:, :, s, 1 + j] = nodes[j][1] - nodes[j][0] - 1
    n = int(bounds[-1]) + 8
    r = rng.choice(np.asarray([0.0, 0.01, 0.02, 0.05], np.float32), size=(L, H, n))
    return util, cost, r, bounds, n


def _tree_closed(taken):
    L, H, S, _ = taken.shape
    for l in range(L):
        for h in range(H):
            for s in range(S):
                for o in range(1, 16):
                    if taken[l, h, s, o]:
                        assert taken[l, h, s, O.op_parent(o)]


def _gid(H, S, l, h, s, o):
    return ((l * H + h) * S + s) * 16 + o


def scan_greedy(util, cost, taken, remaining):
    """Brute force: keep a list of exposed ops, scan it for the best each step."""
    L, H, S, _ = util.shape
    exposed = []
    for l in range(L):
        for h in range(H):
            for s in range(S):
                t = taken[l, h, s]
                if not t[0]:
                    exposed.append((l, h, s, 0))
                    continue
                for o in range(1, 16):
                    if not t[o] and t[O.op_parent(o)]:
                        exposed.append((l, h, s, o))
    while exposed:
        best = None
        for e in exposed:
            k = (float(util[e]), -_gid(H, S, *e))
            if best is None or k > best[0]:
                best = (k, e)
        e = best[1]
        exposed.remove(e)
        if cost[e] <= remaining:
            remaining -= int(cost[e])
            taken[e] = True
            l, h, s, o = e
            for c in range(1, 16):
                if O.op_parent(c) == o:
                    exposed.append((l, h, s, c))
    return remaining


def effective_key_greedy(util, cost, taken, remaining):
    """Sort untaken ops by (running-min key along the path desc, rank inside the
    block of equal running minimum), then take each op whose parent is taken and
    whose cost fits, in that order."""
    L, H, S, _ = util.shape
    entries = []
    for l in range(L):
        for h in range(H):
            for s in range(S):
                t = taken[l, h, s]
                key = {o: (float(util[l, h, s, o]), -_gid(H, S, l, h, s, o)) for o in range(16)}
                eff = {}
                for o in range(16):                      # parents come before children
                    if t[o]:
                        continue
                    p = O.op_parent(o)
                    eff[o] = key[o] if (p < 0 or t[p]) else min(key[o], eff[p])
                rank = {}
                for o, e in eff.items():
                    if e == key[o] and o not in rank:    # o is a block head
                        pool = [o]
                        k = 0
                        while pool:
                            b = max(pool, key=lambda x: key[x])
                            pool.remove(b)
                            rank[b] = k; k += 1
                            pool += [c for c in range(1, 16) if O.op_parent(c) == b
                                     and c in eff and eff[c] == e]
                for o, e in eff.items():
                    entries.append(((e[0], e[1], -rank[o]), (l, h, s, o)))
    entries.sort(key=lambda x: x[0], reverse=True)
    for _, e in entries:
        l, h, s, o = e
        p = O.op_parent(o)
        if (p < 0 or taken[l, h, s, p]) and cost[e] <= remaining:
            taken[e] = True
            remaining -= int(cost[e])
    return remaining


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("budget_frac", [0.05, 0.3, 0.7, 1.0])
def test_heap_greedy_equals_scan_and_effective_key(seed, budget_frac):
    util, cost, r, bounds, n = _instance(seed)
    total = int(cost.sum())
    rem = int(budget_frac * total)
    pre = np.zeros(util.shape, dtype=bool)
    if seed % 3 == 0:                                  # a pre-taken floor path
        pre[0, 1, 2, [0, 1, 2, 4, 8]] = True       # Add, Split(0), Split(1), Split(3), Split(7)
    t1, t2, t3 = pre.copy(), pre.copy(), pre.copy()
    spent = O.greedy_auction(util, cost, t1, rem)
    r2 = scan_greedy(util, cost, t2, rem)
    r3 = effective_key_greedy(util, cost, t3, rem)
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_array_equal(t1, t3)
    assert rem - spent == r2 == r3
    _tree_closed(t1)
    assert ((t1 & ~pre) * cost).sum() == spent <= rem


def floor_prefix(r, sens, bounds, cost, cap_entries, cap_tokens, cuts=None):
    """Floor in prefix form: within the stop prefix every earlier candidate was
    taken, so a candidate's cost is fixed by which groups it opens first."""
    L, H, n = r.shape
    end = int(bounds[-1])
    cands = []
    for l in range(L):
        for h in range(H):
            for i in range(end):
                if r[l, h, i] > 0:
                    key = np.float32(r[l, h, i]) * np.float32(sens[l, h])
                    cands.append((-float(key), (l * H + h) * n + i, l, h, i))
    cands.sort()
    seen = set()
    spent = 0
    tokens = 0
    taken = np.zeros(cost.shape, dtype=bool)
    for _, _, l, h, i in cands:
        if cap_tokens >= 0 and tokens >= cap_tokens:
            break
        s = int(np.searchsorted(bounds, i, side="right") - 1)
        leaf, path = _path(i, bounds, s, None if cuts is None else cuts[l, h, s])
        groups = [(l, h, s, j) for j in path]
        if (l, h, s, leaf) in seen:
            continue
        c = 0
        if (l, h, s, 0) not in seen:
            c += int(cost[l, h, s, 0])
        for j in path:
            if (l, h, s, j) not in seen:
                c += int(cost[l, h, s, 1 + j])
        if spent + c > cap_entries:
            break
        spent += c
        tokens += 1
        seen.update(groups)
        taken[l, h, s, [0] + [1 + j for j in path]] = True
    return taken, spent, tokens


def _path(i, bounds, s, cuts=None):
    nodes = O.tree_nodes(int(bounds[s]), int(bounds[s + 1]), cuts)
    j = 0
    path = [0]
    while j < 7:
        j = 2 * j + 1 if i < nodes[2 * j + 1][1] else 2 * j + 2
        path.append(j)
    return j, path


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("cap", [0, 5, 23, 60, 400])
@pytest.mark.parametrize("cap_tokens", [-1, 3])
def test_floor_equals_prefix_form(seed, cap, cap_tokens):
    util, cost, r, bounds, n = _instance(seed)
    sens = np.random.default_rng(seed).choice(np.float32([0.5, 1.0, 2.0]), size=(2, 2))
    t1 = np.zeros(cost.shape, dtype=bool)
    sp, tk = O.singleton_floor(r, sens, bounds, cost, cap, cap_tokens, t1)
    t2, sp2, tk2 = floor_prefix(r, sens, bounds, cost, cap, cap_tokens)
    np.testing.assert_array_equal(t1, t2)
    assert (sp, tk) == (sp2, tk2)
    assert sp <= cap and (cap_tokens < 0 or tk <= cap_tokens)
    assert (t1 * cost).sum() == sp
    _tree_closed(t1)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("cap", [5, 23, 400])
def test_floor_equals_prefix_form_on_curvature_trees(seed, cap):
    """The same cross-check on curvature-chosen trees (reading R18): every
    (l, h) has its own cuts, the leaf split costs follow the leaves' sizes."""
    util, cost, r, bounds, n = _instance(seed)
    rng = np.random.default_rng(100 + seed)
    L, H, S = cost.shape[:3]
    cuts = np.zeros((L, H, S, 7), dtype=np.int64)
    for l in range(L):
        for h in range(H):
            kap = rng.uniform(0, 0.2, n) + (rng.uniform(size=n) < 0.1) * 1.5
            cuts[l, h] = O.slot_cuts(kap, bounds)
            for s_ in range(S):
                nodes = O.tree_nodes(int(bounds[s_]), int(bounds[s_ + 1]), cuts[l, h, s_])
                for j in range(7, 15):
                    cost[l, h, s_, 1 + j] = nodes[j][1] - nodes[j][0] - 1
    mid = np.asarray([[(a + b) // 2 for a, b in O.tree_nodes(int(bounds[k]), int(bounds[k + 1]))[:7]]
                      for k in range(S)])
    assert (cuts != mid[None, None]).any()                 # not all midpoint trees
    sens = np.ones((L, H), np.float32)
    t1 = np.zeros(cost.shape, dtype=bool)
    sp, tk = O.singleton_floor(r, sens, bounds, cost, cap, -1, t1, cuts)
    t2, sp2, tk2 = floor_prefix(r, sens, bounds, cost, cap, -1, cuts)
    np.testing.assert_array_equal(t1, t2)
    assert (sp, tk) == (sp2, tk2)
    assert (t1 * cost).sum() == sp <= cap
    _tree_closed(t1)


def test_floor_takes_top_token_first():
    util, cost, r, bounds, n = _instance(3)
    r[:] = 0
    r[1, 0, 45] = 1.0
    r[0, 1, 3] = 0.5
    t = np.zeros(cost.shape, dtype=bool)
    sp, tk = O.singleton_floor(r, np.ones((2, 2), np.float32), bounds, cost, 1000, -1, t)
    assert tk == 2
    s = int(np.searchsorted(bounds, 45, side="right") - 1)
    leaf, path = _path(45, bounds, s)
    assert t[1, 0, s, 1 + leaf] and t[1, 0, s, 0]
    # cost of a fresh path = Add + 3 ancestor splits + (leaf size - 1)
    nodes = O.tree_nodes(int(bounds[s]), int(bounds[s + 1]))
    assert (t[1, 0] * cost[1, 0]).sum() == 4 + (nodes[leaf][1] - nodes[leaf][0] - 1)


# ------------------------------------------------------------------ whole-sequence select + pack
def _score_seq(cfg, seq, sens):
    L, H = cfg.L, cfg.H
    S = len(seq.slot_bounds) - 1
    util = np.zeros((L, H, S, 16)); cost = np.zeros((L, H, S, 16), dtype=np.int64)
    r = np.zeros((L, H, seq.n))
    for l in range(L):
        for h in range(H):
            res = O.score_and_value_head(seq.K[l, h], seq.V[l, h], seq.Qp[l, h * cfg.G:(h + 1) * cfg.G],
                                         seq.n, cfg.P, seq.slot_bounds, float(sens[l, h]))
            util[l, h], cost[l, h], r[l, h] = res.util, res.cost, res.r
    return util, cost, r


@pytest.fixture(scope="module")
def tiny_scored():
    cfg = W.get_config("tiny")
    wl = W.make_workload(cfg)
    seq = wl.seqs[0]
    return cfg, wl, seq, _score_seq(cfg, seq, wl.head_sens)


def _select(cfg, seq, sens, scored, **kw):
    util, cost, r = scored
    c = cfg.replace(**kw) if kw else cfg
    return O.select_sequence(util, cost, r, sens, seq.slot_bounds, seq.n, c.W, c.budget_ratio,
                             c.budget_entries_per_lh, c.floor_cap_frac, c.floor_cap_tokens)


def test_budget_never_exceeded_and_window_counted(tiny_scored):
    cfg, wl, seq, scored = tiny_scored
    for beta in (0.07, 0.1, 0.25, 0.5, 0.9):
        sel = _select(cfg, seq, wl.head_sens, scored, budget_ratio=beta)
        assert sel.lens.sum() <= sel.B_tot
        assert sel.floor_spent <= int(math.floor(cfg.floor_cap_frac * sel.B_alloc))
        assert sel.floor_tokens <= cfg.floor_cap_tokens
        assert (sel.lens >= cfg.W).all()
        assert sel.lens.sum() - cfg.W * cfg.L * cfg.H == sel.floor_spent + sel.auction_spent
        _tree_closed(sel.taken)


def test_full_budget_takes_everything_and_pack_is_the_input(tiny_scored):
    """At 100% budget every tree expands to token leaves and the packed cache is the
    original cache, bit for bit, with log m = 0 (GraceKV '05 Physical cache packing')."""
    cfg, wl, seq, scored = tiny_scored
    sel = _select(cfg, seq, wl.head_sens, scored, budget_ratio=1.0)
    assert sel.taken.all()
    for l in range(cfg.L):
        for h in range(cfg.H):
            K, V, lm, ps = O.pack_head(seq.K[l, h], seq.V[l, h], scored[2][l, h], seq.slot_bounds,
                                       sel.taken[l, h], seq.n, cfg.W, cfg.rope_base, cfg.value_floor)
            np.testing.assert_array_equal(K, seq.K[l, h].astype(np.float64))
            np.testing.assert_array_equal(V, seq.V[l, h].astype(np.float64))
            assert (lm == 0).all()
            np.testing.assert_array_equal(ps, np.arange(seq.n))


def test_window_only_budget_packs_only_the_window(tiny_scored):
    cfg, wl, seq, scored = tiny_scored
    sel = _select(cfg, seq, wl.head_sens, scored, budget_ratio=cfg.W / seq.n)
    assert not sel.taken.any()
    K, V, lm, ps = O.pack_head(seq.K[0, 0], seq.V[0, 0], scored[2][0, 0], seq.slot_bounds,
                               sel.taken[0, 0], seq.n, cfg.W, cfg.rope_base, cfg.value_floor)
    np.testing.assert_array_equal(ps, np.arange(seq.n - cfg.W, seq.n))


def test_pack_order_lengths_and_offsets(tiny_scored):
    cfg, wl, seq, scored = tiny_scored
    sel = _select(cfg, seq, wl.head_sens, scored)
    for l in range(cfg.L):
        for h in range(cfg.H):
            K, V, lm, ps = O.pack_head(seq.K[l, h], seq.V[l, h], scored[2][l, h], seq.slot_bounds,
                                       sel.taken[l, h], seq.n, cfg.W, cfg.rope_base, cfg.value_floor)
            assert len(K) == sel.lens[l, h]
            assert (np.diff(ps) > 0).all()                # entries sorted by position
            exact = lm == 0
            ints = ps[exact].astype(np.int64)
            np.testing.assert_array_equal(K[exact], seq.K[l, h][ints])   # exact tokens bit-exact
            assert (lm[~exact] > 0).all() or (~exact).sum() == 0 or (lm[~exact] >= 0).all()
    caps, offs = O.offsets(sel.lens[None], 5)
    flat = caps.reshape(-1)
    assert offs.reshape(-1)[0] == 0
    np.testing.assert_array_equal(np.diff(offs.reshape(-1)), flat[:-1])
    # cache bytes: entries x (2 d esize + 8) (K, V, log m, position)
    assert sel.lens.sum() * (2 * cfg.d * 4 + 8) == sel.B_tot * (2 * cfg.d * 4 + 8) or \
        sel.lens.sum() <= sel.B_tot


# ------------------------------------------------------------------ head-level hybrid (R16)
def _hybrid_instance(seed, L=3, H=2):
    util, cost, _, bounds, n = _instance(seed, L=L, H=H)
    rng = np.random.default_rng(1000 + seed)
    # multiples of 1/64: every float64 sum of them is exact, so the ranking is fixed
    r = rng.choice(np.asarray([0.0, 1 / 64, 1 / 32, 5 / 64], np.float32), size=(L, H, n))
    return util, cost, r, bounds, n


def _brute_full(r, end, F):
    L, H, _ = r.shape
    imp = [(sum(float(x) for x in r[l, h, :end]), l * H + h) for l in range(L) for h in range(H)]
    ranked = sorted(imp, key=lambda t: (-t[0], t[1]))
    full = np.zeros(L * H, dtype=bool)
    for _, k in ranked[:F]:
        full[k] = True
    return full.reshape(L, H)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("frac", [0.2, 0.4, 0.5])
def test_hybrid_full_heads_budget_and_lengths(seed, frac):
    util, cost, r, bounds, n = _hybrid_instance(seed)
    L, H = 3, 2
    W, end = n - int(bounds[-1]), int(bounds[-1])
    F = int(math.floor(frac * L * H))
    sens = np.ones((L, H), np.float32)
    sel = O.select_sequence(util, cost, r, sens, bounds, n, W, 0.7, 0, 0.3, -1,
                            head_full_frac=frac)
    full = _brute_full(r, end, F)
    assert full.sum() == F
    np.testing.assert_array_equal(full, O.full_heads(r, end, frac))
    assert sel.taken[full].all()                               # every token exact
    np.testing.assert_array_equal(sel.lens[full], n)
    B_tot, B_alloc, _ = O.budget(n, L, H, W, 0.7, 0, 0.3)
    assert sel.B_alloc == B_alloc - F * (n - W)
    assert int(sel.lens.sum()) <= B_tot                        # the budget holds overall
    assert int(sel.lens[~full].sum()) - W * (L * H - F) == sel.floor_spent + sel.auction_spent
    _tree_closed(sel.taken)


def test_hybrid_off_is_the_plain_selection():
    util, cost, r, bounds, n = _hybrid_instance(3)
    sens = np.ones((3, 2), np.float32)
    W = n - int(bounds[-1])
    a = O.select_sequence(util, cost, r, sens, bounds, n, W, 0.5, 0, 0.3, -1)
    b = O.select_sequence(util, cost, r, sens, bounds, n, W, 0.5, 0, 0.3, -1, head_full_frac=0.0)
    np.testing.assert_array_equal(a.taken, b.taken)


def test_hybrid_with_every_head_full_is_the_full_cache():
    util, cost, r, bounds, n = _hybrid_instance(5)
    sens = np.ones((3, 2), np.float32)
    W = n - int(bounds[-1])
    sel = O.select_sequence(util, cost, r, sens, bounds, n, W, 1.0, 0, 0.3, -1, head_full_frac=1.0)
    assert sel.taken.all() and (sel.lens == n).all() and sel.B_alloc == 0


def test_hybrid_leaving_no_budget_keeps_only_the_other_windows():
    # L*H = 4, F = 2: per-(l,h) budget W + (n - W) / 2 leaves B_alloc = 0
    util, cost, r, bounds, n = _hybrid_instance(6, L=2, H=2)
    W = n - int(bounds[-1])
    per_lh = W + (n - W) // 2
    assert (n - W) % 2 == 0
    sens = np.ones((2, 2), np.float32)
    sel = O.select_sequence(util, cost, r, sens, bounds, n, W, 0.0, per_lh, 0.3, -1,
                            head_full_frac=0.5)
    full = O.full_heads(r, int(bounds[-1]), 0.5)
    assert sel.B_alloc == 0
    np.testing.assert_array_equal(sel.lens[full], n)
    np.testing.assert_array_equal(sel.lens[~full], W)
    assert not sel.taken[~full].any()


def test_floor_never_spends_beyond_the_allocatable_budget(tiny_scored):
    """The floor cap is a hard maximum within the budget ([GK] technical details:
    the singleton cap is a maximum, not a guaranteed spend); even a cap fraction
    above 1 and no token cap cannot make the floor spend more than B_alloc."""
    cfg, wl, seq, scored = tiny_scored
    for beta in (0.15, 0.3):
        sel = _select(cfg, seq, wl.head_sens, scored, budget_ratio=beta, floor_cap_frac=1.5,
                      floor_cap_tokens=-1)
        assert sel.floor_spent <= sel.B_alloc
        assert sel.lens.sum() <= sel.B_tot
        _tree_closed(sel.taken)


def test_offsets_hand_worked():
    """Packed layout: capacity = length + decode reserve per (b, l, h), offsets
    the exclusive prefix sum of the capacities in (b, l, h) order.  Lengths
    (3, 5, 2, 4) with reserve 2: capacities (5, 7, 4, 6), offsets (0, 5, 12, 16)."""
    caps, offs = O.offsets(np.array([[[3, 5], [2, 4]]]), 2)
    np.testing.assert_array_equal(caps.reshape(-1), [5, 7, 4, 6])
    np.testing.assert_array_equal(offs.reshape(-1), [0, 5, 12, 16])
