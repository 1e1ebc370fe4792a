"""Pins for the three-way salient-token child sets (reading R19, f3; GraceKV
"Technical details and default settings": tree construction may isolate a
salient token with a three-way child set; "Exact-information safeguard": Split
/ Extract of a name-bearing span before the exact leaf).

A depth-2 node [a, b) isolates its most relevant token t when both sides keep
2..15 tokens: children [a, t), token t, [t+1, b); its split costs 2.  Pinned by
hand-worked trees, exhaustive frontier enumeration, the cost/entry identity,
the floor's prefix form, and the full-budget pack equal to the input."""

import numpy as np
import pytest

import oracle as O
from synth import workloads as W
from tests.test_oracle_select import _tree_closed, effective_key_greedy, scan_greedy


def test_salient_token_hand_worked():
    r = np.zeros(64)
    # midpoint tree of [0, 64): depth-2 nodes [0,16) [16,32) [32,48) [48,64)
    r[7] = 5.0                       # node 3: isolate 7 -> leaves [0,7), [8,16)
    r[17] = 4.0                      # node 4: max at 17 = a+1 -> side of 1 token: binary
    r[40] = r[41] = 3.0              # node 5: tie -> the smaller position, 40
    r[50:62] = 0.0                   # node 6: all zero -> argmax 48 = a -> binary
    ext = O.salient_tokens(r, 0, 64)
    assert ext == [7, -1, 40, -1]
    nodes = O.tree_nodes(0, 64, None, ext)
    assert nodes[3] == (0, 16) and nodes[7] == (0, 7) and nodes[8] == (8, 16)
    assert nodes[4] == (16, 32) and nodes[9] == (16, 24) and nodes[10] == (24, 32)
    assert nodes[11] == (32, 40) and nodes[12] == (41, 48)
    D = np.ones(15); Dd = np.full(15, 2.0); Rv = np.ones(15)
    sizes = np.array([b - a for a, b in nodes])
    util, cost = O.slot_ops(D, Dd, Rv, sizes, 1.0, ext)
    assert list(cost) == [1, 1, 1, 1, 2, 1, 2, 1, 6, 7, 7, 7, 7, 6, 7, 7]
    # the three-way gain: (D(N) - D(left) - D(right)) / D_drop(N), clamped
    D2 = D.copy(); D2[3] = 1.5; D2[7] = 0.25; D2[8] = 0.5
    u2, _ = O.slot_ops(D2, Dd, Rv, sizes, 1.0, ext)
    assert u2[1 + 3] == pytest.approx((1.5 - 0.75) / 2.0 / 2)


def test_extract_validity_bounds():
    assert O.extract_valid(2, 0, 5) and not O.extract_valid(1, 0, 5)
    assert not O.extract_valid(3, 0, 5)              # right side would be 1 token
    assert O.extract_valid(15, 0, 31) and not O.extract_valid(15, 0, 32)   # right 16 tokens
    assert not O.extract_valid(16, 0, 32)            # left 16 tokens
    with pytest.raises(ValueError):
        O.tree_nodes(0, 64, None, [1, -1, -1, -1])


def _random_tree(rng, c):
    x0 = int(rng.integers(0, 50))
    r = rng.exponential(size=x0 + c + 5)
    ext = O.salient_tokens(r, x0, x0 + c)
    return x0, x0 + c, ext


@pytest.mark.parametrize("c", [16, 20, 37, 64, 90, 112, 124, 128])
def test_leaves_and_salient_tokens_partition_the_slot(c):
    rng = np.random.default_rng(c)
    for _ in range(20):
        x0, y0, ext = _random_tree(rng, c)
        nodes = O.tree_nodes(x0, y0, None, ext)
        pieces = []
        for j in range(3, 7):
            a, b = nodes[j]
            la, lb = nodes[2 * j + 1]
            ra, rb = nodes[2 * j + 2]
            t = ext[j - 3]
            if t >= 0:
                assert (la, lb, ra, rb) == (a, t, t + 1, b) and 2 <= lb - la <= 15
                assert 2 <= rb - ra <= 15
                pieces += [(la, lb), (t, t + 1), (ra, rb)]
            else:
                assert lb == ra and la == a and rb == b
                pieces += [(la, lb), (ra, rb)]
        flat = [i for a, b in pieces for i in range(a, b)]
        assert flat == list(range(x0, y0))
        if c == 128:
            assert ext == [-1] * 4                     # 32-token depth-2 nodes: no room
        for j in range(3, 7):
            a, b = nodes[j]
            if b - a == 31 and ext[j - 3] >= 0:
                assert ext[j - 3] == a + 15            # the one position with 15 + 15


def _all_closed_takens(k_ops=16):
    """Every taken set of one tree closed under op parents (Add first)."""
    out = []
    for bits in range(1 << 8):
        t = np.zeros(16, dtype=bool)
        t[0] = True
        # internal splits 1..7 from the bits, leaves all taken where exposed
        for j in range(7):
            t[1 + j] = bool((bits >> j) & 1)
        ok = all(not t[1 + j] or (j == 0 or t[1 + O.node_parent(j)]) for j in range(7))
        if not ok:
            continue
        for leaf_bits in (0, 0x55, 0xFF):
            u = t.copy()
            for k in range(8):
                j = 7 + k
                u[1 + j] = bool((leaf_bits >> k) & 1) and u[1 + O.node_parent(j)]
            out.append(u)
    return out


def test_frontier_covers_the_slot_once_in_order_and_entries_equal_costs():
    rng = np.random.default_rng(7)
    for c in (40, 64, 77):
        x0, y0, ext = _random_tree(rng, c)
        assert any(t >= 0 for t in ext)
        nodes = O.tree_nodes(x0, y0, None, ext)
        sizes = np.array([b - a for a, b in nodes])
        _, cost = O.slot_ops(np.zeros(15), np.ones(15), np.ones(15), sizes, 1.0, ext)
        for t in _all_closed_takens():
            fr = O.frontier(t, x0, y0, None, ext)
            span = []
            for kind, j in fr:
                span += [j] if kind == "tok" else list(range(*nodes[j]))
            assert span == list(range(x0, y0))
            assert len(fr) == int((t * cost).sum())   # entries = costs of the taken ops
        full = O.frontier(np.ones(16, bool), x0, y0, None, ext)
        assert full == [("tok", i) for i in range(x0, y0)]


def _instance_salient(seed, L=2, H=2, bounds=(0, 16, 48, 112, 176)):
    rng = np.random.default_rng(seed)
    bounds = np.asarray(bounds)
    S = len(bounds) - 1
    n = int(bounds[-1]) + 8
    r = rng.choice(np.asarray([0.0, 0.01, 0.02, 0.05, 0.3], np.float32), size=(L, H, n))
    util = rng.choice(np.float32([0.0, 0.1, 0.2, 0.5]), size=(L, H, S, 16))
    cost = np.zeros((L, H, S, 16), dtype=np.int64)
    ext = np.full((L, H, S, 4), -1, dtype=np.int64)
    for l in range(L):
        for h in range(H):
            for s in range(S):
                x0, y0 = int(bounds[s]), int(bounds[s + 1])
                ext[l, h, s] = O.salient_tokens(r[l, h], x0, y0)
                nodes = O.tree_nodes(x0, y0, None, ext[l, h, s])
                sizes = np.array([b - a for a, b in nodes])
                cost[l, h, s] = O.slot_ops(np.zeros(15), np.ones(15), np.ones(15), sizes, 1.0,
                                           ext[l, h, s])[1]
    return util, cost, r, bounds, n, ext


def _floor_prefix_salient(r, sens, bounds, cost, cap_entries, ext):
    """The floor in prefix form on three-way trees: a candidate's path ends at
    the node whose split makes it exact (its leaf, or the depth-2 node that
    isolates it); its cost counts the path ops not opened by an earlier taken
    candidate."""
    L, H, n = r.shape
    end = int(bounds[-1])
    cands = sorted((-float(np.float32(r[l, h, i]) * np.float32(sens[l, h])), (l * H + h) * n + i,
                    l, h, i) for l in range(L) for h in range(H) for i in range(end)
                   if r[l, h, i] > 0)
    seen, spent, tokens = set(), 0, 0
    taken = np.zeros(cost.shape, dtype=bool)
    for _, _, l, h, i in cands:
        s = int(np.searchsorted(bounds, i, side="right") - 1)
        nodes = O.tree_nodes(int(bounds[s]), int(bounds[s + 1]), None, ext[l, h, s])
        j, path = 0, [0]
        while j < 7 and not (j >= 3 and ext[l, h, s, j - 3] == i):
            j = 2 * j + 1 if i < nodes[2 * j + 1][1] else 2 * j + 2
            path.append(j)
        if (l, h, s, j) in seen:
            continue
        c = (0 if (l, h, s, "add") in seen else int(cost[l, h, s, 0])) + sum(
            int(cost[l, h, s, 1 + k]) for k in path if (l, h, s, k) not in seen)
        if spent + c > cap_entries:
            break
        spent += c
        tokens += 1
        seen.update({(l, h, s, k) for k in path} | {(l, h, s, "add")})
        taken[l, h, s, [0] + [1 + k for k in path]] = True
    return taken, spent, tokens


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("cap", [3, 5, 11, 40, 500])
def test_floor_on_three_way_trees_equals_prefix_form(seed, cap):
    util, cost, r, bounds, n, ext = _instance_salient(seed)
    assert (ext >= 0).any()
    sens = np.ones(r.shape[:2], np.float32)
    t1 = np.zeros(cost.shape, dtype=bool)
    sp, tk = O.singleton_floor(r, sens, bounds, cost, cap, -1, t1, None, ext)
    t2, sp2, tk2 = _floor_prefix_salient(r, sens, bounds, cost, cap, ext)
    np.testing.assert_array_equal(t1, t2)
    assert (sp, tk) == (sp2, tk2) and sp <= cap
    assert (t1 * cost).sum() == sp
    _tree_closed(t1)


def test_floor_path_of_a_salient_token_stops_at_its_depth2_node():
    r = np.zeros((1, 1, 72), np.float32)
    r[0, 0, 7] = 1.0                                  # salient in node 3 of the slot [0, 64)
    bounds = np.array([0, 64])
    ext = np.asarray(O.salient_tokens(r[0, 0], 0, 64))[None, None, None]
    assert ext[0, 0, 0, 0] == 7
    nodes = O.tree_nodes(0, 64, None, ext[0, 0, 0])
    sizes = np.array([b - a for a, b in nodes])
    cost = O.slot_ops(np.zeros(15), np.ones(15), np.ones(15), sizes, 1.0, ext[0, 0, 0])[1][None, None, None]
    for cap, want in ((4, 0), (5, 1)):                # Add + root + node 1 + node 3 (cost 2)
        t = np.zeros((1, 1, 1, 16), dtype=bool)
        sp, tk = O.singleton_floor(r, np.ones((1, 1), np.float32), bounds, cost, cap, -1, t,
                                   None, ext)
        assert tk == want and sp == 5 * want
        if want:
            fr = O.frontier(t[0, 0, 0], 0, 64, None, ext[0, 0, 0])
            assert ("tok", 7) in fr and not t[0, 0, 0, 1 + 7] and not t[0, 0, 0, 1 + 8]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("budget_frac", [0.1, 0.5, 1.0])
def test_auction_on_three_way_trees_equals_scan_and_effective_key(seed, budget_frac):
    util, cost, r, bounds, n, ext = _instance_salient(seed)
    rem = int(budget_frac * int(cost.sum()))
    t1, t2, t3 = (np.zeros(cost.shape, dtype=bool) for _ in range(3))
    spent = O.greedy_auction(util, cost, t1, rem)
    assert rem - spent == scan_greedy(util, cost, t2, rem) == effective_key_greedy(util, cost, t3, rem)
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_array_equal(t1, t3)


def test_full_budget_with_three_way_trees_packs_the_input():
    """With every depth-2 node free to isolate its salient token, a full budget
    still takes every op and the pack is the input, bit for bit ([GK] "05":
    at FullKV scale every tree expands to token leaves)."""
    cfg = W.get_config("tiny").replace(budget_ratio=1.0)
    wl = W.make_workload(cfg)
    s = wl.seqs[0]
    util = np.zeros((1, 2, len(s.slot_bounds) - 1, 16)); cost = np.zeros_like(util, dtype=np.int64)
    rr = np.zeros((1, 2, s.n)); ext = np.zeros((1, 2, len(s.slot_bounds) - 1, 4), np.int64)
    for h in range(2):
        res = O.score_and_value_head(s.K[0, h], s.V[0, h], s.Qp[0, h * cfg.G:(h + 1) * cfg.G], s.n,
                                     cfg.P, s.slot_bounds, 1.0, base=cfg.rope_base, salient=True)
        util[0, h], cost[0, h], rr[0, h], ext[0, h] = res.util, res.cost, res.r, res.extract
    assert (ext >= 0).sum() > 0
    assert ((cost.sum(axis=-1) == np.diff(s.slot_bounds)[None, None])).all()
    sel = O.select_sequence(util, cost, rr, wl.head_sens, s.slot_bounds, s.n, cfg.W, 1.0, 0,
                            cfg.floor_cap_frac, cfg.floor_cap_tokens, extract=ext)
    assert sel.taken.all()
    for h in range(2):
        K, V, lm, ps = O.pack_head(s.K[0, h], s.V[0, h], rr[0, h], s.slot_bounds, sel.taken[0, h],
                                   s.n, cfg.W, cfg.rope_base, cfg.value_floor, None, ext[0, h])
        np.testing.assert_array_equal(K, s.K[0, h])
        np.testing.assert_array_equal(V, s.V[0, h])
        assert (lm == 0).all() and (ps == np.arange(s.n)).all()


def test_salient_relevance_counts_in_its_node_values_and_prototypes():
    """The isolated token belongs to its depth-2 node and the node's ancestors
    (values sum up the tree, [GK] "03 Bottom-up value flow") but to no leaf."""
    cfg = W.get_config("tiny")
    wl = W.make_workload(cfg)
    s = wl.seqs[0]
    res = O.score_and_value_head(s.K[0, 0], s.V[0, 0], s.Qp[0, :cfg.G], s.n, cfg.P, s.slot_bounds,
                                 1.0, base=cfg.rope_base, salient=True)
    for k in range(len(s.slot_bounds) - 1):
        x0, y0 = int(s.slot_bounds[k]), int(s.slot_bounds[k + 1])
        ext = res.extract[k]
        nodes = O.tree_nodes(x0, y0, None, ext)
        Rv = res.Rv[k]
        for j in range(7):
            extra = res.r[ext[j - 3]] if (j >= 3 and ext[j - 3] >= 0) else 0.0
            assert Rv[j] == pytest.approx(Rv[2 * j + 1] + Rv[2 * j + 2] + extra, rel=1e-12)
        assert Rv[0] == pytest.approx(res.r[x0:y0].sum(), rel=1e-12)
        for j in range(3, 7):
            if ext[j - 3] >= 0:
                a, b = nodes[j]
                assert res.r[a:b].argmax() + a == ext[j - 3]
