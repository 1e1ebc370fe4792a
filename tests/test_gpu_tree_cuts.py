"""GPU parity of the curvature-chosen trees (kvc_tree_cuts) and of scoring,
selection and packing on those trees, against the oracle.

kvc_tree_cuts: the key curvature within 2e-5 absolute of the float64 oracle;
every cut bit-exact against the oracle's rule evaluated in fp32 on the device's
curvature (a cut is an integer decided by floating point, so both sides decide
it in the same precision).  Scoring, selection and packing then run on the
device's cut table and are compared with the oracle given the same cuts, with
the tolerances of the midpoint-tree tests.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, token_view, upload_workload

pytestmark = pytest.mark.gpu

KAPPA_ABS = 2e-5


@pytest.fixture(scope="module")
def built():
    from kv_cache_compression_probe_gb300 import build
    build.build()


_WL = {}


def _workload(name):
    if name not in _WL:
        cfg = W.get_config("tiny") if name == "tiny" else W.small_config()
        _WL[name] = W.make_workload(cfg)
    return _WL[name]


def _device_cuts(comp, wl, b, l, h, S):
    """[S, 7] absolute cut positions from the device table."""
    c = comp.cuts[b, l, h, :S, :7].cpu().numpy().astype(np.int64)
    return c + np.asarray(wl.seqs[b].slot_bounds[:S], np.int64)[:, None]


@pytest.fixture(scope="module", params=["tiny", "small-tc", "small-simt"])
def case(request, built):
    from kv_cache_compression_probe_gb300 import kvc
    name = request.param.split("-")[0]
    wl = _workload(name)
    p, comp, d, S_max = upload_workload(wl, tensor_cores=not request.param.endswith("simt"),
                                        tree_cuts=True)
    comp.score(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    return wl, p, comp, d, S_max


def test_key_curvature_and_cuts(case):
    wl, p, comp, d, S_max = case
    cfg = wl.cfg
    kap = comp.tree_kappa.cpu().numpy()
    moved = 0
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        kv = token_view(kap, wl, b)
        for l in range(cfg.L):
            for h in range(cfg.H):
                o = O.key_curvature(s.K[l, h], cfg.rope_base)
                err = np.abs(kv[l, h].astype(np.float64) - o)
                assert err.max() <= KAPPA_ABS, (b, l, h, err.max())
                got = _device_cuts(comp, wl, b, l, h, S)
                want = O.slot_cuts(kv[l, h], s.slot_bounds, np.float32)
                np.testing.assert_array_equal(got, want)
                mid = np.asarray([[((a + c) // 2) for a, c in O.tree_nodes(
                    int(s.slot_bounds[k]), int(s.slot_bounds[k + 1]))[:7]] for k in range(S)])
                moved += int((got != mid).sum())
        assert not comp.cuts[b, :, :, S:].any()
    print(f"cuts off the midpoint: {moved}")
    assert moved > 0                                  # the trees are not all midpoint trees


def _oracle_head(wl, b, l, h, cuts):
    cfg = wl.cfg
    s = wl.seqs[b]
    return O.score_and_value_head(
        s.K[l, h], s.V[l, h], s.Qp[l, h * cfg.G:(h + 1) * cfg.G], s.n, cfg.P, s.slot_bounds,
        float(wl.head_sens[l, h]), base=cfg.rope_base, hop_weight=cfg.hop_weight,
        n_hops=cfg.n_hops, w_part=cfg.w_part, w_value=cfg.w_value,
        value_floor=cfg.value_floor, cuts=cuts)


def test_scoring_on_curvature_trees(case):
    """Op costs bit-exact and utilities within the midpoint tests' tolerance
    against the oracle scored on the device's trees."""
    wl, p, comp, d, S_max = case
    cfg = wl.cfg
    cost = comp.op_cost.cpu().numpy()
    util = comp.op_util.cpu().numpy()
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        for l in range(cfg.L):
            for h in range(cfg.H):
                cuts = _device_cuts(comp, wl, b, l, h, S)
                res = _oracle_head(wl, b, l, h, cuts)
                np.testing.assert_array_equal(cost[b, l, h, :S], res.cost)
                sens = float(wl.head_sens[l, h])
                for k in range(S):
                    nodes = O.tree_nodes(int(s.slot_bounds[k]), int(s.slot_bounds[k + 1]), cuts[k])
                    Rv = np.array([res.r[x:y].sum() for x, y in nodes])
                    scale = np.r_[Rv[0], Rv] * sens / res.cost[k]
                    o = res.util[k]
                    err = np.abs(util[b, l, h, k].astype(np.float64) - o)
                    assert (err <= 1e-5 * np.maximum(np.abs(o), 3 * scale)).all(), (b, l, h, k)


def test_select_and_pack_on_curvature_trees(case):
    """Selection bit-exact against the oracle fed the device's fp32 keys and
    trees; packed entries against the oracle's pack of the same taken set."""
    wl, p, comp, d, S_max = case
    from kv_cache_compression_probe_gb300 import kvc
    cfg = wl.cfg
    comp.select(d["bounds"], d["n_slots"], d["sens"])
    comp.merge_pack(d["K"], d["V"], d["bounds"], d["n_slots"])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    util = comp.op_util.cpu().numpy()
    cost = comp.op_cost.cpu().numpy().astype(np.int64)
    rel = comp.relevance.cpu().numpy()
    taken = comp.taken.cpu().numpy().astype(bool)
    offs = comp.off_lh.cpu().numpy()
    lens = comp.len_lh.cpu().numpy()
    Kp = comp.Kp.float().cpu().numpy(); Vp = comp.Vp.float().cpu().numpy()
    lm = comp.logm.cpu().numpy(); ps = comp.pos.cpu().numpy()
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        r = token_view(rel, wl, b)
        cuts = np.stack([np.stack([_device_cuts(comp, wl, b, l, h, S) for h in range(cfg.H)])
                         for l in range(cfg.L)])
        sel = O.select_sequence(util[b, :, :, :S], cost[b, :, :, :S], r, wl.head_sens,
                                s.slot_bounds, s.n, cfg.W, cfg.budget_ratio,
                                cfg.budget_entries_per_lh, cfg.floor_cap_frac,
                                cfg.floor_cap_tokens, cuts=cuts)
        np.testing.assert_array_equal(taken[b, :, :, :S], sel.taken)
        np.testing.assert_array_equal(lens[b], sel.lens)
        for l in range(cfg.L):
            for h in range(cfg.H):
                K, V, m, pp = O.pack_head(s.K[l, h], s.V[l, h], r[l, h].astype(np.float64),
                                          s.slot_bounds, taken[b, l, h, :S], s.n, cfg.W,
                                          cfg.rope_base, cfg.value_floor, cuts[l, h])
                o, n_ = int(offs[b, l, h]), int(lens[b, l, h])
                assert n_ == len(K)
                np.testing.assert_array_equal(ps[o:o + n_], pp.astype(np.float32))
                exact = m == 0
                np.testing.assert_array_equal(Kp[o:o + n_][exact], K[exact].astype(np.float32))
                if cfg.dtype == "bf16":
                    assert_bf16_close(Kp[o:o + n_], K, "packed K")
                    assert_bf16_close(Vp[o:o + n_], V, "packed V")
                else:
                    assert_f32_close(Kp[o:o + n_], K, "packed K", rel=1e-5, floor_frac=1.0, axis=-1)
                    assert_f32_close(Vp[o:o + n_], V, "packed V", rel=1e-5, floor_frac=1.0, axis=-1)
                np.testing.assert_allclose(lm[o:o + n_], m, rtol=1e-5, atol=1e-6)


def test_invalid_cut_is_reported_and_replaced_by_the_midpoint(built):
    """A cut that would leave a child fewer than 2 tokens per leaf is replaced by
    the midpoint in every kernel (one valid tree) and reported as KVC_EDEVICE."""
    from kv_cache_compression_probe_gb300 import kvc
    wl = _workload("small")
    p, comp, d, S_max = upload_workload(wl, tensor_cores=True, tree_cuts=True)
    kvc.kvc_tree_cuts(p, comp.ctx_len, d["K"], comp.rope_cos, comp.rope_sin, d["bounds"],
                      d["n_slots"], comp.tree_kappa, comp.cuts)
    comp.cuts[0, 0, 0, 0, 0] = 1                     # root cut 1 token into the slot
    comp.cuts[0, 0, 0, 1, 3] = 0                     # a depth-2 cut at its node's start
    kvc.kvc_score(p, comp.ctx_len, d["K"], d["V"], d["Qp"], comp.rope_cos, comp.rope_sin,
                  d["bounds"], d["n_slots"], d["sens"], comp.lse, comp.feats, comp.relevance,
                  comp.op_util, comp.op_cost, comp.ws_score)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == kvc.KVC_EDEVICE
    assert kvc.kvc_device_error() == 0                # read-and-clear
    s = wl.seqs[0]
    cost = comp.op_cost.cpu().numpy()[0, 0, 0]
    for k in (0, 1):
        x0, y0 = int(s.slot_bounds[k]), int(s.slot_bounds[k + 1])
        cuts = [x0 + int(c) for c in comp.cuts[0, 0, 0, k, :7].cpu().numpy()]
        # the replacement: walk the tree, taking the midpoint where a cut is invalid
        nodes = [(x0, y0)]
        for j in range(7):
            a, c = nodes[j]
            depth = 0 if j == 0 else 1 if j < 3 else 2
            leaves = 2 ** (2 - depth)
            t = cuts[j]
            if not (2 * leaves <= t - a <= 16 * leaves and 2 * leaves <= c - t <= 16 * leaves):
                t = (a + c) // 2
            nodes += [(a, t), (t, c)]
        leaf_costs = [b_ - a_ - 1 for a_, b_ in nodes[7:]]
        np.testing.assert_array_equal(cost[k, 8:], leaf_costs)
