"""GPU parity of the three-way salient-token child sets (reading R19, f3),
against the oracle, on midpoint and on curvature-chosen trees, with the
tensor-core and the SIMT scoring paths.

The choice of the isolated token is an integer decided by comparing float32
relevances, so it is checked bit-exact against the oracle's rule applied to
the device's relevance.  Then, with the device's trees: op costs bit-exact,
utilities within the tolerance of the midpoint tests, the selection bit-exact
on the device's fp32 keys, and the packed entries against the oracle's pack of
the same taken set; a full budget packs the input bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, token_view, upload_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from kv_cache_compression_probe_gb300 import build
    build.build()


_WL = {}


# slot lengths whose depth-2 nodes span every case of the three-way rule: 4
# tokens (never), 5 (only t = a + 2), 6..8, 15..16, 31 (only t = a + 15), 32
# (never), 18..19
EDGE_SLOTS = (16, 20, 24, 31, 62, 124, 128, 75)


def _workload(name):
    if name not in _WL:
        if name == "edges":
            wl = W.make_workload(W.get_config("tiny"))
            s = wl.seqs[0]
            assert sum(EDGE_SLOTS) == s.n - wl.cfg.W
            s.slot_bounds = np.concatenate([[0], np.cumsum(EDGE_SLOTS)]).astype(np.int32)
            _WL[name] = wl
        else:
            cfg = W.get_config("tiny") if name == "tiny" else W.small_config()
            _WL[name] = W.make_workload(cfg)
    return _WL[name]


def _device_trees(comp, wl, b, l, h, S, curvature):
    """(binary cuts [S, 7] absolute or None, extract [S, 4] absolute or -1) from
    the device's cut table."""
    tab = comp.cuts[b, l, h, :S].cpu().numpy().astype(np.int64)
    x0 = np.asarray(wl.seqs[b].slot_bounds[:S], np.int64)
    flags = tab[:, 7]
    ext = np.full((S, 4), -1, np.int64)
    for j in range(3, 7):
        on = (flags >> (j - 3)) & 1
        ext[:, j - 3] = np.where(on == 1, x0 + tab[:, j], -1)
    cuts = (tab[:, :7] + x0[:, None]) if curvature else None
    return cuts, ext


@pytest.fixture(scope="module",
                params=["tiny", "small-tc", "small-simt", "small-tc-curv", "tiny-curv", "edges",
                        "edges-curv"])
def case(request, built):
    from kv_cache_compression_probe_gb300 import kvc
    name = request.param.split("-")[0]
    curvature = request.param.endswith("curv")
    wl = _workload(name)
    p, comp, d, S_max = upload_workload(wl, tensor_cores="simt" not in request.param,
                                        tree_cuts=curvature, salient=True)
    comp.score(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    return wl, p, comp, d, S_max, curvature


def test_salient_choice_bit_exact(case):
    wl, p, comp, d, S_max, curvature = case
    cfg = wl.cfg
    rel = comp.relevance.cpu().numpy()
    n_ext = 0
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        r = token_view(rel, wl, b)
        for l in range(cfg.L):
            for h in range(cfg.H):
                cuts, ext = _device_trees(comp, wl, b, l, h, S, curvature)
                for k in range(S):
                    want = O.salient_tokens(r[l, h].astype(np.float64), int(s.slot_bounds[k]),
                                            int(s.slot_bounds[k + 1]),
                                            None if cuts is None else cuts[k])
                    np.testing.assert_array_equal(ext[k], want, err_msg=f"{(b, l, h, k)}")
                n_ext += int((ext >= 0).sum())
        assert not comp.cuts[b, :, :, S:].any()
    print(f"depth-2 nodes isolating a salient token: {n_ext}")
    assert n_ext > 0


def _oracle_head(wl, b, l, h, cuts, r_dev):
    cfg = wl.cfg
    s = wl.seqs[b]
    return O.score_and_value_head(
        s.K[l, h], s.V[l, h], s.Qp[l, h * cfg.G:(h + 1) * cfg.G], s.n, cfg.P, s.slot_bounds,
        float(wl.head_sens[l, h]), base=cfg.rope_base, hop_weight=cfg.hop_weight,
        n_hops=cfg.n_hops, w_part=cfg.w_part, w_value=cfg.w_value,
        value_floor=cfg.value_floor, cuts=cuts, salient=True, salient_r=r_dev)


def test_scoring_on_three_way_trees(case):
    """Relevance as without extraction; op costs bit-exact and utilities within
    the midpoint tests' tolerance against the oracle on the device's trees."""
    wl, p, comp, d, S_max, curvature = case
    cfg = wl.cfg
    cost = comp.op_cost.cpu().numpy()
    util = comp.op_util.cpu().numpy()
    rel = comp.relevance.cpu().numpy()
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        r = token_view(rel, wl, b)
        for l in range(cfg.L):
            for h in range(cfg.H):
                cuts, ext = _device_trees(comp, wl, b, l, h, S, curvature)
                res = _oracle_head(wl, b, l, h, cuts, r[l, h].astype(np.float64))
                np.testing.assert_array_equal(res.extract, ext)
                assert_f32_close(r[l, h], res.r, "relevance", rel=1e-5)
                np.testing.assert_array_equal(cost[b, l, h, :S], res.cost)
                sens = float(wl.head_sens[l, h])
                for k in range(S):
                    nodes = O.tree_nodes(int(s.slot_bounds[k]), int(s.slot_bounds[k + 1]),
                                         None if cuts is None else cuts[k], ext[k])
                    Rv = np.array([res.r[x:y].sum() for x, y in nodes])   # depth-2 spans hold t
                    scale = np.r_[Rv[0], Rv] * sens / res.cost[k]
                    o = res.util[k]
                    err = np.abs(util[b, l, h, k].astype(np.float64) - o)
                    assert (err <= 1e-5 * np.maximum(np.abs(o), 3 * scale)).all(), (b, l, h, k)


def test_select_and_pack_on_three_way_trees(case):
    """Selection bit-exact against the oracle fed the device's fp32 keys and
    trees; packed entries against the oracle's pack of the same taken set."""
    wl, p, comp, d, S_max, curvature = case
    cfg = wl.cfg
    from kv_cache_compression_probe_gb300 import kvc
    comp.select(d["bounds"], d["n_slots"], d["sens"])
    comp.merge_pack(d["K"], d["V"], d["bounds"], d["n_slots"])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    util = comp.op_util.cpu().numpy()
    cost = comp.op_cost.cpu().numpy().astype(np.int64)
    rel = comp.relevance.cpu().numpy()
    taken = comp.taken.cpu().numpy().astype(bool)
    lens = comp.len_lh.cpu().numpy()
    offs = comp.off_lh.cpu().numpy()
    Kp = comp.Kp.float().cpu().numpy(); Vp = comp.Vp.float().cpu().numpy()
    lm = comp.logm.cpu().numpy(); ps = comp.pos.cpu().numpy()
    floor_salient = 0
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        r = token_view(rel, wl, b)
        trees = [[_device_trees(comp, wl, b, l, h, S, curvature) for h in range(cfg.H)]
                 for l in range(cfg.L)]
        cuts = None if not curvature else np.stack([[t[0] for t in row] for row in trees])
        ext = np.stack([[t[1] for t in row] for row in trees])
        sel = O.select_sequence(util[b, :, :, :S], cost[b, :, :, :S], r, wl.head_sens,
                                s.slot_bounds, s.n, cfg.W, cfg.budget_ratio,
                                cfg.budget_entries_per_lh, cfg.floor_cap_frac,
                                cfg.floor_cap_tokens, cuts=cuts, extract=ext)
        np.testing.assert_array_equal(taken[b, :, :, :S], sel.taken)
        np.testing.assert_array_equal(lens[b], sel.lens)
        for l in range(cfg.L):
            for h in range(cfg.H):
                K, V, m, pp = O.pack_head(s.K[l, h], s.V[l, h], r[l, h].astype(np.float64),
                                          s.slot_bounds, taken[b, l, h, :S], s.n, cfg.W,
                                          cfg.rope_base, cfg.value_floor,
                                          None if cuts is None else cuts[l, h], ext[l, h])
                o, n_ = int(offs[b, l, h]), int(lens[b, l, h])
                assert n_ == len(K)
                np.testing.assert_array_equal(ps[o:o + n_], pp.astype(np.float32))
                exact = m == 0
                np.testing.assert_array_equal(Kp[o:o + n_][exact], K[exact].astype(np.float32))
                np.testing.assert_array_equal(Vp[o:o + n_][exact], V[exact].astype(np.float32))
                if cfg.dtype == "bf16":
                    assert_bf16_close(Kp[o:o + n_], K, "packed K")
                    assert_bf16_close(Vp[o:o + n_], V, "packed V")
                else:
                    assert_f32_close(Kp[o:o + n_], K, "packed K", rel=1e-5, floor_frac=1.0, axis=-1)
                    assert_f32_close(Vp[o:o + n_], V, "packed V", rel=1e-5, floor_frac=1.0, axis=-1)
                np.testing.assert_allclose(lm[o:o + n_], m, rtol=1e-5, atol=1e-6)
        # three-way depth-2 splits taken: their isolated tokens are stored exact
        floor_salient += int((taken[b, :, :, :S, 4:8] & (ext >= 0)).sum())
    print(f"isolated tokens stored exact: {floor_salient}")


def test_full_budget_packs_the_input_with_three_way_trees(built):
    cfg = W.get_config("tiny").replace(budget_ratio=1.0)
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl, salient=True)
    comp.compress(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert bool(comp.taken.bool().all())
    assert int(comp.cuts[..., 7].bool().sum()) > 0
    s = wl.seqs[0]
    offs = comp.off_lh.cpu().numpy(); lens = comp.len_lh.cpu().numpy()
    for l in range(cfg.L):
        for h in range(cfg.H):
            o, n_ = int(offs[0, l, h]), int(lens[0, l, h])
            assert n_ == s.n
            np.testing.assert_array_equal(comp.Kp[o:o + n_].cpu().numpy(), s.K[l, h])
            np.testing.assert_array_equal(comp.Vp[o:o + n_].cpu().numpy(), s.V[l, h])
            assert (comp.logm[o:o + n_].cpu().numpy() == 0).all()
