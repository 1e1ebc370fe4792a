"""GPU parity of kvc_score, kvc_select and kvc_merge_pack against the oracle.

Per-call parity: every call is compared with the oracle fed the same inputs
(select gets the GPU's fp32 utilities and relevance; pack gets the same taken
set).  End-to-end: the GPU's chain against the oracle's own chain, with any
difference in the taken set explained by near-ties of the oracle's keys.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import (assert_bf16_close, assert_f32_close, token_view, upload_workload)
from tests.oracle_pipeline import score_all

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from kv_cache_compression_probe_gb300 import build
    build.build()


def _cases():
    return {
        "tiny": W.get_config("tiny"),
        "small": W.small_config(),
    }


_ORACLE = {}


@pytest.fixture(scope="module", params=["tiny", "small-tc", "small-simt"])
def case(request, built):
    """tiny: fp32, d 64 (SIMT scoring); small: bf16, d 128, scored with the
    tcgen05 passes (small-tc) and with the SIMT passes (small-simt)."""
    name = request.param.split("-")[0]
    cfg = _cases()[name]
    if name not in _ORACLE:
        wl = W.make_workload(cfg)
        _ORACLE[name] = (wl, score_all(wl))
    wl, run = _ORACLE[name]
    p, comp, d, S_max = upload_workload(wl, tensor_cores=not request.param.endswith("simt"))
    comp.score(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    from kv_cache_compression_probe_gb300 import kvc
    assert kvc.kvc_device_error() == 0
    return cfg, wl, run, p, comp, d, S_max


def test_score_row_stats(case):
    cfg, wl, run, p, comp, d, S_max = case
    assert_f32_close(comp.lse.cpu().numpy(), run.lse, "lse", rel=1e-5)


def test_score_features_and_relevance(case):
    cfg, wl, run, p, comp, d, S_max = case
    feats = comp.feats.cpu().numpy()
    rel = comp.relevance.cpu().numpy()
    for b in range(cfg.B):
        f = token_view(feats, wl, b, 5)
        r = token_view(rel, wl, b)
        for k, name in enumerate(["alpha", "|v|", "sigma", "H", "pos"]):
            assert_f32_close(f[..., k], run.feats[b][..., k], name, rel=1e-5, axis=-1)
        assert_f32_close(r, run.r[b], "relevance", rel=1e-5, axis=-1)


def test_score_utilities(case):
    cfg, wl, run, p, comp, d, S_max = case
    cost = comp.op_cost.cpu().numpy()
    util = comp.op_util.cpu().numpy()
    np.testing.assert_array_equal(cost, run.cost)
    # A utility is scale * gain with scale = R(N) * sens / cost and gain in [0, 1]
    # a clamped difference of normalised distortions, so fp32 reaches it to an
    # absolute accuracy relative to the scale (cancellation), not to |u|:
    # |g - o| <= 1e-5 * max(|o|, 3 * scale).
    scale_only = 0
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        for l in range(cfg.L):
            for h in range(cfg.H):
                r = run.r[b][l, h]
                sens = float(wl.head_sens[l, h])
                for k in range(S):
                    nodes = O.tree_nodes(int(s.slot_bounds[k]), int(s.slot_bounds[k + 1]))
                    Rv = np.array([r[x:y].sum() for x, y in nodes])
                    scale = np.r_[Rv[0], Rv] * sens / run.cost[b, l, h, k]
                    o = run.util[b, l, h, k]
                    err = np.abs(util[b, l, h, k].astype(np.float64) - o)
                    assert (err <= 1e-5 * np.maximum(np.abs(o), 3 * scale)).all(), (b, l, h, k, err, o)
                    scale_only += int(((err > 1e-5 * np.abs(o))).sum())
    print(f"ops within tolerance only through the scale term: {scale_only}")


def test_select_bit_exact_on_gpu_utilities(case):
    """Selection is bit-exact against the oracle fed the GPU's fp32 keys."""
    cfg, wl, run, p, comp, d, S_max = case
    comp.select(d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    from kv_cache_compression_probe_gb300 import kvc
    assert kvc.kvc_device_error() == 0
    util = comp.op_util.cpu().numpy()
    cost = comp.op_cost.cpu().numpy().astype(np.int64)
    rel = comp.relevance.cpu().numpy()
    taken = comp.taken.cpu().numpy().astype(bool)
    lens = np.zeros((cfg.B, cfg.L, cfg.H), np.int64)
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        sel = O.select_sequence(util[b, :, :, :S], cost[b, :, :, :S], token_view(rel, wl, b),
                                wl.head_sens, s.slot_bounds, s.n, cfg.W, cfg.budget_ratio,
                                cfg.budget_entries_per_lh, cfg.floor_cap_frac, cfg.floor_cap_tokens)
        np.testing.assert_array_equal(taken[b, :, :, :S], sel.taken)
        assert not taken[b, :, :, S:].any()
        lens[b] = sel.lens
    np.testing.assert_array_equal(comp.len_lh.cpu().numpy(), lens)
    caps, offs = O.offsets(lens, cfg.decode_reserve)
    np.testing.assert_array_equal(comp.cap_lh.cpu().numpy(), caps)
    np.testing.assert_array_equal(comp.off_lh.cpu().numpy(), offs)
    assert int(comp.total.cpu()[0]) == int(caps.sum())


def test_pack_matches_oracle(case):
    cfg, wl, run, p, comp, d, S_max = case
    comp.select(d["bounds"], d["n_slots"], d["sens"])
    comp.merge_pack(d["K"], d["V"], d["bounds"], d["n_slots"])
    torch.cuda.synchronize()
    from kv_cache_compression_probe_gb300 import kvc
    assert kvc.kvc_device_error() == 0
    taken = comp.taken.cpu().numpy().astype(bool)
    rel = comp.relevance.cpu().numpy()
    offs = comp.off_lh.cpu().numpy()
    lens = comp.len_lh.cpu().numpy()
    Kp = comp.Kp.float().cpu().numpy(); Vp = comp.Vp.float().cpu().numpy()
    lm = comp.logm.cpu().numpy(); ps = comp.pos.cpu().numpy()
    rel_only = 0
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        r = token_view(rel, wl, b)
        for l in range(cfg.L):
            for h in range(cfg.H):
                K, V, m, pp = O.pack_head(s.K[l, h], s.V[l, h], r[l, h].astype(np.float64),
                                          s.slot_bounds, taken[b, l, h, :S], s.n, cfg.W,
                                          cfg.rope_base, cfg.value_floor)
                o, n_ = int(offs[b, l, h]), int(lens[b, l, h])
                assert n_ == len(K)
                np.testing.assert_array_equal(ps[o:o + n_], pp.astype(np.float32))
                exact = m == 0
                np.testing.assert_array_equal(Kp[o:o + n_][exact], K[exact].astype(np.float32))
                np.testing.assert_array_equal(Vp[o:o + n_][exact], V[exact].astype(np.float32))
                if cfg.dtype == "bf16":
                    rel_only += assert_bf16_close(Kp[o:o + n_], K, "packed K")
                    rel_only += assert_bf16_close(Vp[o:o + n_], V, "packed V")
                else:
                    assert_f32_close(Kp[o:o + n_], K, "packed K", rel=1e-5, floor_frac=1.0, axis=-1)
                    assert_f32_close(Vp[o:o + n_], V, "packed V", rel=1e-5, floor_frac=1.0, axis=-1)
                np.testing.assert_allclose(lm[o:o + n_], m, rtol=1e-5, atol=1e-6)
    print(f"elements passing only through the relative bf16 term: {rel_only}")


def test_end_to_end_taken_set_against_oracle_chain(case):
    """The GPU chain's taken set equals the oracle chain's (float64 keys) except
    where near-ties (keys within 1e-6 relative) fell the other way: the device's
    set must be the oracle's selection under one resolution of those ties (the
    device's own key order inside each near-tie run); every differing op is a
    reported tie.  Any other difference fails."""
    cfg, wl, run, p, comp, d, S_max = case
    from tests.tie_check import band_needed, check_sequence
    comp.select(d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    taken = comp.taken.cpu().numpy().astype(bool)
    util = comp.op_util.cpu().numpy()
    rel = comp.relevance.cpu().numpy()
    cost = comp.op_cost.cpu().numpy().astype(np.int64)
    ties = 0
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        args = (run.util[b, :, :, :S], util[b, :, :, :S], cost[b, :, :, :S], run.r[b],
                token_view(rel, wl, b), wl.head_sens, taken[b, :, :, :S], s.slot_bounds, s.n, cfg)
        try:
            rep = check_sequence(*args)
        except AssertionError as e:
            raise AssertionError(f"sequence {b}: {e}; band needed: {band_needed(*args)}") from None
        assert not taken[b, :, :, S:].any()
        ties += rep.diff_ops
    print(f"end-to-end: taken bits differing from the oracle chain through 1e-6 ties: {ties}")


def test_full_budget_packs_the_input_bit_exact(built):
    cfg = W.get_config("tiny").replace(budget_ratio=1.0)
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl)
    comp.compress(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert bool(comp.taken[..., :].bool().all())
    offs = comp.off_lh.cpu().numpy(); lens = comp.len_lh.cpu().numpy()
    s = wl.seqs[0]
    for l in range(cfg.L):
        for h in range(cfg.H):
            o, n_ = int(offs[0, l, h]), int(lens[0, l, h])
            assert n_ == s.n
            np.testing.assert_array_equal(comp.Kp[o:o + n_].cpu().numpy(), s.K[l, h])
            np.testing.assert_array_equal(comp.Vp[o:o + n_].cpu().numpy(), s.V[l, h])
            assert (comp.logm[o:o + n_].cpu().numpy() == 0).all()


def test_window_only_budget(built):
    cfg = W.get_config("tiny")
    cfg = cfg.replace(budget_ratio=cfg.W / cfg.n)
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl)
    comp.compress(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert not bool(comp.taken.bool().any())
    assert (comp.len_lh.cpu().numpy() == cfg.W).all()


def test_phase_timing_reports_the_tensor_core_phases(built):
    """kvc_set_phase_timing / kvc_score_phase_ms: a timed tensor-core kvc_score
    call reports five positive phase durations whose sum stays within the
    call's own event-timed duration; results are the same as untimed."""
    from kv_cache_compression_probe_gb300 import kvc
    cfg = W.small_config()
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl, tensor_cores=True)
    comp.score(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    ref = comp.op_util.clone()
    kvc.kvc_set_phase_timing(True)
    try:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        comp.score(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
        e1.record()
        ms = kvc.kvc_score_phase_ms(5)
    finally:
        kvc.kvc_set_phase_timing(False)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    assert len(ms) == 5 and all(x > 0.0 for x in ms)
    assert sum(ms) <= e0.elapsed_time(e1) * 1.01 + 1e-3
    assert torch.equal(comp.op_util, ref)
    assert kvc.kvc_score_phase_ms(2) == ms[:2]     # the last timed call, re-read


def test_compression_graph_replay_equals_eager(built):
    """Compressor.compress(graph=True): the captured score, select and pack
    calls replayed (twice) give the eager calls' results bit for bit."""
    from kv_cache_compression_probe_gb300 import kvc
    cfg = W.small_config()
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl, tensor_cores=True)
    args = (d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    comp.compress(*args)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (comp.op_util, comp.taken, comp.len_lh, comp.Kp, comp.Vp, comp.logm)]
    for _ in range(2):
        comp.compress(*args, graph=True)
        torch.cuda.synchronize()
        assert kvc.kvc_device_error() == 0
        got = (comp.op_util, comp.taken, comp.len_lh, comp.Kp, comp.Vp, comp.logm)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    assert comp.graph_launches > 0


@pytest.mark.parametrize("tree_cuts", [False, True])
def test_compress_from_host_equals_compress(built, tree_cuts):
    """Compressor.compress_from_host (layer chunks copied on a second stream while
    earlier chunks are scored) gives exactly the outputs of copying everything
    first and calling compress(); with curvature-chosen trees each chunk cuts
    its own layers' trees into its slice of the cut table."""
    from kv_cache_compression_probe_gb300 import kvc
    cfg = W.small_config(B=1, L=4, H=2, n=1500, n_min=1500)
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl, tensor_cores=True, tree_cuts=tree_cuts)
    comp.compress(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    ref = [t.clone() for t in (comp.lse, comp.feats, comp.op_util, comp.taken, comp.len_lh,
                               comp.Kp, comp.Vp, comp.logm, comp.pos)]
    if tree_cuts:
        ref += [comp.cuts.clone(), comp.tree_kappa.clone()]
        comp.cuts.zero_()
    h = [t.cpu().pin_memory() for t in (d["K"], d["V"], d["Qp"])]
    K2, V2, Q2 = (torch.zeros_like(d["K"]), torch.zeros_like(d["V"]), torch.zeros_like(d["Qp"]))
    comp.compress_from_host(h[0], h[1], h[2], K2, V2, Q2, d["bounds"], d["n_slots"], d["sens"],
                            chunks=3, copy_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    assert torch.equal(K2, d["K"]) and torch.equal(V2, d["V"]) and torch.equal(Q2, d["Qp"])
    got = [comp.lse, comp.feats, comp.op_util, comp.taken, comp.len_lh, comp.Kp, comp.Vp,
           comp.logm, comp.pos]
    if tree_cuts:
        got += [comp.cuts, comp.tree_kappa]
    assert len(got) == len(ref)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
