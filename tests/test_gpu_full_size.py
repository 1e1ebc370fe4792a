"""Full-size parity: every workload at the sizes of the benchmark and the pages,
run through the path in the benchmark's launch configuration (tensor-core
scoring, selection, pack, then the decode steps replayed as one CUDA graph),
and checked against the float64 oracle on sampled (layer, KV head) pairs plus
checks that hold at any size:
  * probe LSE, features, relevance, op costs and utilities of sampled pairs;
  * the selection of every sequence, bit-exact against the oracle run on the
    device's fp32 keys (the budget couples every pair of a sequence, so the
    whole sequence is compared), with lengths, capacities and offsets;
  * on the 16K Mistral-shaped workload, end to end: the oracle's own float64
    scoring of all 256 (layer, KV head) pairs (a spawn process pool), then its
    selection; the device's taken set must equal it up to near-ties (keys
    within 1e-6 relative, resolved in the device's order), which are counted;
  * the packed entries of the sampled pairs (oracle pack of the device's
    taken set) and every decode output of theirs over all decode steps.
The long-context case takes its slots from the device's curvature partition
(checked against the oracle first).  The serving batch (90 GB of K and V) has
its own test with inputs generated on the device
(tests/test_gpu_full_size_serving.py).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import (assert_bf16_close, assert_f32_close, dev, params_for,
                               token_view, upload_workload)
from tests.partition_lambda import partition_lambda

pytestmark = [pytest.mark.gpu, pytest.mark.gpu_full]

# the kernels whose results the end-to-end selection report depends on
PARITY_SOURCES = ("kv_cache_compression_probe_gb300/csrc/kvc_score.cu",
                  "kv_cache_compression_probe_gb300/csrc/kvc_score_tc.cu",
                  "kv_cache_compression_probe_gb300/csrc/kvc_select.cu",
                  "kv_cache_compression_probe_gb300/csrc/kvc_common.cuh")

CASES = {
    "mistral16k": dict(cfg=lambda: W.get_config("mistral16k"), heads=[(0, 0, 0), (0, 17, 5)],
                       end_to_end=True),
    "aggressive": dict(cfg=lambda: W.get_config("aggressive"), heads=[(0, 3, 2)]),
    "long": dict(cfg=lambda: W.get_config("long"), heads=[(1, 9, 4)], partition=True),
}


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


def _procs():
    return max(1, min(16, os.cpu_count() or 4))


def _partition_on_device(kvc, cfg, wl):
    """a0 on the device from the synthetic hidden states; checks kappa and the cuts
    against the oracle and installs the device's slots in the workload."""
    ns = np.asarray([s.n for s in wl.seqs])
    n_max = int(ns.max())
    dh = cfg.hidden_dim
    hid = np.zeros((cfg.B, n_max, dh), np.float32)
    for b, s in enumerate(wl.seqs):
        hid[b, :s.n] = W.hidden_states(cfg, b, s.n, s.planted)
    S_max = max(int(n - cfg.W) // 16 + 1 for n in ns)
    p = params_for(cfg, n_max=n_max, S_max=S_max)
    ws = kvc.workspace(kvc.KVC_WS_PARTITION, p)
    kappa = torch.zeros((cfg.B, n_max), device="cuda")
    bounds = torch.zeros((cfg.B, S_max + 1), dtype=torch.int32, device="cuda")
    nsl = torch.zeros((cfg.B,), dtype=torch.int32, device="cuda")
    kvc.kvc_partition(p, dev(ns.astype(np.int32)), dev(hid, torch.bfloat16), dh, kappa, bounds,
                      nsl, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    kg = kappa.cpu().numpy().astype(np.float64)
    bg, ng = bounds.cpu().numpy(), nsl.cpu().numpy()
    for b, s in enumerate(wl.seqs):
        end = s.n - cfg.W
        hb = W.round_bf16(hid[b, :s.n]).astype(np.float64)
        assert np.abs(kg[b, :s.n] - O.curvature(hb)).max() < 2e-5
        cuts = O.partition_dp(kg[b], end, lam=partition_lambda(kg[b], end))
        np.testing.assert_array_equal(bg[b, :int(ng[b]) + 1], cuts)
        s.slot_bounds = cuts.astype(np.int32)


def _check_head_scores(cfg, wl, b, l, h, lse, feats, rel, util, cost):
    s = wl.seqs[b]
    res = O.score_and_value_head(s.K[l, h], s.V[l, h], s.Qp[l, h * cfg.G:(h + 1) * cfg.G], s.n,
                                 cfg.P, s.slot_bounds, float(wl.head_sens[l, h]),
                                 base=cfg.rope_base, hop_weight=cfg.hop_weight, n_hops=cfg.n_hops,
                                 w_part=cfg.w_part, w_value=cfg.w_value,
                                 value_floor=cfg.value_floor)
    tag = f"(b={b}, l={l}, h={h})"
    assert_f32_close(lse[b, l, h], res.lse, f"lse {tag}", rel=1e-5)
    f = token_view(feats, wl, b, 5)[l, h]
    for k, name in enumerate(["alpha", "|v|", "sigma", "H", "pos"]):
        assert_f32_close(f[:, k], res.feats[:, k], f"{name} {tag}", rel=1e-5, axis=-1)
    assert_f32_close(token_view(rel, wl, b)[l, h], res.r, f"relevance {tag}", rel=1e-5, axis=-1)
    S = len(s.slot_bounds) - 1
    np.testing.assert_array_equal(cost[b, l, h, :S], res.cost)
    sens = float(wl.head_sens[l, h])
    for k in range(S):
        nodes = O.tree_nodes(int(s.slot_bounds[k]), int(s.slot_bounds[k + 1]))
        Rv = np.array([res.r[x:y].sum() for x, y in nodes])
        scale = np.r_[Rv[0], Rv] * sens / res.cost[k]
        o = res.util[k]
        err = np.abs(util[b, l, h, k].astype(np.float64) - o)
        assert (err <= 1e-5 * np.maximum(np.abs(o), 3 * scale)).all(), (tag, k, err.max())


def _end_to_end_selection(name, cfg, wl, util, cost, rel, taken):
    """The device's taken set against the oracle chain's own (float64 scoring of
    every (l,h), then its floor and auction), up to near-ties of 1e-6 relative.
    With KVC_PARITY_REPORT set, the counts are written there as JSON."""
    from tests.oracle_pipeline import score_sequence_parallel
    from tests.tie_check import TIE_REL, band_needed, check_sequence, utility_slack
    report = {"workload": name, "tie_band_rel": TIE_REL, "sequences": []}
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        u64, c64, r64 = score_sequence_parallel(wl, b, _procs())
        np.testing.assert_array_equal(cost[b, :, :, :S], c64)
        n_ops, n_rel, n_scale, worst = utility_slack(u64, util[b, :, :, :S], c64, r64,
                                                     wl.head_sens, s.slot_bounds)
        # fp32 reaches most utilities to 1e-5 relative; the rest are near zero
        # after the clamped difference cancels and pass through the scale term
        assert n_scale <= 0.05 * n_ops, (n_scale, n_ops)
        args = (u64, util[b, :, :, :S], c64, r64, token_view(rel, wl, b), wl.head_sens,
                taken[b, :, :, :S], s.slot_bounds, s.n, cfg)
        try:
            rep = check_sequence(*args)
        except AssertionError as e:
            raise AssertionError(f"{name}, sequence {b}: {e}; band needed: {band_needed(*args)}") from None
        report["sequences"].append(dict(b=b, ops=int(c64.size), ties_reported=rep.diff_ops,
                                        tie_runs_reordered=rep.runs_moved_util,
                                        floor_tie_runs_reordered=rep.runs_moved_floor,
                                        util_max_abs_err=rep.max_abs_err,
                                        util_max_rel_err=rep.max_rel_err,
                                        util_within_1e5_rel=n_rel,
                                        util_within_scale_term_only=n_scale,
                                        util_worst_err_over_bound=worst))
    print(f"{name} end-to-end selection: {report}")
    path = os.environ.get("KVC_PARITY_REPORT")
    if path:
        import hashlib
        h = hashlib.sha256()
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        for f in PARITY_SOURCES:
            h.update(open(os.path.join(root, f), "rb").read())
        report["source_sha256"] = h.hexdigest()
        report["source_files"] = list(PARITY_SOURCES)
        report["command"] = ("KVC_PARITY_REPORT=<path> python -m pytest "
                             "tests/test_gpu_full_size.py -k mistral16k -m gpu -q")
        with open(path, "w") as f:
            json.dump(report, f, indent=1)


@pytest.mark.parametrize("name", list(CASES))
def test_full_size_against_sampled_oracle(kvc, name):
    spec = CASES[name]
    cfg = spec["cfg"]()
    D = cfg.n_decode
    wl = W.make_workload_parallel(cfg, _procs())
    if spec.get("partition"):
        _partition_on_device(kvc, cfg, wl)
    p, comp, d, S_max = upload_workload(wl, tensor_cores=True)
    comp.compress(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0

    lse, feats, rel = comp.lse.cpu().numpy(), comp.feats.cpu().numpy(), comp.relevance.cpu().numpy()
    util, cost = comp.op_util.cpu().numpy(), comp.op_cost.cpu().numpy().astype(np.int64)
    taken = comp.taken.cpu().numpy().astype(bool)
    lens, caps, offs = comp.len_lh.cpu().numpy(), comp.cap_lh.cpu().numpy(), comp.off_lh.cpu().numpy()

    # a1-a4 on the sampled pairs
    for (b, l, h) in spec["heads"]:
        _check_head_scores(cfg, wl, b, l, h, lse, feats, rel, util, cost)

    # a5: every sequence, bit-exact on the device's fp32 keys
    want_lens = np.zeros_like(lens, dtype=np.int64)
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        sel = O.select_sequence(util[b, :, :, :S], cost[b, :, :, :S], token_view(rel, wl, b),
                                wl.head_sens, s.slot_bounds, s.n, cfg.W, cfg.budget_ratio,
                                cfg.budget_entries_per_lh, cfg.floor_cap_frac, cfg.floor_cap_tokens)
        np.testing.assert_array_equal(taken[b, :, :, :S], sel.taken, err_msg=f"taken, sequence {b}")
        assert not taken[b, :, :, S:].any()
        assert int(sel.lens.sum()) - cfg.W * cfg.L * cfg.H <= sel.B_alloc
        want_lens[b] = sel.lens
    np.testing.assert_array_equal(lens, want_lens)
    if spec.get("end_to_end"):
        _end_to_end_selection(name, cfg, wl, util, cost, rel, taken)
    wc, wo = O.offsets(want_lens, cfg.decode_reserve)
    np.testing.assert_array_equal(caps, wc)
    np.testing.assert_array_equal(offs, wo)

    # a3 + a6 on the sampled pairs; their packed entries seed the decode oracle
    Kp, Vp = comp.Kp.float().cpu().numpy(), comp.Vp.float().cpu().numpy()
    lm, ps = comp.logm.cpu().numpy(), comp.pos.cpu().numpy()
    caches = {}
    for (b, l, h) in spec["heads"]:
        s = wl.seqs[b]
        S = len(s.slot_bounds) - 1
        r = token_view(rel, wl, b)[l, h].astype(np.float64)
        K_, V_, m_, p_ = O.pack_head(s.K[l, h], s.V[l, h], r, s.slot_bounds, taken[b, l, h, :S],
                                     s.n, cfg.W, cfg.rope_base, cfg.value_floor)
        o, n_ = int(offs[b, l, h]), int(lens[b, l, h])
        assert n_ == len(K_)
        np.testing.assert_array_equal(ps[o:o + n_], p_.astype(np.float32))
        exact = m_ == 0
        np.testing.assert_array_equal(Kp[o:o + n_][exact], K_[exact].astype(np.float32))
        assert_bf16_close(Kp[o:o + n_], K_, f"packed K {(b, l, h)}")
        assert_bf16_close(Vp[o:o + n_], V_, f"packed V {(b, l, h)}")
        np.testing.assert_allclose(lm[o:o + n_], m_, rtol=1e-5, atol=1e-6)
        caches[(b, l, h)] = (Kp[o:o + n_].astype(np.float64), Vp[o:o + n_].astype(np.float64),
                             lm[o:o + n_].astype(np.float64))
    del Kp, Vp

    # a7: D decode steps as one graph replay; every output of the sampled pairs
    dec = [W.decode_inputs(cfg, t) for t in range(D)]
    bf = torch.bfloat16
    q_all = dev(np.stack([x[0] for x in dec]), bf)
    kn_all = dev(np.stack([x[1] for x in dec]), bf)
    vn_all = dev(np.stack([x[2] for x in dec]), bf)
    out = torch.empty(tuple(q_all.shape), dtype=bf, device="cuda")
    comp.decode_many(q_all, kn_all, vn_all, out)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    got = out.float().cpu().numpy()
    for (b, l, h), cache in caches.items():
        for t in range(D):
            q, kn, vn = dec[t][0][b, l, h * cfg.G:(h + 1) * cfg.G], dec[t][1][b, l, h], dec[t][2][b, l, h]
            want, *cache = O.decode_step_head(q, kn, vn, *cache)
            assert_bf16_close(got[t, b, l, h * cfg.G:(h + 1) * cfg.G], want, f"decode {(b, l, h)} step {t}")
    np.testing.assert_array_equal(comp.len_lh.cpu().numpy(), lens + D)
