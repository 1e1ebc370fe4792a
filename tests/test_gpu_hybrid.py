"""GPU parity of the head-level hybrid selection (reading R16: the top fraction of
heads by relevance mass outside the window keep every token) against the
oracle, and the pack of those heads against their input."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import token_view, upload_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from kv_cache_compression_probe_gb300 import build
    build.build()


@pytest.mark.parametrize("frac", [0.2, 0.34])
def test_hybrid_selection_matches_oracle_and_full_heads_pack_their_input(built, frac):
    from kv_cache_compression_probe_gb300 import kvc
    cfg = W.small_config(L=2, H=3, budget_ratio=0.5)
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl, tensor_cores=True, head_full_frac=frac)
    comp.compress(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    util = comp.op_util.cpu().numpy()
    cost = comp.op_cost.cpu().numpy().astype(np.int64)
    rel = comp.relevance.cpu().numpy()
    taken = comp.taken.cpu().numpy().astype(bool)
    lens, offs = comp.len_lh.cpu().numpy(), comp.off_lh.cpu().numpy()
    Kp, Vp, lm = comp.Kp.float().cpu().numpy(), comp.Vp.float().cpu().numpy(), comp.logm.cpu().numpy()
    F = int(np.floor(frac * cfg.L * cfg.H))
    for b, s in enumerate(wl.seqs):
        S = len(s.slot_bounds) - 1
        r = token_view(rel, wl, b)
        sel = O.select_sequence(util[b, :, :, :S], cost[b, :, :, :S], r, wl.head_sens,
                                s.slot_bounds, s.n, cfg.W, cfg.budget_ratio,
                                cfg.budget_entries_per_lh, cfg.floor_cap_frac,
                                cfg.floor_cap_tokens, head_full_frac=frac)
        np.testing.assert_array_equal(taken[b, :, :, :S], sel.taken)
        np.testing.assert_array_equal(lens[b], sel.lens)
        full = O.full_heads(r, int(s.slot_bounds[-1]), frac)
        assert full.sum() == F
        for l in range(cfg.L):
            for h in range(cfg.H):
                if not full[l, h]:
                    continue
                o = int(offs[b, l, h])
                assert lens[b, l, h] == s.n
                np.testing.assert_array_equal(Kp[o:o + s.n], s.K[l, h])
                np.testing.assert_array_equal(Vp[o:o + s.n], s.V[l, h])
                assert (lm[o:o + s.n] == 0).all()
        B_tot = O.budget(s.n, cfg.L, cfg.H, cfg.W, cfg.budget_ratio, 0, cfg.floor_cap_frac)[0]
        assert int(lens[b].sum()) <= B_tot


def test_hybrid_reports_a_budget_too_small_for_the_full_heads(built):
    from kv_cache_compression_probe_gb300 import kvc
    cfg = W.small_config(L=2, H=3, budget_ratio=0.5)
    wl = W.make_workload(cfg)
    # half the heads full at a 50% budget leaves less than the other windows
    p, comp, d, S_max = upload_workload(wl, tensor_cores=True, head_full_frac=0.5)
    comp.compress(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == kvc.KVC_EBUDGET
