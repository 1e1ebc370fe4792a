"""Full-size parity of the serving batch: 64 sequences with contexts drawn from
4096..16384, all 32 layers x 8 KV heads, 25% budget per sequence, then 512
batched decode steps replayed as one CUDA graph.

Its 90 GB of bf16 K and V are generated on the device (synth.device_gen: the
same recipe as the host generator, drawn from torch's generator), so the
inputs never exist as host arrays.  Checked against the float64 oracle:
  * the selection of every one of the 64 sequences (the budget of a sequence
    is pooled over its 256 (layer, KV head) pairs), bit-exact against the
    oracle's floor and auction run on the device's fp32 keys, with lengths,
    capacities and offsets (a spawn process pool, one sequence per task);
  * on sampled (sequence, layer, KV head) triples, whose inputs are copied back
    from the device: probe LSE, features, relevance, op costs and utilities,
    the packed entries and every decode output over the 512 steps.
"""
import os

import numpy as np
import pytest
import torch

import oracle as O
from synth import device_gen as DG
from synth import workloads as W
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, dev, params_for

pytestmark = [pytest.mark.gpu, pytest.mark.gpu_full]

HEADS = [(0, 0, 0), (37, 1, 6), (63, 31, 7)]


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


def _select_job(job):
    b, util, cost, r, sens, bounds, n, cfg = job
    sel = O.select_sequence(util.astype(np.float64), cost, r.astype(np.float32), sens, bounds, n,
                            cfg.W, cfg.budget_ratio, cfg.budget_entries_per_lh,
                            cfg.floor_cap_frac, cfg.floor_cap_tokens)
    return b, sel.taken, sel.lens, sel.B_alloc


def test_serving_batch_full_size(kvc):
    import multiprocessing as mp
    from kv_cache_compression_probe_gb300.pipeline import Compressor, pad_bounds
    cfg = W.get_config("serving")
    L, H, G, P, d, D = cfg.L, cfg.H, cfg.G, cfg.P, cfg.d, cfg.n_decode
    ns = W.context_lengths(cfg)
    rows = int(ns.sum()) * L * H
    bf = torch.bfloat16
    K = torch.empty((rows, d), dtype=bf, device="cuda")
    V = torch.empty_like(K)
    Qp = torch.empty((cfg.B, L, H * G, P, d), dtype=bf, device="cuda")
    ns, bounds = DG.fill_workload(cfg, K, V, Qp)
    S_max = max(len(bd) - 1 for bd in bounds)
    p = params_for(cfg, n_max=int(ns.max()), S_max=S_max)
    comp = Compressor(p, [int(n) for n in ns], tensor_cores=True)
    dbounds = dev(pad_bounds(bounds, S_max))
    nsl = dev(np.asarray([len(bd) - 1 for bd in bounds], np.int32))
    sens_h = np.ones((L, H), np.float32)
    comp.compress(K, V, Qp, dbounds, nsl, dev(sens_h))
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0

    util, cost = comp.op_util.cpu().numpy(), comp.op_cost.cpu().numpy().astype(np.int64)
    taken = comp.taken.cpu().numpy().astype(bool)
    lens, caps, offs = comp.len_lh.cpu().numpy(), comp.cap_lh.cpu().numpy(), comp.off_lh.cpu().numpy()
    starts = np.concatenate([[0], np.cumsum(ns * L * H)])

    # a5: every sequence, bit-exact on the device's fp32 keys
    jobs = []
    for b in range(cfg.B):
        S = len(bounds[b]) - 1
        n = int(ns[b])
        r = comp.relevance[starts[b]:starts[b + 1]].cpu().numpy().reshape(L, H, n)
        jobs.append((b, util[b, :, :, :S], cost[b, :, :, :S], r, sens_h, bounds[b], n, cfg))
    want_lens = np.zeros_like(lens, dtype=np.int64)
    with mp.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 4))) as pool:
        for b, t_b, l_b, b_alloc in pool.imap_unordered(_select_job, jobs):
            S = len(bounds[b]) - 1
            np.testing.assert_array_equal(taken[b, :, :, :S], t_b, err_msg=f"taken, sequence {b}")
            assert not taken[b, :, :, S:].any()
            assert int(l_b.sum()) - cfg.W * L * H <= b_alloc
            want_lens[b] = l_b
    del jobs
    np.testing.assert_array_equal(lens, want_lens)
    wc, wo = O.offsets(want_lens, cfg.decode_reserve)
    np.testing.assert_array_equal(caps, wc)
    np.testing.assert_array_equal(offs, wo)

    # a1-a4, a3 + a6 on the sampled triples (inputs copied back from the device)
    lm_all, ps_all = comp.logm.cpu().numpy(), comp.pos.cpu().numpy()
    caches = {}
    for (b, l, h) in HEADS:
        n = int(ns[b])
        S = len(bounds[b]) - 1
        r0 = int(starts[b]) + (l * H + h) * n
        Kh = K[r0:r0 + n].float().cpu().numpy()
        Vh = V[r0:r0 + n].float().cpu().numpy()
        Qh = Qp[b, l, h * G:(h + 1) * G].float().cpu().numpy()
        res = O.score_and_value_head(Kh, Vh, Qh, n, P, bounds[b], 1.0, base=cfg.rope_base,
                                     hop_weight=cfg.hop_weight, n_hops=cfg.n_hops,
                                     w_part=cfg.w_part, w_value=cfg.w_value,
                                     value_floor=cfg.value_floor)
        tag = f"(b={b}, l={l}, h={h})"
        assert_f32_close(comp.lse[b, l, h].cpu().numpy(), res.lse, f"lse {tag}", rel=1e-5)
        f = comp.feats[r0:r0 + n].cpu().numpy()
        for k, name in enumerate(["alpha", "|v|", "sigma", "H", "pos"]):
            assert_f32_close(f[:, k], res.feats[:, k], f"{name} {tag}", rel=1e-5, axis=-1)
        rel_h = comp.relevance[r0:r0 + n].cpu().numpy()
        assert_f32_close(rel_h, res.r, f"relevance {tag}", rel=1e-5, axis=-1)
        np.testing.assert_array_equal(cost[b, l, h, :S], res.cost)
        for k in range(S):
            nodes = O.tree_nodes(int(bounds[b][k]), int(bounds[b][k + 1]))
            Rv = np.array([res.r[x:y].sum() for x, y in nodes])
            scale = np.r_[Rv[0], Rv] / res.cost[k]
            o = res.util[k]
            err = np.abs(util[b, l, h, k].astype(np.float64) - o)
            assert (err <= 1e-5 * np.maximum(np.abs(o), 3 * scale)).all(), (tag, k, err.max())
        K_, V_, m_, p_ = O.pack_head(Kh, Vh, rel_h.astype(np.float64), bounds[b],
                                     taken[b, l, h, :S], n, cfg.W, cfg.rope_base, cfg.value_floor)
        o, n_ = int(offs[b, l, h]), int(lens[b, l, h])
        assert n_ == len(K_)
        Kp = comp.Kp[o:o + n_].float().cpu().numpy()
        Vp = comp.Vp[o:o + n_].float().cpu().numpy()
        np.testing.assert_array_equal(ps_all[o:o + n_], p_.astype(np.float32))
        exact = m_ == 0
        np.testing.assert_array_equal(Kp[exact], K_[exact].astype(np.float32))
        assert_bf16_close(Kp, K_, f"packed K {tag}")
        assert_bf16_close(Vp, V_, f"packed V {tag}")
        np.testing.assert_allclose(lm_all[o:o + n_], m_, rtol=1e-5, atol=1e-6)
        caches[(b, l, h)] = (Kp.astype(np.float64), Vp.astype(np.float64),
                             lm_all[o:o + n_].astype(np.float64))

    # a7: D batched decode steps as one graph replay; every output of the sampled triples
    q_all, kn_all, vn_all = DG.decode_inputs(cfg, D, "cuda")
    out = torch.empty(tuple(q_all.shape), dtype=bf, device="cuda")
    comp.decode_many(q_all, kn_all, vn_all, out)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    for (b, l, h), cache in caches.items():
        q = q_all[:, b, l, h * G:(h + 1) * G].float().cpu().numpy()
        kn = kn_all[:, b, l, h].float().cpu().numpy()
        vn = vn_all[:, b, l, h].float().cpu().numpy()
        got = out[:, b, l, h * G:(h + 1) * G].float().cpu().numpy()
        for t in range(D):
            want, *cache = O.decode_step_head(q[t], kn[t], vn[t], *cache)
            assert_bf16_close(got[t], want, f"decode {(b, l, h)} step {t}")
    np.testing.assert_array_equal(comp.len_lh.cpu().numpy(), lens + D)
