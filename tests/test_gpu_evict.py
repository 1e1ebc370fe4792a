"""GPU parity of NEXT f2, per-step top-B eviction with the heuristic score
(DistillCache Algorithm 1 and 3.1.1, reading R17), against the oracle's
evict_step over several steps:
  * each step's attention output over the appended cache;
  * alpha (mean attention probability per entry) within the tolerance the
    arithmetic allows (tensor-core path: row sums of bf16-rounded numerators);
  * the kept set bit-exact against the oracle's top-B run on the device's alpha
    (ties to the earlier token), with the K, V rows and positions it kept, and
    against the oracle's own top-B wherever alpha is not within tolerance of
    the cut.  Eviction is in place and leaves the rows in no position order,
    so rows are matched by position (the oracle keeps its cache in position
    order, where the lower index is the earlier token);
  * a CUDA-graph replay of the same steps equal to the eager run.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


def _setup(kvc, cfg, T, ratio, b_min, tc, scores=True):
    from kv_cache_compression_probe_gb300.pipeline import EvictingCache
    wl = W.make_workload(cfg)
    ns = [s.n for s in wl.seqs]
    n_max = max(ns)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    K = np.zeros((cfg.B, cfg.L, cfg.H, n_max, cfg.d), np.float32)
    V = np.zeros_like(K)
    for b, s in enumerate(wl.seqs):
        K[b, :, :, :s.n] = s.K
        V[b, :, :, :s.n] = s.V
    p = kvc.make_params(B=cfg.B, L=cfg.L, H=cfg.H, G=cfg.G, d=cfg.d, P=cfg.P, W=cfg.W,
                        dtype=kvc.KVC_BF16 if cfg.dtype == "bf16" else kvc.KVC_F32,
                        n_max=n_max, S_max=1)
    cache = EvictingCache(p, dev(K, dt), dev(V, dt), ns, T, ratio, b_min, tensor_cores=tc,
                          scores=scores)
    steps = [W.decode_inputs(cfg, t) for t in range(T)]
    return wl, ns, cache, steps, dt


def _step_tensors(steps, ns, dt):
    q = dev(np.stack([x[0] for x in steps]), dt)
    kn = dev(np.stack([x[1] for x in steps]), dt)
    vn = dev(np.stack([x[2] for x in steps]), dt)
    T = len(steps)
    nseen = dev(np.asarray([[n + t + 1 for n in ns] for t in range(T)], np.int64))
    posn = dev(np.asarray([[n + t for n in ns] for t in range(T)], np.float32))
    return q, kn, vn, nseen, posn


CASES = [
    # (dtype, tensor-core decode, alpha from the decode's scores, ratio, b_min)
    ("bf16", True, True, 0.25, 32),
    ("bf16", True, False, 0.25, 32),     # alpha recomputed from K
    ("bf16", False, True, 0.25, 32),
    ("f32", False, True, 0.25, 32),
    ("f32", False, False, 0.25, 32),
    ("bf16", True, True, 0.5, 10000),    # the minimum budget covers the cache: nothing evicted
    ("bf16", True, True, 0.0, 1),        # one entry survives each step
]


@pytest.mark.parametrize("dtype,tc,scores,ratio,b_min", CASES)
def test_eviction_steps_match_oracle(kvc, dtype, tc, scores, ratio, b_min):
    cfg = W.small_config(B=2, L=2, H=2, n=700, n_min=450, dtype=dtype, P=32, W=32)
    T = 4
    wl, ns, cache, steps, dt = _setup(kvc, cfg, T, ratio, b_min, tc, scores)
    q, kn, vn, nseen, posn = _step_tensors(steps, ns, dt)
    out = torch.empty(tuple(q.shape), dtype=dt, device="cuda")
    # oracle state: the tokens each sequence still holds, with their positions
    Ko = [s.K.astype(np.float64) for s in wl.seqs]
    Vo = [s.V.astype(np.float64) for s in wl.seqs]
    Po = [np.arange(s.n, dtype=np.float64) for s in wl.seqs]
    arel = 4e-3 if tc else 1e-4
    LH0 = [(l, h) for l in range(cfg.L) for h in range(cfg.H)]
    for t in range(T):
        rows_pos = [cache.entries(b, 0, 0)[2].astype(np.float64) for b in range(cfg.B)]
        cache.step(q[t], kn[t], vn[t], out[t], nseen[t], posn[t])
        torch.cuda.synchronize()
        assert kvc.kvc_device_error() == 0
        got = out[t].float().cpu().numpy()
        ag = cache.alpha.cpu().numpy().astype(np.float64)
        for b in range(cfg.B):
            qb, knb, vnb = steps[t][0][b], steps[t][1][b], steps[t][2][b]
            n_seen = ns[b] + t + 1
            c = Ko[b].shape[2]
            o_out, o_alpha, o_keep = O.evict_step(qb, knb, vnb, Ko[b], Vo[b], n_seen, ratio, b_min)
            if dtype == "bf16":
                assert_bf16_close(got[b], o_out, f"out b={b} t={t}")
            else:
                assert_f32_close(got[b], o_out, f"out b={b} t={t}", rel=1e-4)
            # device rows -> position order (the new token was appended as row c)
            rp = np.r_[rows_pos[b], float(n_seen - 1)]
            order = np.argsort(rp, kind="stable")
            Px = np.r_[Po[b], float(n_seen - 1)]
            np.testing.assert_array_equal(rp[order], Px)
            a = ag[b, :c + 1][order]
            err = np.abs(a - o_alpha)
            assert (err <= arel * o_alpha + 1e-7).all(), (b, t, (err / (o_alpha + 1e-7)).max())
            Bb = min(c + 1, O.evict_budget(n_seen, ratio, b_min))
            keep = O.top_b(a, Bb)                               # on the device's alpha
            # the oracle's own choice differs only at entries within tolerance of the cut
            diff = np.setxor1d(keep, o_keep)
            if len(diff) and Bb < c + 1:
                cut = np.sort(o_alpha)[::-1][Bb - 1] if Bb > 0 else np.inf
                assert (np.abs(o_alpha[diff] - cut) <= 2 * (arel * cut + 1e-7)).all(), (b, t, diff)
            Kx = np.concatenate([Ko[b], knb[:, :, None].astype(np.float64)], axis=2)
            Vx = np.concatenate([Vo[b], vnb[:, :, None].astype(np.float64)], axis=2)
            if scores:                  # the decode's exported base-2 scores of every row
                for (l, h) in (LH0[0], LH0[-1]):
                    o = ((b * cfg.L + l) * cfg.H + h) * cache.cap
                    sg = cache.scores[o:o + c + 1].cpu().numpy()[order]
                    so = (Kx[l, h] @ qb[l, h * cfg.G:(h + 1) * cfg.G].astype(np.float64).T
                          / np.sqrt(cfg.d) / np.log(2.0))
                    assert_f32_close(sg, so, f"scores b={b} l={l} h={h} t={t}", rel=1e-4,
                                     floor_frac=1e-2)
            first = None
            for (l, h) in LH0:
                Kg, Vg, pg = cache.entries(b, l, h)
                assert len(pg) == len(keep), (b, l, h, t)
                if first is None:
                    first = pg
                np.testing.assert_array_equal(pg, first)       # one row order for every (l,h)
                srt = np.argsort(pg, kind="stable")
                np.testing.assert_array_equal(pg[srt], Px[keep].astype(np.float32))
                np.testing.assert_array_equal(Kg[srt], Kx[l, h, keep].astype(np.float32))
                np.testing.assert_array_equal(Vg[srt], Vx[l, h, keep].astype(np.float32))
            Ko[b], Vo[b], Po[b] = Kx[:, :, keep], Vx[:, :, keep], Px[keep]
    assert (cache.logm == 0).all()


def test_graph_replay_equals_eager(kvc):
    cfg = W.small_config(B=2, L=2, H=2, n=700, n_min=450, P=32, W=32)
    T = 6
    res = []
    for graph in (False, True):
        wl, ns, cache, steps, dt = _setup(kvc, cfg, T, 0.25, 32, True)
        q, kn, vn, nseen, posn = _step_tensors(steps, ns, dt)
        out = torch.empty(tuple(q.shape), dtype=dt, device="cuda")
        launches = cache.run_many(q, kn, vn, out, nseen, posn, graph=graph)
        torch.cuda.synchronize()
        assert kvc.kvc_device_error() == 0
        # decode (attention with its own work list, merge), alpha (groups, sum),
        # eviction (plan, moves)
        assert launches == T * 6
        rows = [int(x) for x in cache.len_lh.cpu()]
        res.append((out.float().cpu(), cache.K.float().cpu(), cache.pos.cpu(), rows))
    (o1, k1, p1, r1), (o2, k2, p2, r2) = res
    assert r1 == r2
    assert torch.equal(o1, o2) and torch.equal(p1, p2) and torch.equal(k1, k2)


def test_inconsistent_lengths_are_reported(kvc):
    cfg = W.small_config(B=1, L=2, H=2, n=300, n_min=300, P=32, W=32)
    wl, ns, cache, steps, dt = _setup(kvc, cfg, 2, 0.25, 32, False)
    cache.len_lh[1] -= 1                     # one (l,h) of the sequence out of step
    q, kn, vn, nseen, posn = _step_tensors(steps, ns, dt)
    out = torch.empty(tuple(q.shape), dtype=dt, device="cuda")
    cache.step(q[0], kn[0], vn[0], out[0], nseen[0], posn[0])
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == kvc.KVC_EDEVICE


def test_bad_arguments_are_rejected(kvc):
    cfg = W.small_config(B=1, L=1, H=2, n=300, n_min=300, P=32, W=32)
    wl, ns, c, steps, dt = _setup(kvc, cfg, 1, 0.25, 32, True)
    n = torch.ones(1, dtype=torch.int64, device="cuda")
    for ratio, b_min, ws in ((-0.5, 4, c.ws_evict), (0.25, -1, c.ws_evict),
                             (0.25, 4, c.ws_evict[:8])):
        with pytest.raises(kvc.KvcError):
            kvc.kvc_evict_topb(c.p, c.alpha, n, ratio, b_min, c.K, c.V, c.pos, c.logm, c.off_lh,
                               c.len_lh, ws)
    qz = torch.zeros(1, 1, 8, 128, dtype=dt, device="cuda")
    with pytest.raises(kvc.KvcError):            # alpha's workspace too small
        kvc.kvc_token_alpha(c.p, qz, c.K, c.scores, c.len_lh, c.off_lh, c.lse, c.alpha,
                            c.ws_evict[:8])
    with pytest.raises(kvc.KvcError):            # neither scores nor (q, K)
        kvc.kvc_token_alpha(c.p, None, None, None, c.len_lh, c.off_lh, c.lse, c.alpha,
                            c.ws_evict)
