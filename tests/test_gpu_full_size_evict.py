"""Full-size parity of NEXT f2 (per-step top-B eviction with the attention score,
DistillCache Algorithm 1 and 3.1.1, reading R17) on the Mistral-7B-shaped 16K
workload: 32 layers x 8 KV heads, bf16, r = 0.25, B_min = 32, in the eviction
leg's launch configuration (tensor-core decode exporting LSE and scores, each
step a CUDA-graph replay).  Per step, against the oracle's evict_step run on
the device's cache contents just before the step (a device snapshot), one
(layer, KV head) at a time (alpha is the mean of the per-head means, every
head having G query heads):
  * alpha over every cache row;
  * the kept set bit-exact on the device's alpha (ties to the earlier token),
    with the kept K, V and positions of sampled (layer, KV head) pairs;
  * the attention outputs of the sampled pairs.
The first step evicts the 16K prompt to 4096 rows, the later ones one row.
"""
import os

import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import assert_bf16_close, dev

pytestmark = [pytest.mark.gpu, pytest.mark.gpu_full]

SAMPLED = [(0, 0), (17, 5), (31, 7)]


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


def test_eviction_full_size_against_oracle(kvc):
    from kv_cache_compression_probe_gb300.pipeline import EvictingCache
    cfg = W.get_config("mistral16k")
    T, ratio, b_min = 3, 0.25, 32
    L, H, G, d, n = cfg.L, cfg.H, cfg.G, cfg.d, cfg.n
    wl = W.make_workload_parallel(cfg, max(1, min(16, os.cpu_count() or 4)))
    s = wl.seqs[0]
    p = kvc.make_params(B=1, L=L, H=H, G=G, d=d, P=cfg.P, W=cfg.W, dtype=kvc.KVC_BF16, n_max=n,
                        S_max=1)
    cache = EvictingCache(p, dev(s.K[None], torch.bfloat16), dev(s.V[None], torch.bfloat16), [n],
                          T + 1, ratio, b_min)
    del wl, s
    dec = [W.decode_inputs(cfg, t) for t in range(T)]
    bf = torch.bfloat16
    q = dev(np.stack([x[0] for x in dec]), bf)
    kn = dev(np.stack([x[1] for x in dec]), bf)
    vn = dev(np.stack([x[2] for x in dec]), bf)
    nseen = dev(np.asarray([[n + t + 1] for t in range(T)], np.int64))
    posn = dev(np.asarray([[n + t] for t in range(T)], np.float32))
    out = torch.empty(tuple(q.shape), dtype=bf, device="cuda")
    cap = cache.cap
    f64 = lambda x: x.float().cpu().numpy().astype(np.float64)  # noqa: E731
    for t in range(T):
        c = int(cache.len_lh[0])
        K0, V0, P0 = cache.K.clone(), cache.V.clone(), cache.pos.clone()
        cache.run_many(q[t:t + 1], kn[t:t + 1], vn[t:t + 1], out[t:t + 1], nseen[t:t + 1],
                       posn[t:t + 1], graph=True)
        torch.cuda.synchronize()
        assert kvc.kvc_device_error() == 0
        n_seen = n + t + 1
        qh, knh, vnh = dec[t][0][0], dec[t][1][0], dec[t][2][0]
        got = out[t, 0].float().cpu().numpy()
        alpha_o = np.zeros(c + 1)
        for l in range(L):
            for h in range(H):
                o = (l * H + h) * cap
                Kc = f64(K0[o:o + c])[None, None]
                Vc = f64(V0[o:o + c])[None, None]
                qq = qh[l:l + 1, h * G:(h + 1) * G]
                oo, al, _ = O.evict_step(qq, knh[l:l + 1, h:h + 1], vnh[l:l + 1, h:h + 1], Kc, Vc,
                                         n_seen, ratio, b_min)
                alpha_o += al
                if (l, h) in SAMPLED:
                    assert_bf16_close(got[l, h * G:(h + 1) * G], oo[0], f"out (l={l}, h={h}) t={t}")
        alpha_o /= L * H                                  # mean of the per-head means
        ag = cache.alpha[0, :c + 1].cpu().numpy().astype(np.float64)
        err = np.abs(ag - alpha_o)
        assert (err <= 4e-3 * alpha_o + 1e-7).all(), (t, (err / (alpha_o + 1e-7)).max())
        assert abs(ag.sum() - 1.0) < 4e-3
        # the kept set on the device's alpha, ties to the earlier token
        rp = np.r_[P0[:c].cpu().numpy().astype(np.float64), float(n_seen - 1)]
        order = np.argsort(rp, kind="stable")
        Bb = min(c + 1, O.evict_budget(n_seen, ratio, b_min))
        keep_rows = order[O.top_b(ag[order], Bb)]          # device rows before the step
        lens = cache.len_lh.cpu().numpy()
        assert (lens == Bb).all()
        for (l, h) in SAMPLED:
            o = (l * H + h) * cap
            Kx = np.concatenate([f64(K0[o:o + c]), knh[l, h][None].astype(np.float64)])
            Vx = np.concatenate([f64(V0[o:o + c]), vnh[l, h][None].astype(np.float64)])
            pg = cache.pos[o:o + Bb].cpu().numpy()
            srt = np.argsort(pg, kind="stable")
            want = np.sort(rp[keep_rows])
            np.testing.assert_array_equal(pg[srt], want.astype(np.float32))
            kr = keep_rows[np.argsort(rp[keep_rows], kind="stable")]
            np.testing.assert_array_equal(f64(cache.K[o:o + Bb])[srt], Kx[kr])
            np.testing.assert_array_equal(f64(cache.V[o:o + Bb])[srt], Vx[kr])
        del K0, V0, P0
        torch.cuda.empty_cache()
