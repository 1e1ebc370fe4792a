"""GPU parity of kvc_decode_attn against the float64 oracle decode (reading R10:
append with multiplicity one, then attend including the new token)."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import DT, assert_bf16_close, assert_f32_close, dev, params_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


def _rand_cache(rng, B, L, H, d, lens, reserve, dtype, nan_reserve=False):
    lens = np.asarray(lens, dtype=np.int64).reshape(B, L, H)
    caps, offs = O.offsets(lens, reserve)
    rows = int(caps.sum())
    Kp = rng.standard_normal((rows, d)).astype(np.float32)
    Vp = rng.standard_normal((rows, d)).astype(np.float32)
    lm = np.where(rng.uniform(size=rows) < 0.7, 0.0, rng.uniform(0, 3, size=rows)).astype(np.float32)
    if dtype == "bf16":
        Kp, Vp = W.round_bf16(Kp), W.round_bf16(Vp)
    if nan_reserve:
        # rows past each (l,h)'s entries hold NaN: no kernel may let them reach an output
        for o, n, c in zip(offs.reshape(-1), lens.reshape(-1), caps.reshape(-1)):
            Kp[o + n:o + c] = np.nan
            Vp[o + n:o + c] = np.nan
            lm[o + n:o + c] = np.nan
    return lens, caps, offs, Kp, Vp, lm


def _run_decode(kvc, cfg, lens, caps, offs, Kp, Vp, lm, steps, seed, tc=False):
    """tc: give the call the packed extent, which selects the tensor-core
    decode for bf16 / d = 128 (without it the SIMT kernel runs)."""
    B, L, H, G, d = cfg.B, cfg.L, cfg.H, cfg.G, cfg.d
    p = params_for(cfg, n_max=max(int(lens.max()) + 64, cfg.W + 16), S_max=1,
                   packed_rows=Kp.shape[0] if tc else 0)
    dt = DT[cfg.dtype]
    dKp, dVp = dev(Kp, dt), dev(Vp, dt)
    dlm = dev(lm)
    dpos = torch.zeros(Kp.shape[0], dtype=torch.float32, device="cuda")
    dlen = dev(lens.astype(np.int32))
    dcap = dev(caps.astype(np.int32))
    doff = dev(offs.astype(np.int64))
    ws = kvc.workspace(kvc.KVC_WS_DECODE, p, zero=True)
    out = torch.empty((B, L, H * G, d), dtype=dt, device="cuda")
    cur = {}
    for b in range(B):
        for l in range(L):
            for h in range(H):
                o, c = int(offs[b, l, h]), int(lens[b, l, h])
                cur[(b, l, h)] = (Kp[o:o + c].astype(np.float64), Vp[o:o + c].astype(np.float64),
                                  lm[o:o + c].astype(np.float64))
    rng = np.random.default_rng(seed)
    outs = []
    for t in range(steps):
        q = rng.standard_normal((B, L, H * G, d)).astype(np.float32)
        kn = rng.standard_normal((B, L, H, d)).astype(np.float32)
        vn = rng.standard_normal((B, L, H, d)).astype(np.float32)
        if cfg.dtype == "bf16":
            q, kn, vn = W.round_bf16(q), W.round_bf16(kn), W.round_bf16(vn)
        posn = torch.full((B,), 1000.0 + t, device="cuda")
        kvc.kvc_decode_attn(p, dev(q, dt), dev(kn, dt), dev(vn, dt), posn, dKp, dVp, dlm, dpos, dlen,
                            dcap, doff, out, ws)
        err = kvc.kvc_device_error()
        got = out.float().cpu().numpy()
        want = np.zeros_like(got, dtype=np.float64)
        cap_hit = False
        for (b, l, h), (Kc, Vc, lc) in list(cur.items()):
            o4, K2, V2, l2 = O.decode_step_head(q[b, l, h * G:(h + 1) * G], kn[b, l, h], vn[b, l, h],
                                                Kc, Vc, lc)
            want[b, l, h * G:(h + 1) * G] = o4
            if Kc.shape[0] + 1 <= caps[b, l, h]:
                cur[(b, l, h)] = (K2, V2, l2)
            else:
                cap_hit = True
        outs.append((got, want, err, cap_hit))
    return outs, dlen, dKp, dlm, doff


@pytest.mark.parametrize("dtype,d,G,tc", [("bf16", 128, 4, False), ("f32", 64, 4, False),
                                          ("bf16", 128, 1, False), ("bf16", 64, 8, False),
                                          ("f32", 128, 2, False), ("bf16", 128, 4, True),
                                          ("bf16", 128, 1, True), ("bf16", 128, 2, True),
                                          ("bf16", 128, 8, True)])
def test_decode_matches_oracle_ragged(kvc, dtype, d, G, tc):
    cfg = W.small_config(B=2, L=2, H=3, G=G, d=d, dtype=dtype, P=16, W=16, n_decode=3)
    rng = np.random.default_rng(7)
    lens = [0, 1, 255, 256, 257, 600, 1023, 31, 512, 2, 800, 100]
    lens, caps, offs, Kp, Vp, lm = _rand_cache(rng, 2, 2, 3, d, lens, 3, dtype,
                                               nan_reserve=(dtype == "bf16"))
    outs, dlen, dKp, dlm, doff = _run_decode(kvc, cfg, lens, caps, offs, Kp, Vp, lm, 3, seed=1,
                                             tc=tc)
    for got, want, err, cap_hit in outs:
        assert err == 0 and not cap_hit
        if dtype == "bf16":
            assert_bf16_close(got, want, "decode out")
        else:
            # fp32: error relative to the scale of each output vector (a convex
            # combination of values), see the tolerance notes in the design doc
            assert_f32_close(got, want, "decode out", rel=1e-5, floor_frac=1.0, axis=-1)
    np.testing.assert_array_equal(dlen.cpu().numpy(), (lens + 3).astype(np.int32))
    lmv = dlm.cpu().numpy()
    for i in range(3):
        assert (lmv[offs.reshape(-1) + lens.reshape(-1) + i] == 0).all()


def test_tensor_core_decode_with_more_than_1024_heads(kvc):
    """Above 1024 (b,l,h) the work list comes from the plan kernel instead of
    each attention CTA's own scan: the same parity over 1056 ragged caches."""
    cfg = W.small_config(B=1, L=33, H=32, G=1, d=128, dtype="bf16", P=16, W=16, n_decode=2)
    rng = np.random.default_rng(11)
    lens = rng.integers(0, 700, size=33 * 32)
    lens, caps, offs, Kp, Vp, lm = _rand_cache(rng, 1, 33, 32, 128, lens, 2, "bf16")
    outs, dlen, dKp, dlm, doff = _run_decode(kvc, cfg, lens, caps, offs, Kp, Vp, lm, 2, seed=5,
                                             tc=True)
    for got, want, err, cap_hit in outs:
        assert err == 0 and not cap_hit
        assert_bf16_close(got, want, "decode out")
    np.testing.assert_array_equal(dlen.cpu().numpy(), (lens + 2).astype(np.int32))


@pytest.mark.parametrize("tc", [False, True])
def test_decode_capacity_overflow_reports_and_still_attends(kvc, tc):
    cfg = W.small_config(B=1, L=1, H=2, G=4, d=128, dtype="bf16", P=16, W=16, n_decode=0)
    rng = np.random.default_rng(3)
    lens, caps, offs, Kp, Vp, lm = _rand_cache(rng, 1, 1, 2, 128, [300, 40], 0, "bf16")
    outs, dlen, *_ = _run_decode(kvc, cfg, lens, caps, offs, Kp, Vp, lm, 1, seed=2, tc=tc)
    got, want, err, cap_hit = outs[0]
    assert err == kvc.KVC_ECAPACITY and cap_hit
    assert_bf16_close(got, want, "decode out at capacity")
    np.testing.assert_array_equal(dlen.cpu().numpy().reshape(-1), [300, 40])


def test_decode_over_oracle_packed_tiny_cache(kvc):
    """Decode over the cache the oracle packs for the tiny config."""
    from tests.oracle_pipeline import pack_all, score_all, select_all
    cfg = W.get_config("tiny")
    wl = W.make_workload(cfg)
    run = score_all(wl)
    sels = select_all(wl, run.util, run.cost, run.r)
    ent, lens, caps, offs = pack_all(wl, [s.taken for s in sels], run.r)
    rows = int(caps.sum())
    Kp = np.zeros((rows, cfg.d), np.float32); Vp = np.zeros_like(Kp); lm = np.zeros(rows, np.float32)
    for (b, l, h), (K, V, m, _) in ent.items():
        o = int(offs[b, l, h])
        Kp[o:o + len(K)] = K; Vp[o:o + len(K)] = V; lm[o:o + len(K)] = m
    outs, *_ = _run_decode(kvc, cfg, lens, caps, offs, Kp, Vp, lm, 4, seed=5)
    for got, want, err, _ in outs:
        assert err == 0
        assert_f32_close(got, want, "tiny decode", rel=1e-5, floor_frac=1.0, axis=-1)


def test_tc_decode_skips_and_reports_entries_past_the_packed_extent(kvc):
    """An (l,h) whose entries would run past packed_rows is skipped (length and
    output untouched) and reported; the other (l,h) still decode."""
    cfg = W.small_config(B=1, L=1, H=2, G=4, d=128, dtype="bf16", P=16, W=16, n_decode=2)
    rng = np.random.default_rng(9)
    lens, caps, offs, Kp, Vp, lm = _rand_cache(rng, 1, 1, 2, 128, [200, 300], 2, "bf16")
    p = params_for(cfg, n_max=400, S_max=1, packed_rows=int(offs[0, 0, 1]) + 100)
    bf = torch.bfloat16
    dKp, dVp, dlm = dev(Kp, bf), dev(Vp, bf), dev(lm)
    dpos = torch.zeros(Kp.shape[0], device="cuda")
    dlen = dev(lens.astype(np.int32))
    ws = kvc.workspace(kvc.KVC_WS_DECODE, p, zero=True)
    out = torch.full((1, 1, 8, 128), 7.0, dtype=bf, device="cuda")
    q = W.round_bf16(rng.standard_normal((1, 1, 8, 128)).astype(np.float32))
    kn = W.round_bf16(rng.standard_normal((1, 1, 2, 128)).astype(np.float32))
    vn = W.round_bf16(rng.standard_normal((1, 1, 2, 128)).astype(np.float32))
    kvc.kvc_decode_attn(p, dev(q, bf), dev(kn, bf), dev(vn, bf), None, dKp, dVp, dlm, dpos, dlen,
                        dev(caps.astype(np.int32)), dev(offs.astype(np.int64)), out, ws)
    assert kvc.kvc_device_error() == kvc.KVC_EDEVICE
    np.testing.assert_array_equal(dlen.cpu().numpy().reshape(-1), [201, 300])
    got = out.float().cpu().numpy()
    assert (got[0, 0, 4:] == 7.0).all()
    o = int(offs[0, 0, 0])
    want, *_ = O.decode_step_head(q[0, 0, :4], kn[0, 0, 0], vn[0, 0, 0],
                                  Kp[o:o + 200].astype(np.float64), Vp[o:o + 200].astype(np.float64),
                                  lm[o:o + 200].astype(np.float64))
    assert_bf16_close(got[0, 0, :4], want, "decode of the in-extent head")


@pytest.mark.parametrize("tc", [False, True])
def test_layer_range_decode_equals_all_layers(kvc, tc):
    """kvc_decode_attn_layers called layer by layer (batch 2, so a layer's
    (b,l,h) are strided in the per-(b,l,h) arrays) gives, bit for bit, the
    outputs, lengths and appended rows of kvc_decode_attn over all layers."""
    B, L, H, G, d = 2, 3, 2, 4, 128
    cfg = W.small_config(B=B, L=L, H=H, G=G, d=d, dtype="bf16", P=16, W=16, n_decode=2)
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 900, size=B * L * H)
    lens, caps, offs, Kp, Vp, lm = _rand_cache(rng, B, L, H, d, lens, 3, "bf16")
    p = params_for(cfg, n_max=max(int(lens.max()) + 64, cfg.W + 16), S_max=1,
                   packed_rows=Kp.shape[0] if tc else 0)
    bf = torch.bfloat16
    caches = []
    for _ in range(2):
        caches.append(dict(K=dev(Kp, bf), V=dev(Vp, bf), lm=dev(lm),
                           pos=torch.zeros(Kp.shape[0], device="cuda"),
                           len=dev(lens.astype(np.int32)),
                           ws=kvc.workspace(kvc.KVC_WS_DECODE, p, zero=True)))
    cap, off = dev(caps.astype(np.int32)), dev(offs.astype(np.int64))
    for t in range(2):
        q = dev(W.round_bf16(rng.standard_normal((B, L, H * G, d)).astype(np.float32)), bf)
        kn = dev(W.round_bf16(rng.standard_normal((B, L, H, d)).astype(np.float32)), bf)
        vn = dev(W.round_bf16(rng.standard_normal((B, L, H, d)).astype(np.float32)), bf)
        posn = torch.full((B,), 500.0 + t, device="cuda")
        a, c = caches
        out_a = torch.empty((B, L, H * G, d), dtype=bf, device="cuda")
        kvc.kvc_decode_attn(p, q, kn, vn, posn, a["K"], a["V"], a["lm"], a["pos"], a["len"], cap,
                            off, out_a, a["ws"])
        out_c = torch.empty_like(out_a)
        for l in range(L):
            o = torch.empty((B, 1, H * G, d), dtype=bf, device="cuda")
            kvc.kvc_decode_attn_layers(p, l, l + 1, q[:, l:l + 1].contiguous(),
                                       kn[:, l:l + 1].contiguous(), vn[:, l:l + 1].contiguous(),
                                       posn, c["K"], c["V"], c["lm"], c["pos"], c["len"], cap, off,
                                       o, c["ws"])
            out_c[:, l:l + 1] = o
        torch.cuda.synchronize()
        assert kvc.kvc_device_error() == 0
        assert torch.equal(out_a, out_c)
        for k in ("len", "K", "V", "lm", "pos"):
            assert torch.equal(a[k], c[k]), k
    with pytest.raises(kvc.KvcError):
        kvc.kvc_decode_attn_layers(p, 2, 2, q[:, :1].contiguous(), kn[:, :1].contiguous(),
                                   vn[:, :1].contiguous(), posn, c["K"], c["V"], c["lm"], c["pos"],
                                   c["len"], cap, off, out_c[:, :1].contiguous(), c["ws"])
