"""Bounded device waits (KVC_ETIMEOUT) on the GPU, without any fault.

kvc_set_wait_limit shortens the first wait of every pipeline stage and makes
the producers withhold their copies, so each consumer's wait can end only by
its limit: the kernels must give up, wait out what they issued, free their
tensor memory, record KVC_ETIMEOUT and return.  The context must stay usable:
after restoring the defaults (and zeroing the decode workspace, as kvc.h asks
after a timeout) the same call gives correct results again."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, dev, params_for, upload_workload

pytestmark = pytest.mark.gpu

DEFAULT_NS = 2_000_000_000


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    yield K
    K.kvc_set_wait_limit(DEFAULT_NS, False)


def test_wait_limit_arguments_are_checked(kvc):
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_set_wait_limit(10, False)
    assert ei.value.status == kvc.KVC_EINVAL
    with pytest.raises(kvc.KvcError):
        kvc.kvc_set_wait_limit(DEFAULT_NS + 1, False)
    kvc.kvc_set_wait_limit(DEFAULT_NS, False)


@pytest.mark.parametrize("tc", [True, False], ids=["tcgen05", "simt"])
def test_decode_wait_times_out_then_decodes_correctly(kvc, tc):
    cfg = W.small_config(B=1, L=2, H=3, G=4, d=128, dtype="bf16", P=16, W=16, n_decode=2)
    rng = np.random.default_rng(3)
    lens = np.asarray([0, 1, 300, 512, 513, 1100], np.int64).reshape(1, 2, 3)
    caps, offs = O.offsets(lens, 2)
    rows = int(caps.sum())
    Kp = W.round_bf16(rng.standard_normal((rows, 128)).astype(np.float32))
    Vp = W.round_bf16(rng.standard_normal((rows, 128)).astype(np.float32))
    lm = np.where(rng.uniform(size=rows) < 0.7, 0.0, rng.uniform(0, 3, size=rows)).astype(np.float32)
    p = params_for(cfg, n_max=int(lens.max()) + 64, S_max=1, packed_rows=rows if tc else 0)
    bf = torch.bfloat16
    q = W.round_bf16(rng.standard_normal((1, 2, 12, 128)).astype(np.float32))
    kn = W.round_bf16(rng.standard_normal((1, 2, 3, 128)).astype(np.float32))
    vn = W.round_bf16(rng.standard_normal((1, 2, 3, 128)).astype(np.float32))
    ws = kvc.workspace(kvc.KVC_WS_DECODE, p, zero=True)
    out = torch.empty((1, 2, 12, 128), dtype=bf, device="cuda")

    def call():
        c = [dev(Kp, bf), dev(Vp, bf), dev(lm), torch.zeros(rows, device="cuda"),
             dev(lens.astype(np.int32))]
        kvc.kvc_decode_attn(p, dev(q, bf), dev(kn, bf), dev(vn, bf), None, *c,
                            dev(caps.astype(np.int32)), dev(offs.astype(np.int64)), out, ws)
        torch.cuda.synchronize()
        return c

    assert kvc.kvc_device_error() == 0
    kvc.kvc_set_wait_limit(200_000, True)           # 0.2 ms, no copies issued
    try:
        call()
        assert kvc.kvc_device_error() == kvc.KVC_ETIMEOUT
    finally:
        kvc.kvc_set_wait_limit(DEFAULT_NS, False)
    ws.zero_()
    call()
    assert kvc.kvc_device_error() == 0
    got = out.float().cpu().numpy()
    for l in range(2):
        for h in range(3):
            o, n = int(offs[0, l, h]), int(lens[0, l, h])
            want, *_ = O.decode_step_head(q[0, l, h * 4:(h + 1) * 4], kn[0, l, h], vn[0, l, h],
                                          Kp[o:o + n].astype(np.float64),
                                          Vp[o:o + n].astype(np.float64),
                                          lm[o:o + n].astype(np.float64))
            assert_bf16_close(got[0, l, h * 4:(h + 1) * 4], want, f"decode (l={l}, h={h})")


def test_score_wait_times_out_then_scores_correctly(kvc):
    """The tensor-core passes of kvc_score (probe row statistics, per-key
    features, hop passes, node statistics) all time out; then a normal call
    matches the oracle."""
    cfg = W.small_config(B=1, L=1, H=2, n=640, n_min=640)
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl, tensor_cores=True)
    args = (d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    comp.score(*args)                               # reference: before any timeout
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    ref = [t.clone() for t in (comp.lse, comp.feats, comp.relevance, comp.op_util, comp.op_cost)]
    kvc.kvc_set_wait_limit(200_000, True)
    try:
        comp.score(*args)
        torch.cuda.synchronize()
        assert kvc.kvc_device_error() == kvc.KVC_ETIMEOUT
    finally:
        kvc.kvc_set_wait_limit(DEFAULT_NS, False)
    comp.score(*args)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    for a, b in zip(ref, (comp.lse, comp.feats, comp.relevance, comp.op_util, comp.op_cost)):
        assert torch.equal(a, b)
    s = wl.seqs[0]
    lse = comp.lse.cpu().numpy()
    rel = comp.relevance.cpu().numpy().reshape(cfg.L, cfg.H, s.n)
    for h in range(cfg.H):
        res = O.score_and_value_head(s.K[0, h], s.V[0, h], s.Qp[0, h * cfg.G:(h + 1) * cfg.G], s.n,
                                     cfg.P, s.slot_bounds, 1.0, base=cfg.rope_base)
        assert_f32_close(lse[0, 0, h], res.lse, "lse", rel=1e-5)
        assert_f32_close(rel[0, h], res.r, "relevance", rel=1e-5)
