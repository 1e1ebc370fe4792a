"""Decode over many steps as one CUDA graph (DecodeGraph) against the same steps
issued one call at a time: identical outputs, lengths and appended rows."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import dev, params_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


@pytest.mark.parametrize("tc", [True, False])
def test_graph_decode_matches_eager_steps(kvc, tc):
    from kv_cache_compression_probe_gb300.pipeline import DecodeGraph
    T = 6
    cfg = W.small_config(B=2, L=2, H=3, G=4, d=128, dtype="bf16", P=16, W=16, n_decode=T)
    rng = np.random.default_rng(21)
    lens = np.asarray([0, 1, 255, 256, 257, 600, 1023, 31, 512, 2, 800, 100], np.int64).reshape(2, 2, 3)
    caps, offs = O.offsets(lens, 2 * T)              # room for two replays
    rows = int(caps.sum())
    Kp = W.round_bf16(rng.standard_normal((rows, 128)).astype(np.float32))
    Vp = W.round_bf16(rng.standard_normal((rows, 128)).astype(np.float32))
    lm = np.where(rng.uniform(size=rows) < 0.7, 0.0, rng.uniform(0, 3, size=rows)).astype(np.float32)
    p = params_for(cfg, n_max=int(lens.max()) + 64, S_max=1, packed_rows=rows if tc else 0)
    bf = torch.bfloat16

    def cache():
        return [dev(Kp, bf), dev(Vp, bf), dev(lm), torch.zeros(rows, device="cuda"),
                dev(lens.astype(np.int32))]

    A, B = cache(), cache()
    dcap, doff = dev(caps.astype(np.int32)), dev(offs.astype(np.int64))
    wsA = kvc.workspace(kvc.KVC_WS_DECODE, p, zero=True)
    wsB = kvc.workspace(kvc.KVC_WS_DECODE, p, zero=True)
    q = dev(W.round_bf16(rng.standard_normal((T, 2, 2, 12, 128)).astype(np.float32)), bf)
    kn = dev(W.round_bf16(rng.standard_normal((T, 2, 2, 3, 128)).astype(np.float32)), bf)
    vn = dev(W.round_bf16(rng.standard_normal((T, 2, 2, 3, 128)).astype(np.float32)), bf)
    pn = torch.arange(T * 2, dtype=torch.float32, device="cuda").view(T, 2) + 5000.0
    outA = torch.empty((T, 2, 2, 12, 128), dtype=bf, device="cuda")
    outB = torch.empty_like(outA)
    for t in range(T):
        kvc.kvc_decode_attn(p, q[t], kn[t], vn[t], pn[t], A[0], A[1], A[2], A[3], A[4], dcap, doff,
                            outA[t], wsA)
    g = DecodeGraph(p, q, kn, vn, pn, B[0], B[1], B[2], B[3], B[4], dcap, doff, outB, wsB)
    # tensor cores with <= 1024 (b,l,h): attention (own work list) + merge;
    # SIMT: split-K kernel + length commit
    assert g.launches == T * 2
    g.replay()
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    assert torch.equal(outA, outB)
    for x, y in zip(A, B):
        assert torch.equal(x, y)
    assert (B[4].cpu().numpy() == (lens + T)).all()
    # a second replay continues from the advanced lengths with new inputs
    q.copy_(q.flip(0))
    for t in range(T):
        kvc.kvc_decode_attn(p, q[t], kn[t], vn[t], pn[t], A[0], A[1], A[2], A[3], A[4], dcap, doff,
                            outA[t], wsA)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outA, outB)
    assert torch.equal(A[4], B[4])
