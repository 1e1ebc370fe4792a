"""The allocation-free decode entry point.

Some callers cannot allocate device memory for the library (a serving engine
whose pool already holds all free HBM for KV blocks, or a host framework whose
plugin interface cannot pass a workspace and forbids cudaMalloc / cudaFree in
extensions).  kvc_decode_attn_noalloc serves them with a fixed scratch array in
the library's device image.  This test calls it through the C ABI and checks it
against kvc_decode_attn (which takes a caller workspace) on two calls in a row,
on both decode kernels: the SIMT split-K kernel (no packed extent given), and
the tensor-core kernel (bf16, d = 128, packed extent given) with its work list
built inside the attention kernel (at most 1024 (b,l,h)) and written by the
plan kernel into the static array (more than 1024).
It lives in its own file, collected last, and needs nothing from other tests.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import assert_bf16_close, dev, params_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


CASES = {
    # name: (B, L, H, G, lengths or None for a seeded draw, tensor-core decode)
    "simt": (2, 2, 3, 4, [0, 1, 255, 256, 257, 600, 1023, 31, 512, 2, 800, 100], False),
    "tc-in-kernel-list": (2, 2, 3, 4, [0, 1, 255, 256, 257, 600, 1023, 31, 512, 2, 800, 100], True),
    "tc-plan-kernel": (1, 33, 32, 2, None, True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_decode_matches_workspace_decode(kvc, name):
    B, L, H, G, lens, tc = CASES[name]
    cfg = W.small_config(B=B, L=L, H=H, G=G, d=128, dtype="bf16", P=16, W=16, n_decode=4)
    rng = np.random.default_rng(11)
    if lens is None:
        lens = rng.integers(0, 700, size=B * L * H)
    lens = np.asarray(lens, np.int64).reshape(B, L, H)
    assert (B * L * H > 1024) == (name == "tc-plan-kernel")
    caps, offs = O.offsets(lens, 4)
    rows = int(caps.sum())
    Kp = W.round_bf16(rng.standard_normal((rows, 128)).astype(np.float32))
    Vp = W.round_bf16(rng.standard_normal((rows, 128)).astype(np.float32))
    lm = np.where(rng.uniform(size=rows) < 0.7, 0.0, rng.uniform(0, 3, size=rows)).astype(np.float32)
    p = params_for(cfg, n_max=int(lens.max()) + 64, S_max=1, packed_rows=rows if tc else 0)
    assert kvc.kvc_workspace_bytes(kvc.KVC_WS_DECODE, p) <= kvc.KVC_DECODE_STATIC_SCRATCH_BYTES
    bf = torch.bfloat16

    def cache():
        return [dev(Kp, bf), dev(Vp, bf), dev(lm), torch.zeros(rows, device="cuda"),
                dev(lens.astype(np.int32))]

    A, Bc = cache(), cache()
    dcap, doff = dev(caps.astype(np.int32)), dev(offs.astype(np.int64))
    ws = kvc.workspace(kvc.KVC_WS_DECODE, p, zero=True)
    outA = torch.empty((B, L, H * G, 128), dtype=bf, device="cuda")
    outB = torch.empty_like(outA)
    for t in range(2):
        q = dev(W.round_bf16(rng.standard_normal((B, L, H * G, 128)).astype(np.float32)), bf)
        kn = dev(W.round_bf16(rng.standard_normal((B, L, H, 128)).astype(np.float32)), bf)
        vn = dev(W.round_bf16(rng.standard_normal((B, L, H, 128)).astype(np.float32)), bf)
        n0 = kvc.kvc_launch_count()
        kvc.kvc_decode_attn(p, q, kn, vn, None, A[0], A[1], A[2], A[3], A[4], dcap, doff, outA, ws)
        n1 = kvc.kvc_launch_count()
        kvc.kvc_decode_attn_noalloc(p, q, kn, vn, None, Bc[0], Bc[1], Bc[2], Bc[3], Bc[4], dcap,
                                    doff, outB)
        n2 = kvc.kvc_launch_count()
        torch.cuda.synchronize()
        assert kvc.kvc_device_error() == 0
        assert n2 - n1 == n1 - n0 > 0          # the same kernels, on the same path
        assert_bf16_close(outB.float().cpu().numpy(), outA.float().cpu().numpy(),
                          f"allocation-free decode ({name}), call {t}")
        assert torch.equal(A[4], Bc[4])
        assert torch.equal(A[0], Bc[0]) and torch.equal(A[1], Bc[1])
        assert torch.equal(A[2], Bc[2])
    assert (Bc[4].cpu().numpy() == (lens + 2)).all()


def test_noalloc_rejects_problems_beyond_its_scratch(kvc):
    cfg = W.small_config(B=4, L=64, H=64, G=4, d=128, dtype="bf16", P=16, W=16)
    p = params_for(cfg, n_max=131072, S_max=1)
    assert kvc.kvc_workspace_bytes(kvc.KVC_WS_DECODE, p) > (48 << 20)
    t = torch.zeros(16, device="cuda")
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_decode_attn_noalloc(p, t, t, t, None, t, t, t, t, t.int(), t.int(), t.long(), t)
    assert ei.value.status == kvc.KVC_ESCRATCH
