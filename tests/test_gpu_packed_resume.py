"""Resuming decode from a saved packed cache: compress, decode some steps,
save the packed cache to .npz, load it into a fresh Compressor (as a new
process would) and decode the next steps on both.  Outputs, lengths and every
stored row must agree bit for bit."""
import numpy as np
import pytest
import torch

from synth import workloads as W
from tests.gpu_helpers import dev, upload_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


@pytest.mark.parametrize("tc", [True, False], ids=["tcgen05", "simt"])
def test_decode_resumes_from_a_saved_cache(kvc, tmp_path, tc):
    cfg = W.small_config()
    cfg = cfg.replace(n_decode=6)
    wl = W.make_workload(cfg)
    p, comp, d, S_max = upload_workload(wl, tensor_cores=tc)
    comp.compress(d["K"], d["V"], d["Qp"], d["bounds"], d["n_slots"], d["sens"])
    dec = [W.decode_inputs(cfg, t) for t in range(6)]
    dt = comp.Kp.dtype
    q, kn, vn = (dev(np.stack([x[i] for x in dec]), dt) for i in range(3))
    out = torch.empty(tuple(q.shape), dtype=dt, device="cuda")
    comp.decode_many(q[:3], kn[:3], vn[:3], out[:3], graph=False)
    path = str(tmp_path / "packed.npz")
    comp.save_packed(path)

    p2, comp2, _, _ = upload_workload(wl, tensor_cores=tc)
    comp2.load_packed(path)
    out2 = torch.empty_like(out)
    comp.decode_many(q[3:], kn[3:], vn[3:], out[3:], graph=False)
    comp2.decode_many(q[3:], kn[3:], vn[3:], out2[3:], graph=False)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    assert torch.equal(out[3:].view(torch.int16) if dt == torch.bfloat16 else out[3:],
                       out2[3:].view(torch.int16) if dt == torch.bfloat16 else out2[3:])
    assert torch.equal(comp.len_lh, comp2.len_lh)
    rows = int(comp.cap_lh.to(torch.int64).sum())
    for n in ("Kp", "Vp", "logm", "pos"):
        a, b = getattr(comp, n)[:rows], getattr(comp2, n)[:rows]
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), n
