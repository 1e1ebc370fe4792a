"""Packed-cache .npz files (checkpoint/replay of the compressed cache): a
write/read round trip is bit for bit, bf16 rows included, and only the rows
of the (b, l, h) capacities are stored.  CPU only."""
import numpy as np
import pytest
import torch

from kv_cache_compression_probe_gb300 import kvc
from kv_cache_compression_probe_gb300.pipeline import read_packed, write_packed


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_round_trip_is_bit_exact(tmp_path, dt):
    g = torch.Generator().manual_seed(3)
    B, L, H, d = 1, 2, 3, 16
    cap = torch.tensor([[5, 0, 7], [3, 9, 1]], dtype=torch.int32).view(B, L, H)
    off = torch.cumsum(torch.cat([torch.zeros(1, dtype=torch.int64), cap.view(-1).to(torch.int64)]),
                       0)[:-1].view(B, L, H)
    rows = int(cap.sum())
    extra = 4                                         # buffer rows past the capacities
    t = {"Kp": torch.randn(rows + extra, d, generator=g).to(dt),
         "Vp": torch.randn(rows + extra, d, generator=g).to(dt),
         "logm": torch.rand(rows + extra, generator=g),
         "pos": torch.arange(rows + extra, dtype=torch.float32),
         "len_lh": (cap - 1).clamp(min=0), "cap_lh": cap, "off_lh": off}
    p = kvc.make_params(B=B, L=L, H=H, G=2, d=d, P=4, W=2,
                        dtype=kvc.KVC_BF16 if dt == torch.bfloat16 else kvc.KVC_F32,
                        n_max=64, S_max=3, decode_reserve=2, budget_ratio=0.3)
    f = tmp_path / "cache.npz"
    write_packed(str(f), p, t)
    params, r = read_packed(str(f))
    assert params["B"] == B and params["d"] == d and params["decode_reserve"] == 2
    assert abs(params["budget_ratio"] - 0.3) < 1e-15 and "tree_cuts" not in params
    for n in ("Kp", "Vp", "logm", "pos"):
        assert r[n].shape[0] == rows and r[n].dtype == t[n].dtype
        assert torch.equal(r[n].view(torch.uint8), t[n][:rows].contiguous().view(torch.uint8))
    for n in ("len_lh", "cap_lh", "off_lh"):
        assert torch.equal(r[n], t[n])


def test_rejects_another_format(tmp_path):
    f = tmp_path / "x.npz"
    np.savez(f, format=np.int64(99))
    with pytest.raises(ValueError):
        read_packed(str(f))
