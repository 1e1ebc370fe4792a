"""GPU parity of kvc_partition (a0: curvature of the normalised hidden-state
trajectory, then the slot-length dynamic program) against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from synth import workloads as W
from tests.gpu_helpers import DT, dev, params_for
from tests.partition_lambda import partition_lambda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_probe_gb300 import build, kvc as K
    build.build()
    return K


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_partition_matches_oracle(kvc, dtype):
    cfg = W.get_config("long").replace(B=2, n=2400, n_min=1700, L=1, H=1, hidden_dim=256,
                                       dtype=dtype)
    ns = W.context_lengths(cfg)
    n_max = int(ns.max())
    dh = cfg.hidden_dim
    hid = np.zeros((cfg.B, n_max, dh), np.float32)
    planted = []
    for b in range(cfg.B):
        pb = W.planted_bounds(cfg, b, int(ns[b]))
        planted.append(pb)
        hid[b, :ns[b]] = W.hidden_states(cfg, b, int(ns[b]), pb)
    S_max = max(int(n - cfg.W) // 16 + 1 for n in ns)
    p = params_for(cfg, n_max=n_max, S_max=S_max)
    ws = kvc.workspace(kvc.KVC_WS_PARTITION, p)
    kappa = torch.zeros((cfg.B, n_max), device="cuda")
    bounds = torch.zeros((cfg.B, S_max + 1), dtype=torch.int32, device="cuda")
    nsl = torch.zeros((cfg.B,), dtype=torch.int32, device="cuda")
    kvc.kvc_partition(p, dev(ns.astype(np.int32)), dev(hid, DT[dtype]), dh, kappa, bounds, nsl, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error() == 0
    kg = kappa.cpu().numpy().astype(np.float64)
    bg = bounds.cpu().numpy()
    ng = nsl.cpu().numpy()
    for b in range(cfg.B):
        n = int(ns[b])
        end = n - cfg.W
        ko = O.curvature(hid[b, :n].astype(np.float64))
        # curvature: 1 - cos of fp32 differences; absolute tolerance
        assert np.abs(kg[b, :n] - ko).max() < 2e-5
        # the DP on the same kappa and the same lambda is bit-exact
        cuts = O.partition_dp(kg[b], end, lam=partition_lambda(kg[b], end))
        S = int(ng[b])
        np.testing.assert_array_equal(bg[b, :S + 1], cuts)
        assert all(16 <= y - x <= 128 for x, y in zip(cuts[:-1], cuts[1:]))
        # functional: cuts land on the planted turns
        inner = planted[b][1:-1]
        hit = np.mean([np.abs(cuts - t).min() <= 2 for t in inner])
        assert hit >= 0.9
