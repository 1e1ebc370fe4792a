"""Helpers shared by the GPU parity tests (device upload, tolerances)."""
import numpy as np
import torch

from kv_cache_compression_probe_gb300 import kvc

DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def dev(x, dtype=None, device="cuda"):
    t = torch.as_tensor(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device).contiguous()


def assert_bf16_close(got, want, what, abs_tol=2e-2, rel=2.0 ** -8):
    """bf16 tolerance (reading R12): |g - o| <= 2e-2 + 2^-8 |o|, o = float64 oracle."""
    g = np.asarray(got, np.float64)
    o = np.asarray(want, np.float64)
    err = np.abs(g - o)
    bad = err > abs_tol + rel * np.abs(o)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {err.max()}"
    rel_only = (err > abs_tol) & ~bad
    return int(rel_only.sum())


def assert_f32_close(got, want, what, rel=1e-5, floor_frac=1e-3, axis=None):
    """fp32 tolerance: |g - o| <= rel * max(|o|, floor_frac * max|o|)."""
    g = np.asarray(got, np.float64)
    o = np.asarray(want, np.float64)
    scale = np.abs(o).max(axis=axis, keepdims=axis is not None) if o.size else 1.0
    den = np.maximum(np.abs(o), floor_frac * scale)
    err = np.abs(g - o) / np.where(den > 0, den, 1.0)
    bad = err > rel
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max rel {err.max()}"


def params_for(cfg, n_max=None, S_max=None, **over):
    kw = dict(B=cfg.B, L=cfg.L, H=cfg.H, G=cfg.G, d=cfg.d, P=cfg.P, W=cfg.W,
              dtype=kvc.KVC_BF16 if cfg.dtype == "bf16" else kvc.KVC_F32,
              n_max=n_max or cfg.n, S_max=S_max or 1, rope_base=cfg.rope_base,
              hop_weight=cfg.hop_weight, n_hops=cfg.n_hops, w_part=cfg.w_part,
              w_value=cfg.w_value, value_floor=cfg.value_floor, budget_ratio=cfg.budget_ratio,
              budget_entries_per_lh=cfg.budget_entries_per_lh, floor_cap_frac=cfg.floor_cap_frac,
              floor_cap_tokens=cfg.floor_cap_tokens, decode_reserve=cfg.decode_reserve)
    kw.update(over)
    return kvc.make_params(**kw)


def upload_workload(wl, tensor_cores=True, tree_cuts=False, salient=False, **over):
    """Device copies of a synthetic workload plus a Compressor sized for it."""
    from kv_cache_compression_probe_gb300.pipeline import Compressor, pad_bounds
    cfg = wl.cfg
    S_max = max(len(s.slot_bounds) - 1 for s in wl.seqs)
    p = params_for(cfg, n_max=max(s.n for s in wl.seqs), S_max=S_max, **over)
    dt = DT[cfg.dtype]
    K = np.concatenate([s.K.reshape(-1, cfg.d) for s in wl.seqs])
    V = np.concatenate([s.V.reshape(-1, cfg.d) for s in wl.seqs])
    Qp = np.stack([s.Qp for s in wl.seqs])
    d = dict(K=dev(K, dt), V=dev(V, dt), Qp=dev(Qp, dt),
             bounds=dev(pad_bounds([s.slot_bounds for s in wl.seqs], S_max)),
             n_slots=dev(np.asarray([len(s.slot_bounds) - 1 for s in wl.seqs], np.int32)),
             sens=dev(wl.head_sens))
    comp = Compressor(p, [s.n for s in wl.seqs], tensor_cores=tensor_cores, tree_cuts=tree_cuts,
                      salient=salient)
    return p, comp, d, S_max


def token_view(x, wl, b, width=None):
    """Slice sequence b's [L, H, n(, width)] block out of a token-layout array."""
    cfg = wl.cfg
    start = sum(cfg.L * cfg.H * s.n for s in wl.seqs[:b])
    n = wl.seqs[b].n
    blk = x[start:start + cfg.L * cfg.H * n]
    return blk.reshape(cfg.L, cfg.H, n, *(() if width is None else (width,)))
