"""Benchmark of the budgeted KV-compression + ragged-decode hot path on GB300.

One step = one pass of the whole path over one synthetic batch:
kvc_score -> kvc_select -> kvc_merge_pack (compression after prefill), then
`decode_steps` calls of kvc_decode_attn (all layers per call, append + attend).
Workload (default): the Mistral-7B-shaped 16K cache (32 layers, 8 KV / 32 query
heads, d 128, bf16, batch 1, 25% budget, 128-token window, 1% singleton cap,
256 decode steps).  Inputs are seeded synthetic caches (see synth/), resident
in HBM for `value`; `e2e` copies them from pinned host memory every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent
replica of the workload (the path shards by sequence; no collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV tokens compressed/s and ragged decode-attn GB/s (fraction of HBM/TC peak)"
DC_B_MIN = 32          # DistillCache Algorithm 1: minimum budget
UNIT = "KV tokens/s"


# --------------------------------------------------------------------------- inputs
def _gen_head(args):
    from synth import workloads as W
    cfg, b, l, h, n, bounds, cnt = args
    K, V, Q, _ = W.gen_head(cfg, b, l, h, n, bounds, cnt)
    return l, h, K, V, Q


def make_inputs(cfg, pool):
    """Host arrays of the synthetic workload (generated in parallel by heads)."""
    from synth import workloads as W
    seqs = []
    for b, n in enumerate(W.context_lengths(cfg)):
        n = int(n)
        bounds = W.planted_bounds(cfg, b, n)
        counts = W._needle_counts(cfg, b, n)
        jobs = [(cfg, b, l, h, n, bounds, int(counts[l * cfg.H + h]))
                for l in range(cfg.L) for h in range(cfg.H)]
        K = np.zeros((cfg.L, cfg.H, n, cfg.d), np.float32)
        V = np.zeros_like(K)
        Qp = np.zeros((cfg.L, cfg.H * cfg.G, cfg.P, cfg.d), np.float32)
        for l, h, k, v, q in pool.imap_unordered(_gen_head, jobs, chunksize=4):
            K[l, h] = k; V[l, h] = v; Qp[l, h * cfg.G:(h + 1) * cfg.G] = q
        seqs.append((n, bounds, K, V, Qp))
    return seqs


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi every 20 ms during the timed region: median SM clock, max clock and
    any throttle reason seen; only samples stamped inside [begin, end] count."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.proc = None
        # the raw samples go to a scratch file; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"kvc_bench_clocks_{os.getpid()}.csv")
        self.gpu = gpu_index
        self.t_begin = self.t_end = None

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        t0 = time.time()                              # sampling is live once a line lands
        while time.time() - t0 < 10.0 and self.proc.poll() is None:
            self.f.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
            except (ValueError, IndexError):
                ts = None
            if ts is not None and self.t_begin is not None and self.t_end is not None:
                if ts < self.t_begin - 0.02 or ts > self.t_end + 0.02:
                    continue
            try:
                sm.append(float(parts[2])); smax.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_traffic(name: str, src_files):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source (hash match); else None."""
    path = os.path.join(ROOT, "profiles", f"{name}.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    h = hashlib.sha256()
    for f in src_files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch")


# the kernels the committed end-to-end selection record depends on (the same
# list as tests/test_gpu_full_size.py)
PARITY_SOURCES = ("kv_cache_compression_probe_gb300/csrc/kvc_score.cu",
                  "kv_cache_compression_probe_gb300/csrc/kvc_score_tc.cu",
                  "kv_cache_compression_probe_gb300/csrc/kvc_select.cu",
                  "kv_cache_compression_probe_gb300/csrc/kvc_common.cuh")


def select_roofline(cfg, seqs, sel_ms, hbm):
    """kvc_select against HBM: each of the up to 8 radix passes (8-bit digits of
    a 64-bit key) of the floor reads every token's weight byte and relevance
    (5 B) and each of the auction reads every op's key and cost (12 B); the
    tail replays and offsets are negligible.  The passes are many small
    launches, so the call is bound by launch and reduction latency."""
    LH = cfg.L * cfg.H
    ops = sum(LH * (len(s[1]) - 1) * 16 for s in seqs)
    toks = sum(LH * s[0] for s in seqs)
    nbytes = 8 * (ops * 12 + toks * 5)
    gbs = nbytes / (sel_ms * 1e-3) / 1e9
    return {"bound": "latency (launches and reductions)", "achieved": gbs, "peak": hbm,
            "unit": "GB/s", "frac": gbs / hbm, "algorithmic_bytes": nbytes,
            "bytes_note": "8 radix passes x (ops x 12 B + tokens x 5 B), an upper bound"}


def parity_record(name: str):
    """The end-to-end selection parity of a workload (device chain against the
    float64 oracle chain, near-ties within 1e-6 counted) as written by the
    full-size GPU test and committed under profiles/; marked stale when the
    kernels it depends on changed since."""
    path = os.path.join(ROOT, "profiles", f"parity_{name}.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    h = hashlib.sha256()
    for f in PARITY_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    seqs = rec.get("sequences", [])
    return {"source": "profiles/parity_%s.json (tests/test_gpu_full_size.py)" % name,
            "current": rec.get("source_sha256") == h.hexdigest(),
            "selection_end_to_end": "device taken set == oracle chain's up to 1e-6 ties",
            "tie_band_rel": rec.get("tie_band_rel"),
            "ops": sum(x["ops"] for x in seqs),
            "ties_reported": sum(x["ties_reported"] for x in seqs),
            "tie_runs_reordered": sum(x["tie_runs_reordered"] for x in seqs),
            "max_abs_err": max((x["util_max_abs_err"] for x in seqs), default=None),
            "max_rel_err": max((x["util_max_rel_err"] for x in seqs), default=None),
            "util_within_1e5_rel": sum(x.get("util_within_1e5_rel", 0) for x in seqs) or None,
            "util_within_scale_term_only": (sum(x["util_within_scale_term_only"] for x in seqs)
                                            if seqs and "util_within_scale_term_only" in seqs[0]
                                            else None),
            "util_worst_err_over_bound": max((x.get("util_worst_err_over_bound", 0) for x in seqs),
                                             default=None)}


# --------------------------------------------------------------------------- GPU arm
def full_cache_decode_ms(p, cfg, seqs, K, V, q_all, kn_all, vn_all, D, dev, stream):
    """Mean ms per decode step of the same decode call over the uncompressed cache.
    At budget 1 every token is stored exact with ln m = 0 (the full-budget pack
    is the input, bit for bit), so the beta = 1 pack is the token layout with
    the decode reserve after each (b, l, h) range."""
    import torch
    from kv_cache_compression_probe_gb300 import kvc
    LH = cfg.L * cfg.H
    res = p.decode_reserve
    lens, tok0 = [], 0
    for s in seqs:
        lens += [s[0]] * LH
    caps = np.asarray(lens, np.int64) + res
    offs = np.concatenate([[0], np.cumsum(caps)[:-1]])
    rows = int(caps.sum())
    Kf = torch.empty((rows, cfg.d), dtype=K.dtype, device=dev)
    Vf = torch.empty_like(Kf)
    k = 0
    for s in seqs:
        n = s[0]
        dst = Kf[int(offs[k]):int(offs[k]) + LH * (n + res)].view(LH, n + res, cfg.d)
        dst[:, :n] = K[tok0:tok0 + LH * n].view(LH, n, cfg.d)
        dst = Vf[int(offs[k]):int(offs[k]) + LH * (n + res)].view(LH, n + res, cfg.d)
        dst[:, :n] = V[tok0:tok0 + LH * n].view(LH, n, cfg.d)
        tok0 += LH * n
        k += LH
    pf = type(p).from_buffer_copy(p)
    pf.packed_rows = rows
    logm = torch.zeros(rows, dtype=torch.float32, device=dev)
    pos = torch.zeros(rows, dtype=torch.float32, device=dev)
    len0 = torch.tensor(lens, dtype=torch.int32, device=dev)
    cap = torch.tensor(caps.astype(np.int32), device=dev)
    off = torch.tensor(offs.astype(np.int64), device=dev)
    ws = kvc.workspace(kvc.KVC_WS_DECODE, pf, dev, zero=True)
    out = torch.empty(q_all.shape[1:], dtype=q_all.dtype, device=dev)
    ln = len0.clone()

    def run(steps):
        for t in range(steps):
            kvc.kvc_decode_attn(pf, q_all[t], kn_all[t], vn_all[t], None, Kf, Vf, logm, pos, ln,
                                cap, off, out, ws, stream)

    run(min(3, D))                                       # warm-up
    ln.copy_(len0)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(D)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if kvc.kvc_device_error() != 0:
        raise RuntimeError("device error in the full-cache decode")
    ms = e0.elapsed_time(e1) / D
    del Kf, Vf
    torch.cuda.empty_cache()
    return ms


def evict_leg(p, cfg, seqs, K, V, q_all, kn_all, vn_all, D, dev, stream):
    """NEXT f2 on the same workload: DistillCache per-step top-B eviction with the
    attention score (budget ratio = the workload's, minimum budget 32 as in
    DistillCache Algorithm 1),
    starting from the full prompt cache.  Times the D steps (decode with LSE,
    alpha, top-B + compaction) as one CUDA graph replay and, eagerly, each call
    kind; returns a dict for the JSON line."""
    import torch
    from kv_cache_compression_probe_gb300 import kvc
    from kv_cache_compression_probe_gb300.pipeline import EvictingCache
    LH = cfg.L * cfg.H
    ns = [s[0] for s in seqs]
    B, n_max = len(ns), max(ns)
    if B == 1:
        Kb = K[:LH * ns[0]].view(1, cfg.L, cfg.H, ns[0], cfg.d)
        Vb = V[:LH * ns[0]].view(1, cfg.L, cfg.H, ns[0], cfg.d)
    else:
        Kb = torch.zeros((B, cfg.L, cfg.H, n_max, cfg.d), dtype=K.dtype, device=dev)
        Vb = torch.zeros_like(Kb)
        tok0 = 0
        for b, n in enumerate(ns):
            Kb[b, :, :, :n] = K[tok0:tok0 + LH * n].view(cfg.L, cfg.H, n, cfg.d)
            Vb[b, :, :, :n] = V[tok0:tok0 + LH * n].view(cfg.L, cfg.H, n, cfg.d)
            tok0 += LH * n
    pe = type(p).from_buffer_copy(p)
    pe.decode_reserve = 0
    cache = EvictingCache(pe, Kb, Vb, ns, D + 1, cfg.budget_ratio, DC_B_MIN)
    nseen = torch.tensor([[n + t + 1 for n in ns] for t in range(D)], dtype=torch.int64, device=dev)
    posn = torch.tensor([[n + t for n in ns] for t in range(D)], dtype=torch.float32, device=dev)
    out = torch.empty(tuple(q_all.shape), dtype=q_all.dtype, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    cache.run_many(q_all, kn_all, vn_all, out, nseen, posn, graph=True)     # capture + warm-up
    lens_end = cache.len_lh.cpu().numpy().astype(np.int64)
    reps = []
    for _ in range(3):
        cache.reset()
        torch.cuda.synchronize(dev)
        e0, e1 = ev(), ev()
        e0.record(stream)
        launches = cache.run_many(q_all, kn_all, vn_all, out, nseen, posn, graph=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        reps.append(e0.elapsed_time(e1) / D)
    # eager, per call kind (events between calls)
    cache.reset()
    torch.cuda.synchronize(dev)
    part = {"decode_lse": 0.0, "alpha": 0.0, "topb_evict": 0.0}
    for t in range(D):
        m = [ev() for _ in range(4)]
        m[0].record(stream)
        kvc.kvc_decode_attn_lse(pe, q_all[t], kn_all[t], vn_all[t], posn[t], cache.K, cache.V,
                                cache.logm, cache.pos, cache.len_lh, cache.cap_lh, cache.off_lh,
                                out[t], cache.lse, cache.scores, cache.ws_decode, stream)
        m[1].record(stream)
        kvc.kvc_token_alpha(pe, q_all[t], cache.K, cache.scores, cache.len_lh, cache.off_lh,
                            cache.lse, cache.alpha, cache.ws_evict, stream)
        m[2].record(stream)
        kvc.kvc_evict_topb(pe, cache.alpha, nseen[t], cache.ratio, cache.b_min, cache.K, cache.V,
                           cache.pos, cache.logm, cache.off_lh, cache.len_lh, cache.ws_evict,
                           stream)
        m[3].record(stream)
        torch.cuda.synchronize(dev)
        part["decode_lse"] += m[0].elapsed_time(m[1]) / D
        part["alpha"] += m[1].elapsed_time(m[2]) / D
        part["topb_evict"] += m[2].elapsed_time(m[3]) / D
    if kvc.kvc_device_error() != 0:
        raise RuntimeError("device error in the eviction leg")
    esz = 2 if cfg.dtype == "bf16" else 4
    kept = int(lens_end.sum())                       # entries after the last eviction
    # algorithmic bytes of a steady-state step: decode streams the kept entries
    # (K, V, log m) plus the new token and writes each entry's G scores; alpha
    # reads the scores; the eviction moves one row per (l,h) (read + write K,
    # V, pos, log m)
    LHB = LH * B
    per_step = (kept * (2 * cfg.d * esz + 4) + LHB * (2 * cfg.d * esz + 8) + 2 * kept * cfg.G * 4
                + LHB * 2 * (2 * cfg.d * esz + 8))
    ms = min(reps)
    return {"ms_per_step": ms, "launches_per_step": launches / D,
            "breakdown_ms_per_step_eager": part,
            "entries_after_eviction": kept, "ratio": cfg.budget_ratio, "b_min": DC_B_MIN,
            "algorithmic_bytes_per_step": per_step,
            "hbm_gbs": per_step / (ms * 1e-3) / 1e9,
            "note": "DistillCache Algorithm 1 with the attention score alpha; prompt cache "
                    "evicted to the budget at the first step, then one entry per step"}


def tree_cuts_leg(comp, K, bounds, n_slots, cfg, tokens, hbm, dev, reps=5):
    """f3: device time of kvc_tree_cuts alone (curvature of every key, then the
    cut of every internal tree node), CUDA events around `reps` calls after one
    untimed call.  Algorithmic bytes: K read once, the curvature written and
    read back, 8 bytes of cut table per slot tree."""
    import torch
    from kv_cache_compression_probe_gb300 import kvc
    stream = torch.cuda.current_stream(dev)

    def call():
        kvc.kvc_tree_cuts(comp.p, comp.ctx_len, K, comp.rope_cos, comp.rope_sin, bounds,
                          n_slots, comp.tree_kappa, comp.cuts, stream)
    call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / reps
    esz = 2 if cfg.dtype == "bf16" else 4
    rows = tokens * cfg.L * cfg.H
    trees = cfg.B * cfg.L * cfg.H * comp.p.S_max
    nbytes = rows * (cfg.d * esz + 8) + trees * 8
    cuts = comp.cuts[..., :7].to(torch.int64)
    bd = bounds.to(torch.int64)
    x0 = bd[:, None, None, :-1].expand(-1, cfg.L, cfg.H, -1)
    y0 = bd[:, None, None, 1:].expand(-1, cfg.L, cfg.H, -1)
    valid = (torch.arange(comp.p.S_max, device=bd.device)[None, :] < n_slots[:, None].to(torch.int64))
    root_off = (cuts[..., 0] != (y0 - x0) // 2)[valid[:, None, None, :].expand_as(x0)]
    return {"ms": ms, "hbm_gbs": nbytes / (ms * 1e-3) / 1e9, "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm,
            "algorithmic_bytes": nbytes,
            "root_cut_off_midpoint_frac": float(root_off.float().mean().cpu()),
            "note": "kvc_tree_cuts (key_curv_kernel + tree_cut_kernel), timed alone; it also "
                    "runs inside every timed step's scoring call"}


def compression_reps(comp, K, V, Qp, bounds, n_slots, cfg, tokens, graph, dev, reps=20):
    """Compression alone (kvc_score + kvc_select + kvc_merge_pack, graph replays
    when the step uses them): `reps` repetitions after the step's warm-ups, each
    bracketed by CUDA events on the launching stream; per-call and total
    medians.  K and V (2 GB at 16K) exceed L2, so no flush is added."""
    import torch
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    per = {"score": [], "select": [], "merge_pack": [], "total": []}
    for _ in range(reps):
        m = [ev() for _ in range(4)]
        m[0].record(stream)
        comp.score(K, V, Qp, bounds, n_slots, graph=graph)
        m[1].record(stream)
        comp.select(bounds, n_slots, graph=graph)
        m[2].record(stream)
        comp.merge_pack(K, V, bounds, n_slots, graph=graph)
        m[3].record(stream)
        torch.cuda.synchronize(dev)
        per["score"].append(m[0].elapsed_time(m[1]))
        per["select"].append(m[1].elapsed_time(m[2]))
        per["merge_pack"].append(m[2].elapsed_time(m[3]))
        per["total"].append(m[0].elapsed_time(m[3]))
    med = {k: statistics.median(v) for k, v in per.items()}
    return {"reps": reps, "median_ms": med,
            "kv_tokens_per_s": tokens / (med["total"] * 1e-3),
            "lh_entries_per_s": tokens * cfg.L * cfg.H / (med["total"] * 1e-3),
            "min_ms": min(per["total"]), "max_ms": max(per["total"])}


def scoring_gemm(comp, K, V, Qp, bounds, n_slots, cfg, tokens, tc_peak, dev):
    """Device time of the probe-times-key contraction passes of one kvc_score
    call (CUDA events the library records between its phases when phase
    timing is on; one untimed call outside the timed region).  The
    row-statistics pass and the per-key feature pass each contract every key
    with every probe row: 2 * (G*P) * n * d flops per (b, l, h)."""
    import torch
    from kv_cache_compression_probe_gb300 import kvc
    torch.cuda.synchronize(dev)
    kvc.kvc_set_phase_timing(True)
    try:
        comp.score(K, V, Qp, bounds, n_slots)
        ms = kvc.kvc_score_phase_ms(5)
    finally:
        kvc.kvc_set_phase_timing(False)
    flops = 2.0 * cfg.G * cfg.P * tokens * cfg.L * cfg.H * cfg.d   # one contraction pass
    out = {}
    for name, t in (("probe_rowstats", ms[0]), ("probe_feats", ms[1])):
        tf = flops / (t * 1e-3) / 1e12
        out[name] = {"ms": t, "tflops": tf, "frac_of_bf16_peak": tf / tc_peak}
    out["other_phases_ms"] = {"norms_and_hops": ms[2], "prototypes": ms[3],
                              "node_statistics": ms[4]}
    out["note"] = ("CUDA events between kvc_score's phases (one untimed call); flops = "
                   "2 * G*P * n * d per (b, l, h); peak = measured bf16 burst")
    return out


def full_bytes_ratio(cfg, seqs, avg_entries, D):
    """Entries the full cache streams per decode step over the compressed one."""
    full = sum(s[0] for s in seqs) * cfg.L * cfg.H
    LHB = cfg.L * cfg.H * len(seqs)
    return (full + LHB * (D + 1) / 2.0) / avg_entries


def replica_config(cfg, rank: int):
    """The workload replica `rank` runs: sequences are independent auctions, so
    every rank compresses and decodes its own seeded batch (no collective on the
    data path); rank 0 keeps the base seed."""
    return cfg.replace(seed=cfg.seed + rank) if rank else cfg


def max_over_ranks(vals, world: int, device=None):
    """Element-wise max of `vals` over the ranks of the default process group
    (the job's time is its slowest rank's); identity for one rank."""
    if world <= 1:
        return [float(v) for v in vals]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job units per second: every rank processes `units_per_rank` per
    step and the step takes the slowest rank's time."""
    return units_per_rank * world / (ms_per_step * 1e-3)


def run_gpu(args, cfg, rank, world):
    import torch
    import torch.distributed as dist
    from kv_cache_compression_probe_gb300 import kvc
    from kv_cache_compression_probe_gb300.pipeline import Compressor, pad_bounds
    from synth import workloads as W

    cfg = replica_config(cfg, rank)
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(16, os.cpu_count() or 4)) as pool:
        seqs = make_inputs(cfg, pool)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    S_max = max(len(s[1]) - 1 for s in seqs)
    p = kvc.make_params(B=cfg.B, L=cfg.L, H=cfg.H, G=cfg.G, d=cfg.d, P=cfg.P, W=cfg.W,
                        dtype=kvc.KVC_BF16 if cfg.dtype == "bf16" else kvc.KVC_F32,
                        n_max=max(s[0] for s in seqs), S_max=S_max, rope_base=cfg.rope_base,
                        hop_weight=cfg.hop_weight, n_hops=cfg.n_hops, w_part=cfg.w_part,
                        w_value=cfg.w_value, value_floor=cfg.value_floor,
                        budget_ratio=cfg.budget_ratio,
                        budget_entries_per_lh=cfg.budget_entries_per_lh,
                        floor_cap_frac=cfg.floor_cap_frac, floor_cap_tokens=cfg.floor_cap_tokens,
                        decode_reserve=args.decode_steps + 1, head_full_frac=args.head_full_frac)
    # host (pinned) and device copies of the inputs
    h_K = torch.from_numpy(np.concatenate([s[2].reshape(-1, cfg.d) for s in seqs])).to(dt).pin_memory()
    h_V = torch.from_numpy(np.concatenate([s[3].reshape(-1, cfg.d) for s in seqs])).to(dt).pin_memory()
    h_Q = torch.from_numpy(np.stack([s[4] for s in seqs])).to(dt).pin_memory()
    bounds = torch.from_numpy(pad_bounds([s[1] for s in seqs], S_max)).to(dev)
    n_slots = torch.tensor([len(s[1]) - 1 for s in seqs], dtype=torch.int32, device=dev)
    K, V, Qp = h_K.to(dev), h_V.to(dev), h_Q.to(dev)
    D = args.decode_steps
    dec = [W.decode_inputs(cfg, t) for t in range(D)]
    h_q = torch.from_numpy(np.stack([x[0] for x in dec])).to(dt).pin_memory()
    h_kn = torch.from_numpy(np.stack([x[1] for x in dec])).to(dt).pin_memory()
    h_vn = torch.from_numpy(np.stack([x[2] for x in dec])).to(dt).pin_memory()
    q_all, kn_all, vn_all = h_q.to(dev), h_kn.to(dev), h_vn.to(dev)
    comp = Compressor(p, [s[0] for s in seqs], device=dev, tree_cuts=args.tree_cuts,
                      salient=args.salient)
    out = torch.empty((D,) + tuple(q_all.shape[1:]), dtype=dt, device=dev)
    h_out = torch.empty(out.shape, dtype=dt).pin_memory()
    stream = torch.cuda.current_stream(dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    rec = {"score": [], "select": [], "pack": [], "decode": []}

    cg = not args.eager_compress                     # compression calls as graph replays

    def step(timed: bool, Kx=K, Vx=V, Qx=Qp):
        marks = [ev() for _ in range(4)] if timed else None
        if timed: marks[0].record(stream)
        comp.score(Kx, Vx, Qx, bounds, n_slots, graph=cg)
        nl = comp.graph_launches if cg else 0
        if timed: marks[1].record(stream)
        comp.select(bounds, n_slots, graph=cg)
        nl += comp.graph_launches if cg else 0
        if timed: marks[2].record(stream)
        comp.merge_pack(Kx, Vx, bounds, n_slots, graph=cg)
        nl += comp.graph_launches if cg else 0
        rec["graph_launches"] = rec.get("graph_launches", 0) + nl
        if timed: marks[3].record(stream)
        # D decode steps: one CUDA graph replay (captured on first use) or D calls
        d0, d1 = ev(), ev()
        d0.record(stream)
        nl = comp.decode_many(q_all, kn_all, vn_all, out, graph=not args.eager_decode)
        d1.record(stream)
        rec["graph_launches"] = rec.get("graph_launches", 0) + (0 if args.eager_decode else nl)
        if timed:
            rec["_pending"] = (marks, [(d0, d1)])

    def harvest():
        marks, dmarks = rec.pop("_pending")
        rec["score"].append(marks[0].elapsed_time(marks[1]))
        rec["select"].append(marks[1].elapsed_time(marks[2]))
        rec["pack"].append(marks[2].elapsed_time(marks[3]))
        rec["decode"].append(sum(a.elapsed_time(b) for a, b in dmarks) / D)

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize(dev)
    err = kvc.kvc_device_error()
    if err != 0:
        raise RuntimeError(f"device error {kvc.kvc_status_string(err)} during warm-up")

    clocks = ClockSampler(dev.index)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = kvc.kvc_launch_count()
    rec["graph_launches"] = 0
    t0, t1 = ev(), ev()
    clocks.begin()
    t0.record(stream)
    step_ms = []
    for _ in range(args.steps):
        s0 = ev(); s0.record(stream)
        step(True)
        s1 = ev(); s1.record(stream)
        torch.cuda.synchronize(dev)
        harvest()
        step_ms.append(s0.elapsed_time(s1))
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    host_launches = kvc.kvc_launch_count() - launches0
    graph_launches = rec["graph_launches"]
    # three-way salient child sets of the last timed compression (other legs
    # rewrite the cut table)
    salient_stat = None
    if args.salient:
        bits = np.unpackbits(comp.cuts[..., 7].cpu().numpy().reshape(-1, 1), axis=1)
        salient_stat = {"isolated_tokens": int(bits.sum()),
                        "depth2_nodes": 4 * sum(len(sq[1]) - 1 for sq in seqs) * cfg.L * cfg.H}
    launches = host_launches + graph_launches
    # the same D decode steps issued one call at a time, for comparison
    eager_ms = None
    if not args.eager_decode and not args.profile:
        comp.select(bounds, n_slots)                      # fresh lengths
        comp.merge_pack(K, V, bounds, n_slots)
        torch.cuda.synchronize(dev)
        x0, x1 = ev(), ev()
        x0.record(stream)
        comp.decode_many(q_all, kn_all, vn_all, out, graph=False)
        x1.record(stream)
        torch.cuda.synchronize(dev)
        eager_ms = x0.elapsed_time(x1) / D
    if world > 1:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    clk = clocks.stop()

    # end to end: pinned host inputs -> device, full path, outputs -> host
    e2e_ms = []
    # batch 1: the cache arrives layer chunk by layer chunk on a copy stream while
    # the chunks already on the device are scored (Compressor.compress_from_host)
    pipelined = cfg.B == 1 and not args.serial_e2e
    copy_stream = torch.cuda.Stream(device=dev)
    # one untimed iteration first: the first host copies of a run pay one-time costs
    # the host link's speed varies from iteration to iteration (pinned-page
    # placement, host load): at least 5 timed iterations, and the median
    for it in range(0 if args.profile else max(5, args.steps) + 1):
        torch.cuda.synchronize(dev)
        a0, a1 = ev(), ev()
        a0.record(stream)
        if pipelined:
            comp.compress_from_host(h_K, h_V, h_Q, K, V, Qp, bounds, n_slots, chunks=8,
                                    copy_stream=copy_stream, graph=cg)
            # the decode inputs follow the cache chunks on the copy stream
            with torch.cuda.stream(copy_stream):
                q_all.copy_(h_q, non_blocking=True); kn_all.copy_(h_kn, non_blocking=True)
                vn_all.copy_(h_vn, non_blocking=True)
            stream.wait_stream(copy_stream)
            comp.decode_many(q_all, kn_all, vn_all, out, graph=not args.eager_decode)
        else:
            q_all.copy_(h_q, non_blocking=True); kn_all.copy_(h_kn, non_blocking=True)
            vn_all.copy_(h_vn, non_blocking=True)
            K.copy_(h_K, non_blocking=True); V.copy_(h_V, non_blocking=True)
            Qp.copy_(h_Q, non_blocking=True)
            step(False)
        h_out.copy_(out, non_blocking=True)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        if it > 0:
            e2e_ms.append(a0.elapsed_time(a1))
    h2d = sum(t.numel() * t.element_size() for t in (h_K, h_V, h_Q, h_q, h_kn, h_vn))
    d2h = h_out.numel() * h_out.element_size()

    # compressed vs full: the same decode kernel on the beta = 1 pack
    full_ms = None if args.profile else full_cache_decode_ms(p, cfg, seqs, K, V, q_all, kn_all,
                                                            vn_all, D, dev, stream)

    creps = None if args.profile else compression_reps(comp, K, V, Qp, bounds, n_slots, cfg,
                                                       sum(s[0] for s in seqs), cg, dev)
    gemm = None if args.profile else scoring_gemm(comp, K, V, Qp, bounds, n_slots, cfg,
                                                  sum(s[0] for s in seqs), measured_peaks()[1],
                                                  dev)
    tree = None
    if args.tree_cuts and not args.profile:
        tree = tree_cuts_leg(comp, K, bounds, n_slots, cfg, sum(s[0] for s in seqs),
                             measured_peaks()[0], dev)
    evict = None
    if (args.evict or not args.profile) and not args.no_evict:
        evict = evict_leg(p, cfg, seqs, K, V, q_all, kn_all, vn_all, D, dev, stream)
        evict["hbm_frac"] = evict["hbm_gbs"] / measured_peaks()[0]
        evict["step_over_compressed_decode"] = evict["ms_per_step"] / statistics.mean(rec["decode"])

    # max over ranks
    ms = total_ms / args.steps
    e2e = statistics.median(e2e_ms) if e2e_ms else float("nan")
    ms, e2e = max_over_ranks([ms, e2e], world, dev)

    tokens = sum(s[0] for s in seqs)
    entries = int(comp.len_lh.sum().cpu()) - cfg.L * cfg.H * cfg.B * 0
    d = cfg.d
    esz = 2 if cfg.dtype == "bf16" else 4
    # algorithmic bytes of one decode launch: every stored entry (K, V, log m) once,
    # the new token appended (K, V, log m, pos) and q / out
    lens_at_pack = comp.len_lh.cpu().numpy().astype(np.int64) - (args.warmup * 0)
    dec_ms = statistics.mean(rec["decode"])
    # entries attended per launch averaged over the D steps: len_pack + t + 1
    packed_entries = int(comp.total.cpu()[0]) - cfg.B * cfg.L * cfg.H * p.decode_reserve
    avg_entries = packed_entries + cfg.B * cfg.L * cfg.H * ((D + 1) / 2.0)
    per_entry = 2 * d * esz + 4
    qo = 2 * cfg.B * cfg.L * cfg.H * cfg.G * d * esz
    dec_bytes = avg_entries * per_entry + cfg.B * cfg.L * cfg.H * (2 * d * esz + 8) + qo
    hbm, tc, src = measured_peaks()
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    score_ms = statistics.mean(rec["score"])
    sel_ms = statistics.mean(rec["select"])
    pack_ms = statistics.mean(rec["pack"])
    score_flops = 2.0 * cfg.B * cfg.L * cfg.H * cfg.G * cfg.P * tokens / cfg.B * d * 3 \
        + 2.0 * cfg.B * cfg.L * cfg.H * cfg.P * tokens / cfg.B * d * 2 * cfg.n_hops
    # merge_pack: every token of a covered slot read once (prototype span or exact
    # copy) with its relevance, the window rows, and every stored entry written
    taken_add = comp.taken[..., 0].bool().cpu().numpy()
    covered = 0
    for b, sq in enumerate(seqs):
        slot_len = np.diff(np.asarray(sq[1], np.int64))
        covered += int((taken_add[b, :, :, :len(slot_len)] * slot_len[None, None, :]).sum())
    stored = packed_entries
    pack_bytes = (covered * (2 * d * esz + 4) + cfg.B * cfg.L * cfg.H * cfg.W * 2 * d * esz
                  + stored * (2 * d * esz + 8))
    # score: K and V read once, features written (its HBM roofline's bytes)
    score_bytes = tokens * cfg.L * cfg.H * (2 * d * esz + 5 * 4)
    dec_tc = p.packed_rows > 0 and cfg.dtype == "bf16" and d == 128   # tensor-core decode
    # the committed DRAM capture covers the full 16K workload's launch (256 steps)
    full_16k = (cfg.name == "mistral16k" and not args.layers and D == 256
                and args.head_full_frac == 0.0 and not args.tree_cuts)
    traffic = kernel_traffic("decode_attn_mistral16k",
                             ["kv_cache_compression_probe_gb300/csrc/kvc_decode.cu",
                              "kv_cache_compression_probe_gb300/csrc/kvc_decode_tc.cu"]) \
        if full_16k else None
    line = {
        "metric": METRIC,
        "value": job_throughput(tokens, world, ms),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded random-walk K/V, planted needles and two-hop chains)",
        "config": {"workload": cfg.name + ": " + cfg.description, "batch": cfg.B,
                   "context": cfg.n, "layers": cfg.L, "kv_heads": cfg.H, "q_heads": cfg.H * cfg.G,
                   "head_dim": d, "budget": cfg.budget_ratio, "window": cfg.W,
                   "decode_steps": D, "l2": "inputs larger than L2 (K+V %.2f GB)" %
                   (2 * tokens * cfg.L * cfg.H * d * esz / 1e9), "parallelism": f"replicas x{world}",
                   "head_full_frac": args.head_full_frac,
                   "trees": ("curvature-chosen (kvc_tree_cuts)" if args.tree_cuts else "midpoint")
                            + (", three-way salient child sets" if args.salient else "")},
        "breakdown_ms": {"score": score_ms, "select": sel_ms, "merge_pack": pack_ms,
                         "decode_per_step": dec_ms, "decode_total": dec_ms * D},
        "compress_tokens_per_s": tokens / ((score_ms + sel_ms + pack_ms) * 1e-3),
        "compression_median_of_reps": creps,
        "decode_gbs": dec_gbs,
        "decode_eager_ms_per_step": eager_ms,
        "decode_full_ms_per_step": full_ms,
        "decode_speedup_vs_full": (full_ms / dec_ms) if full_ms else None,
        "decode_full_note": "full = the same decode call on the beta = 1 pack (every token "
                            "stored exact, ln m = 0); ideal speedup = bytes ratio",
        "decode_bytes_ratio_full": full_bytes_ratio(cfg, seqs, avg_entries, D),
        "roofline": {"kernel": ("decode_tc_kernel (+ plan)" if dec_tc
                                else "decode_chunk_kernel (+ commit)"), "bound": "hbm",
                     "achieved": dec_gbs, "peak": hbm, "unit": "GB/s", "frac": dec_gbs / hbm,
                     "peak_source": src + " hbm_gbs (MEASURED_PEAKS.json)",
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": dec_bytes},
        "merge_pack_roofline": {"bound": "hbm", "achieved": pack_bytes / (pack_ms * 1e-3) / 1e9,
                                "peak": hbm, "unit": "GB/s",
                                "frac": pack_bytes / (pack_ms * 1e-3) / 1e9 / hbm,
                                "algorithmic_bytes": pack_bytes},
        "select_roofline": select_roofline(cfg, seqs, sel_ms, hbm),
        "score_hbm_frac": score_bytes / (score_ms * 1e-3) / 1e9 / hbm,
        "score_tflops": score_flops / (score_ms * 1e-3) / 1e12,
        "score_tc_frac_of_bf16_peak": score_flops / (score_ms * 1e-3) / 1e12 / tc,
        "scoring_gemm": gemm,
        "e2e": {"value": job_throughput(tokens, world, e2e), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e,
                "aggregate": "median of %d iterations" % len(e2e_ms),
                "samples_ms": [round(x, 2) for x in e2e_ms],
                "input_copies": ("8 layer chunks on a copy stream, overlapped with scoring "
                                 "(Compressor.compress_from_host)" if pipelined
                                 else "whole inputs, then the step")},
        "evict_per_step_next_f2": evict,
        "tree_cuts_next_f3": tree,
        "parity": parity_record(cfg.name) if (cfg.name == "mistral16k" and not args.layers
                                              and not args.tree_cuts and not args.salient
                                              and args.head_full_frac == 0.0) else None,
        "salient_next_f3": salient_stat,
        "gpu_launches": launches,
        "gpu_launches_detail": {"issued_by_host": host_launches,
                                "in_graph_replays": graph_launches,
                                "compression_as_graphs": cg,
                                "decode_as_graph": not args.eager_decode},
        "clocks": clk,
    }
    return line


# --------------------------------------------------------------------------- other workloads
def workload_leg(name: str, args, dev, with_cpu: bool):
    """One of the other workloads at full size (long context with its curvature
    partition, the 128x aggressive config, the 64-sequence serving batch):
    inputs generated on the device (synth.device_gen), compression timed as
    the median of `reps` graph replays after warm-ups (kvc_partition included
    for the long-context config), then the workload's decode steps as one
    graph replay.  Returns a record with throughput and roofline fractions."""
    import torch
    from kv_cache_compression_probe_gb300 import kvc
    from kv_cache_compression_probe_gb300.pipeline import Compressor, pad_bounds
    from synth import device_gen as DG
    from synth import workloads as W
    cfg = W.get_config(name)
    L, H, G, P, d, D = cfg.L, cfg.H, cfg.G, cfg.P, cfg.d, cfg.n_decode
    esz = 2
    ns = W.context_lengths(cfg)
    tokens = int(ns.sum())
    bf = torch.bfloat16
    K = torch.empty((tokens * L * H, d), dtype=bf, device=dev)
    V = torch.empty_like(K)
    Qp = torch.empty((cfg.B, L, H * G, P, d), dtype=bf, device=dev)
    t_gen = time.perf_counter()
    ns, planted = DG.fill_workload(cfg, K, V, Qp)
    ctx32 = torch.tensor(ns.astype(np.int32), device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    mk = dict(B=cfg.B, L=L, H=H, G=G, d=d, P=P, W=cfg.W, dtype=kvc.KVC_BF16,
              n_max=int(ns.max()), rope_base=cfg.rope_base, budget_ratio=cfg.budget_ratio,
              budget_entries_per_lh=cfg.budget_entries_per_lh, floor_cap_frac=cfg.floor_cap_frac,
              floor_cap_tokens=cfg.floor_cap_tokens, decode_reserve=D + 1)
    partition = None
    if cfg.slots == "curvature":
        dh = cfg.hidden_dim
        hid = torch.zeros((cfg.B, int(ns.max()), dh), dtype=bf, device=dev)
        for b, n in enumerate(ns):
            hid[b, :int(n)] = DG.hidden_states(cfg, b, int(n), planted[b], dev)
        # a first partition with room for any slot count fixes S_max
        S_room = max(int(n - cfg.W) // 16 + 1 for n in ns)
        p0 = kvc.make_params(S_max=S_room, **mk)
        ws0 = kvc.workspace(kvc.KVC_WS_PARTITION, p0, dev)
        kap = torch.empty((cfg.B, int(ns.max())), dtype=torch.float32, device=dev)
        b0 = torch.zeros((cfg.B, S_room + 1), dtype=torch.int32, device=dev)
        n0 = torch.zeros((cfg.B,), dtype=torch.int32, device=dev)
        kvc.kvc_partition(p0, ctx32, hid, dh, kap, b0, n0, ws0)
        S_max = int(n0.max())
        bounds = torch.zeros((cfg.B, S_max + 1), dtype=torch.int32, device=dev)
        n_slots = torch.zeros_like(n0)

        def partition():
            kvc.kvc_partition(p, ctx32, hid, dh, kap, bounds, n_slots, ws0, stream)
    else:
        S_max = max(len(bd) - 1 for bd in planted)
        bounds = torch.from_numpy(pad_bounds(planted, S_max)).to(dev)
        n_slots = torch.tensor([len(bd) - 1 for bd in planted], dtype=torch.int32, device=dev)
    p = kvc.make_params(S_max=S_max, **mk)
    comp = Compressor(p, [int(n) for n in ns], device=dev)
    torch.cuda.synchronize(dev)
    t_gen = time.perf_counter() - t_gen

    def compress():
        if partition is not None:
            partition()
        comp.compress(K, V, Qp, bounds, n_slots, graph=True)

    for _ in range(2):
        compress()
    torch.cuda.synchronize(dev)
    if kvc.kvc_device_error() != 0:
        raise RuntimeError(f"device error in the {name} workload's compression")
    per = {"partition": [], "score": [], "select": [], "merge_pack": [], "total": []}
    for _ in range(args.workload_reps):
        m = [ev() for _ in range(5)]
        m[0].record(stream)
        if partition is not None:
            partition()
        m[1].record(stream)
        comp.score(K, V, Qp, bounds, n_slots, graph=True)
        m[2].record(stream)
        comp.select(bounds, n_slots, graph=True)
        m[3].record(stream)
        comp.merge_pack(K, V, bounds, n_slots, graph=True)
        m[4].record(stream)
        torch.cuda.synchronize(dev)
        for k, (i, j) in zip(per, ((0, 1), (1, 2), (2, 3), (3, 4), (0, 4))):
            per[k].append(m[i].elapsed_time(m[j]))
    med = {k: statistics.median(v) for k, v in per.items()}
    # decode: D steps as one graph replay over the packed cache (fresh lengths)
    q_all, kn_all, vn_all = DG.decode_inputs(cfg, D, dev)
    out = torch.empty(tuple(q_all.shape), dtype=bf, device=dev)
    len0 = comp.len_lh.clone()
    comp.decode_many(q_all, kn_all, vn_all, out)           # capture + warm
    comp.len_lh.copy_(len0)
    torch.cuda.synchronize(dev)
    e0, e1 = ev(), ev()
    e0.record(stream)
    comp.decode_many(q_all, kn_all, vn_all, out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if kvc.kvc_device_error() != 0:
        raise RuntimeError(f"device error in the {name} workload's decode")
    dec_ms = e0.elapsed_time(e1) / D
    hbm, tc, src = measured_peaks()
    LHB = cfg.B * L * H
    packed_entries = int(comp.total.cpu()[0]) - LHB * p.decode_reserve
    avg_entries = packed_entries + LHB * ((D + 1) / 2.0)
    dec_bytes = (avg_entries * (2 * d * esz + 4) + LHB * (2 * d * esz + 8)
                 + 2 * LHB * G * d * esz)
    taken_add = comp.taken[..., 0].bool().cpu().numpy()
    bnd = bounds.cpu().numpy().astype(np.int64)
    nsl = n_slots.cpu().numpy()
    covered = 0
    for b in range(cfg.B):
        slot_len = np.diff(bnd[b, :int(nsl[b]) + 1])
        covered += int((taken_add[b, :, :, :len(slot_len)] * slot_len[None, None, :]).sum())
    pack_bytes = (covered * (2 * d * esz + 4) + LHB * cfg.W * 2 * d * esz
                  + packed_entries * (2 * d * esz + 8))
    score_flops = 2.0 * L * H * G * P * tokens * d * 3 + 2.0 * L * H * P * tokens * d * 2 * cfg.n_hops
    comp_ms = med["total"]
    rec = {
        "workload": cfg.name + ": " + cfg.description, "batch": cfg.B,
        "context": int(ns.max()) if cfg.B == 1 else [int(ns.min()), int(ns.max())],
        "kv_tokens": tokens, "decode_steps": D,
        "ms_per_step": comp_ms + dec_ms * D,
        "kv_tokens_per_s": tokens / ((comp_ms + dec_ms * D) * 1e-3),
        "compression_median_ms": med, "compression_reps": args.workload_reps,
        "compress_kv_tokens_per_s": tokens / (comp_ms * 1e-3),
        "compress_lh_entries_per_s": tokens * L * H / (comp_ms * 1e-3),
        "decode_ms_per_step": dec_ms,
        "decode_roofline": {"bound": "hbm", "achieved": dec_bytes / (dec_ms * 1e-3) / 1e9,
                            "peak": hbm, "unit": "GB/s",
                            "frac": dec_bytes / (dec_ms * 1e-3) / 1e9 / hbm,
                            "algorithmic_bytes_per_launch": dec_bytes},
        "merge_pack_roofline": {"bound": "hbm",
                                "achieved": pack_bytes / (med["merge_pack"] * 1e-3) / 1e9,
                                "peak": hbm, "unit": "GB/s",
                                "frac": pack_bytes / (med["merge_pack"] * 1e-3) / 1e9 / hbm,
                                "algorithmic_bytes": pack_bytes},
        "score_tc_frac_of_bf16_peak": score_flops / (med["score"] * 1e-3) / 1e12 / tc,
        "packed_entries": packed_entries,
        "compression_ratio": tokens * L * H / packed_entries,
        "inputs": "generated on the device (synth.device_gen), %.1f s; K+V %.1f GB" %
                  (t_gen, 2 * tokens * L * H * d * esz / 1e9),
        "peaks": src + " (MEASURED_PEAKS.json)",
    }
    del comp, K, V, Qp, q_all, kn_all, vn_all, out
    torch.cuda.empty_cache()
    if with_cpu:
        rec["cpu_baseline"] = cpu_baseline(cfg, D, single_process=False)
    return rec


def tiny_leg(args, dev, with_cpu: bool):
    """The tiny config (fp32, d = 64: the SIMT scoring, pack and decode kernels):
    the whole workload compressed and decoded, timed like the other legs, and
    the oracle on one process over the whole workload beside it."""
    import torch
    from kv_cache_compression_probe_gb300 import kvc
    from kv_cache_compression_probe_gb300.pipeline import Compressor, pad_bounds
    from synth import workloads as W
    cfg = W.get_config("tiny")
    wl = W.make_workload(cfg)
    D = cfg.n_decode
    S_max = max(len(s.slot_bounds) - 1 for s in wl.seqs)
    p = kvc.make_params(B=cfg.B, L=cfg.L, H=cfg.H, G=cfg.G, d=cfg.d, P=cfg.P, W=cfg.W,
                        dtype=kvc.KVC_F32, n_max=max(s.n for s in wl.seqs), S_max=S_max,
                        rope_base=cfg.rope_base, budget_ratio=cfg.budget_ratio,
                        budget_entries_per_lh=cfg.budget_entries_per_lh,
                        floor_cap_frac=cfg.floor_cap_frac, floor_cap_tokens=cfg.floor_cap_tokens,
                        decode_reserve=D + 1)
    f32 = torch.float32
    K = torch.from_numpy(np.concatenate([s.K.reshape(-1, cfg.d) for s in wl.seqs])).to(dev, f32)
    V = torch.from_numpy(np.concatenate([s.V.reshape(-1, cfg.d) for s in wl.seqs])).to(dev, f32)
    Qp = torch.from_numpy(np.stack([s.Qp for s in wl.seqs])).to(dev, f32)
    bounds = torch.from_numpy(pad_bounds([s.slot_bounds for s in wl.seqs], S_max)).to(dev)
    n_slots = torch.tensor([len(s.slot_bounds) - 1 for s in wl.seqs], dtype=torch.int32,
                           device=dev)
    comp = Compressor(p, [s.n for s in wl.seqs], device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        comp.compress(K, V, Qp, bounds, n_slots, graph=True)
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(max(20, args.workload_reps)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        comp.compress(K, V, Qp, bounds, n_slots, graph=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    comp_ms = statistics.median(times)
    dec = [W.decode_inputs(cfg, t) for t in range(D)]
    q_all = torch.from_numpy(np.stack([x[0] for x in dec])).to(dev, f32)
    kn_all = torch.from_numpy(np.stack([x[1] for x in dec])).to(dev, f32)
    vn_all = torch.from_numpy(np.stack([x[2] for x in dec])).to(dev, f32)
    out = torch.empty(tuple(q_all.shape), dtype=f32, device=dev)
    len0 = comp.len_lh.clone()
    comp.decode_many(q_all, kn_all, vn_all, out)
    comp.len_lh.copy_(len0)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    comp.decode_many(q_all, kn_all, vn_all, out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if kvc.kvc_device_error() != 0:
        raise RuntimeError("device error in the tiny workload")
    dec_ms = e0.elapsed_time(e1) / D
    tokens = sum(s.n for s in wl.seqs)
    rec = {"workload": cfg.name + ": " + cfg.description, "kv_tokens": tokens, "decode_steps": D,
           "dtype": "f32", "paths": "SIMT scoring, pack and decode (fp32, d = 64)",
           "compression_median_ms": comp_ms, "compression_reps": len(times),
           "decode_ms_per_step": dec_ms, "ms_per_step": comp_ms + dec_ms * D,
           "kv_tokens_per_s": tokens / ((comp_ms + dec_ms * D) * 1e-3),
           "note": "a parity-sized case: launch latency bounds every call"}
    if with_cpu:
        secs, toks = oracle_sample(cfg, [(l, h) for l in range(cfg.L) for h in range(cfg.H)], D)
        rec["cpu_baseline"] = {"value": toks / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
                               "sample": "the whole workload, one process", "seconds": secs}
    return rec


# --------------------------------------------------------------------------- oracle (CPU)
def oracle_sample(cfg, heads, decode_steps):
    """The float64 oracle over a bounded sample: `heads` (layer, KV head) pairs of
    sequence 0 scored, selected with the pooled budget scaled to the sample,
    packed and decoded.  Returns (seconds, KV tokens covered)."""
    import oracle as O
    from synth import workloads as W
    n = int(W.context_lengths(cfg)[0])
    bounds = W.planted_bounds(cfg, 0, n)
    counts = W._needle_counts(cfg, 0, n)
    data = {}
    for (l, h) in heads:
        data[(l, h)] = W.gen_head(cfg, 0, l, h, n, bounds, int(counts[l * cfg.H + h]))
    t0 = time.perf_counter()
    S = len(bounds) - 1
    util = np.zeros((1, len(heads), S, 16)); cost = np.zeros((1, len(heads), S, 16), np.int64)
    r = np.zeros((1, len(heads), n))
    for k, (l, h) in enumerate(heads):
        K, V, Q, _ = data[(l, h)]
        res = O.score_and_value_head(K, V, Q, n, cfg.P, bounds, 1.0, base=cfg.rope_base)
        util[0, k], cost[0, k], r[0, k] = res.util, res.cost, res.r
    sel = O.select_sequence(util, cost, r, np.ones((1, len(heads))), bounds, n, cfg.W,
                            cfg.budget_ratio, cfg.budget_entries_per_lh, cfg.floor_cap_frac,
                            cfg.floor_cap_tokens)
    rng = np.random.default_rng(0)
    for k, (l, h) in enumerate(heads):
        K, V, Q, _ = data[(l, h)]
        Kp, Vp, lm, _ = O.pack_head(K, V, r[0, k], bounds, sel.taken[0, k], n, cfg.W,
                                    cfg.rope_base, cfg.value_floor)
        for t in range(decode_steps):
            q = rng.standard_normal((cfg.G, cfg.d)); kn = rng.standard_normal(cfg.d)
            vn = rng.standard_normal(cfg.d)
            _, Kp, Vp, lm = O.decode_step_head(q, kn, vn, Kp, Vp, lm)
    dt = time.perf_counter() - t0
    return dt, n * len(heads) / (cfg.L * cfg.H)


_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _oracle_head_job(job):
    """One (layer, KV head) of the oracle sample, in a worker process: the head is
    generated untimed, then phase 0 (score, hops, utilities) or phase 1 (pack
    and decode steps) is timed."""
    cfg, l, h, phase, payload = job
    import oracle as O
    from synth import workloads as W
    n = int(W.context_lengths(cfg)[0])
    bounds = W.planted_bounds(cfg, 0, n)
    counts = W._needle_counts(cfg, 0, n)
    K, V, Q, _ = W.gen_head(cfg, 0, l, h, n, bounds, int(counts[l * cfg.H + h]))
    t0 = time.perf_counter()
    if phase == 0:
        res = O.score_and_value_head(K, V, Q, n, cfg.P, bounds, 1.0, base=cfg.rope_base)
        out = (res.util, res.cost, res.r)
    else:
        r, taken, steps, seed = payload
        Kp, Vp, lm, _ = O.pack_head(K, V, r, bounds, taken, n, cfg.W, cfg.rope_base,
                                    cfg.value_floor)
        rng = np.random.default_rng(seed)
        for _ in range(steps):
            q = rng.standard_normal((cfg.G, cfg.d)); kn = rng.standard_normal(cfg.d)
            vn = rng.standard_normal(cfg.d)
            _, Kp, Vp, lm = O.decode_step_head(q, kn, vn, Kp, Vp, lm)
        out = None
    return time.perf_counter() - t0, out


def oracle_sample_parallel(cfg, heads, decode_steps, workers):
    """The oracle sample of `oracle_sample` with its per-head phases spread over a
    spawn process pool (one head per worker); wall = slowest scoring worker +
    the pooled selection + slowest pack/decode worker."""
    import oracle as O
    from synth import workloads as W
    n = int(W.context_lengths(cfg)[0])
    bounds = W.planted_bounds(cfg, 0, n)
    ctx = mp.get_context("spawn")
    # one BLAS thread per worker (spawned children read these at start)
    saved = {k: os.environ.get(k) for k in _BLAS_VARS}
    os.environ.update({k: "1" for k in _BLAS_VARS})
    try:
        pool = ctx.Pool(workers)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    with pool:
        ph0 = pool.map(_oracle_head_job, [(cfg, l, h, 0, None) for (l, h) in heads])
        t0 = time.perf_counter()
        util = np.stack([o[1][0] for o in ph0])[None]
        cost = np.stack([o[1][1] for o in ph0])[None]
        r = np.stack([o[1][2] for o in ph0])[None]
        sel = O.select_sequence(util, cost, r, np.ones((1, len(heads))), bounds, n, cfg.W,
                                cfg.budget_ratio, cfg.budget_entries_per_lh, cfg.floor_cap_frac,
                                cfg.floor_cap_tokens)
        t_sel = time.perf_counter() - t0
        ph1 = pool.map(_oracle_head_job, [(cfg, l, h, 1, (r[0, k], sel.taken[0, k], decode_steps, k))
                                          for k, (l, h) in enumerate(heads)])
    wall = max(o[0] for o in ph0) + t_sel + max(o[0] for o in ph1)
    return wall, n * len(heads) / (cfg.L * cfg.H)


def cpu_baseline(cfg, decode_steps, n_heads=4, single_process=True):
    """The oracle on the host cores: all cores (one (layer, KV head) per worker)
    as the reported baseline, and (single_process) one process on `n_heads`
    heads beside it."""
    workers = max(1, min(os.cpu_count() or 1, 16, cfg.L * cfg.H))
    heads = [(k % cfg.L, k // cfg.L) for k in range(workers)]
    pwall, ptoks = oracle_sample_parallel(cfg, heads, decode_steps, workers)
    n_heads = min(n_heads, cfg.L * cfg.H)
    single = None
    if single_process:
        secs, toks = oracle_sample(cfg, [(k % cfg.L, k // cfg.L) for k in range(n_heads)],
                                   decode_steps)
        single = {"value": toks / secs, "cores": os.cpu_count(), "heads": n_heads,
                  "seconds": secs, "note": "one process; numpy's BLAS threads use every core"}
    return {"value": ptoks / pwall, "unit": UNIT, "cores": workers, "kind": "oracle",
            "sample": f"{workers} of {cfg.L * cfg.H} (layer, KV head) pairs of the {cfg.n}-token "
                      f"sequence, one per worker process: score+hops+utilities, floor+auction "
                      f"with the budget pooled over the sample, pack, {decode_steps} decode "
                      f"steps; float64 numpy; wall {pwall:.1f} s (host reports "
                      f"{os.cpu_count()} cores)",
            "seconds": pwall,
            "single_process": single}


def run_reference(args, cfg, rank, world):
    """The oracle as the reference arm: each step is the all-cores oracle sample
    (one (layer, KV head) per worker process) on a fresh set of heads."""
    if rank != 0:
        return None
    workers = max(1, min(os.cpu_count() or 1, 16, cfg.L * cfg.H))
    t_all = time.perf_counter()
    pairs = [(k % cfg.L, (k // cfg.L) % cfg.H) for k in range(cfg.L * cfg.H)]
    for w in range(args.warmup):
        oracle_sample_parallel(cfg, pairs[:1], 2, 1)
    vals = []
    for s in range(args.steps):
        heads = [pairs[(s * workers + k) % len(pairs)] for k in range(workers)]
        vals.append(oracle_sample_parallel(cfg, heads, args.decode_steps, workers))
    secs = sum(v[0] for v in vals)
    toks = sum(v[1] for v in vals)
    value = toks / secs
    sample = (f"per step {workers} (layer, KV head) pairs of the {cfg.n}-token sequence, one per "
              f"worker process (score, hops, utilities, pooled select, pack, "
              f"{args.decode_steps} decode steps); float64 numpy")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cfg.name + ": " + cfg.description},
            "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": workers,
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t_all}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="mistral16k")
    ap.add_argument("--decode-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the layer count (small profiling cases)")
    ap.add_argument("--head-full-frac", type=float, default=0.0,
                    help="head-level hybrid: fraction of heads that keep the full cache")
    ap.add_argument("--tree-cuts", action="store_true",
                    help="curvature-chosen prototype trees (kvc_tree_cuts) instead of midpoint trees")
    ap.add_argument("--salient", action="store_true",
                    help="three-way salient-token child sets in the prototype trees")
    ap.add_argument("--evict", action="store_true",
                    help="time the per-step top-B eviction (DistillCache) leg also under --profile")
    ap.add_argument("--no-evict", action="store_true",
                    help="skip the per-step top-B eviction leg (on by default)")
    ap.add_argument("--serial-e2e", action="store_true",
                    help="end-to-end leg: copy all inputs before the step instead of overlapping")
    ap.add_argument("--eager-compress", action="store_true",
                    help="issue the compression calls directly instead of as CUDA graph replays")
    ap.add_argument("--eager-decode", action="store_true",
                    help="issue the decode steps one call at a time instead of one CUDA graph")
    ap.add_argument("--workloads", default="tiny,long,aggressive,serving",
                    help="other workloads timed after the headline line (comma list; '' = none)")
    ap.add_argument("--workload-reps", type=int, default=20,
                    help="compression repetitions per other workload (median)")
    ap.add_argument("--profile", action="store_true",
                    help="profiling run: no warm-up, one step, no CPU baseline, no e2e leg")
    args = ap.parse_args()
    from synth import workloads as W
    cfg = W.get_config(args.config)
    if args.layers:
        cfg = cfg.replace(L=args.layers)
    if args.profile:
        args.steps, args.warmup, args.no_cpu_baseline = 1, 0, True
    if args.decode_steps is None:
        args.decode_steps = cfg.n_decode
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        line = run_reference(args, cfg, rank, world)
        if line is not None:
            print(json.dumps(line))
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, args.decode_steps)
    line = run_gpu(args, cfg, rank, world)
    if rank == 0:
        line["cpu_baseline"] = cpu
        names = [w for w in args.workloads.split(",") if w] if world == 1 and not args.profile \
            and not args.layers else []
        if names:
            import torch
            torch.cuda.empty_cache()
            dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
            line["other_workloads"] = {w: (tiny_leg(args, dev, not args.no_cpu_baseline)
                                           if w == "tiny" else
                                           workload_leg(w, args, dev, not args.no_cpu_baseline))
                                       for w in names}
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
