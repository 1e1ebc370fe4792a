"""Device-buffer owner for the compression + decode path.

`Compressor` allocates (with torch) every output and workspace the four C-ABI
calls need, builds the RoPE tables with `kvc_rope_table`, and runs
kvc_score -> kvc_select -> kvc_merge_pack and kvc_decode_attn steps.  It only
allocates and marshals; all arithmetic runs in libkvc's kernels.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np
import torch

from . import kvc

TORCH_DT = {kvc.KVC_BF16: torch.bfloat16, kvc.KVC_F32: torch.float32}


def packed_capacity(p: kvc.kvc_params, ctx_len: Sequence[int]) -> int:
    """Rows the packed cache needs at most: every sequence's budget (at least its
    window) plus the decode reserve of every (b, l, h)."""
    LH = p.L * p.H
    rows = 0
    for n in ctx_len:
        per = p.budget_entries_per_lh if p.budget_entries_per_lh > 0 else math.floor(p.budget_ratio * n)
        rows += max(per, p.W) * LH + LH * p.decode_reserve
    return int(rows)


# ---------------------------------------------------------------- packed-cache files
PACKED_FORMAT = 1
_PACKED_ARRAYS = ("Kp", "Vp", "logm", "pos", "len_lh", "cap_lh", "off_lh")


def write_packed(path: str, p: kvc.kvc_params, tensors: dict) -> None:
    """Writes a packed cache to an .npz file: the parameter block's scalar
    fields, and Kp, Vp, logm, pos (the first sum(cap_lh) rows, i.e. every
    (b, l, h)'s entries and its decode reserve) with len_lh, cap_lh and
    off_lh.  bf16 rows are stored as their uint16 bit patterns, so a reload is
    bit for bit.  Tensors may live on any device."""
    rows = int(tensors["cap_lh"].to(torch.int64).sum())
    out = {"format": np.int64(PACKED_FORMAT)}
    for name, ctype in p._fields_:
        if name == "tree_cuts":                      # a pointer: not part of the cache
            continue
        out["param_" + name] = np.asarray(getattr(p, name))
    for name in _PACKED_ARRAYS:
        t = tensors[name].detach()
        if name in ("Kp", "Vp", "logm", "pos"):
            t = t[:rows]
        t = t.cpu().contiguous()
        if t.dtype == torch.bfloat16:
            out[name + "_bf16bits"] = t.view(torch.int16).numpy()
        else:
            out[name] = t.numpy()
    np.savez(path, **out)


def read_packed(path: str):
    """(params dict, tensors dict on the CPU) of a file written by write_packed."""
    with np.load(path) as z:
        if int(z["format"]) != PACKED_FORMAT:
            raise ValueError(f"{path}: packed-cache format {int(z['format'])}, expected {PACKED_FORMAT}")
        params = {k[len("param_"):]: z[k].item() for k in z.files if k.startswith("param_")}
        tensors = {}
        for name in _PACKED_ARRAYS:
            if name + "_bf16bits" in z.files:
                tensors[name] = torch.from_numpy(z[name + "_bf16bits"].copy()).view(torch.bfloat16)
            else:
                tensors[name] = torch.from_numpy(z[name].copy())
    return params, tensors


class Compressor:
    def __init__(self, p: kvc.kvc_params, ctx_len: Sequence[int], device="cuda",
                 tensor_cores: bool = True, tree_cuts: bool = False, salient: bool = False):
        """tree_cuts=True: every scoring call first runs kvc_tree_cuts, and
        scoring, selection and packing use those curvature-chosen trees
        (p.tree_cuts points at this object's cut table); otherwise the
        midpoint trees.  salient=True: the depth-2 nodes may isolate their most
        relevant token in a three-way child set (kvc_params.salient_extract);
        kvc_score records the choice in the cut table, which is reset to the
        binary cuts (kvc_tree_cuts, or zeros for midpoint trees) before every
        scoring call."""
        self.p = p
        self.device = device
        self.ctx_host = [int(n) for n in ctx_len]
        # the tensor-core scoring passes need the exact extent of K
        p.total_ctx = sum(self.ctx_host) if tensor_cores else 0
        assert len(self.ctx_host) == p.B and max(self.ctx_host) <= p.n_max
        B, L, H, R, S = p.B, p.L, p.H, p.G * p.P, p.S_max
        rows = sum(L * H * n for n in self.ctx_host)
        dt = TORCH_DT[p.dtype]
        f32, i32 = torch.float32, torch.int32
        z = dict(device=device)
        self.ctx_len = torch.tensor(self.ctx_host, dtype=i32, **z)
        n_half = 2 * p.n_max
        self.rope_cos = torch.empty((n_half, p.d // 2), dtype=f32, **z)
        self.rope_sin = torch.empty((n_half, p.d // 2), dtype=f32, **z)
        kvc.kvc_rope_table(p.d, p.rope_base, n_half, self.rope_cos, self.rope_sin)
        self.lse = torch.empty((B, L, H, R), dtype=f32, **z)
        self.feats = torch.empty((rows, 5), dtype=f32, **z)
        self.relevance = torch.empty((rows,), dtype=f32, **z)
        self.op_util = torch.empty((B, L, H, S, 16), dtype=f32, **z)
        self.op_cost = torch.empty((B, L, H, S, 16), dtype=i32, **z)
        self.taken = torch.empty((B, L, H, S, 16), dtype=torch.uint8, **z)
        self.len_lh = torch.empty((B, L, H), dtype=i32, **z)
        self.cap_lh = torch.empty((B, L, H), dtype=i32, **z)
        self.off_lh = torch.empty((B, L, H), dtype=torch.int64, **z)
        self.total = torch.empty((1,), dtype=torch.int64, **z)
        cap = packed_capacity(p, self.ctx_host)
        # the tensor-core decode needs the extent of the packed cache
        p.packed_rows = cap if tensor_cores else 0
        self.Kp = torch.empty((cap, p.d), dtype=dt, **z)
        self.Vp = torch.empty((cap, p.d), dtype=dt, **z)
        self.logm = torch.empty((cap,), dtype=f32, **z)
        self.pos = torch.empty((cap,), dtype=f32, **z)
        self.ws_score = kvc.workspace(kvc.KVC_WS_SCORE, p, device)
        self.ws_select = kvc.workspace(kvc.KVC_WS_SELECT, p, device)
        self.ws_pack = kvc.workspace(kvc.KVC_WS_PACK, p, device)
        self.ws_decode = kvc.workspace(kvc.KVC_WS_DECODE, p, device, zero=True)
        self.tree_kappa = torch.empty((rows,), dtype=f32, **z) if tree_cuts else None
        self.curvature_trees = bool(tree_cuts)
        self.cuts = (torch.zeros((B, L, H, S, 8), dtype=torch.uint8, **z)
                     if (tree_cuts or salient) else None)
        p.tree_cuts = self.cuts.data_ptr() if self.cuts is not None else None
        p.salient_extract = 1 if salient else 0
        self._graphs = {}

    # ---------------------------------------------------------------- calls
    # With graph=True a call is captured into a CUDA graph once per set of
    # buffers and replayed on the current stream (the library launches many
    # small kernels per call); the last replay's kernel count is kept in
    # `graph_launches`.
    def _graphed(self, key, fn):
        g = self._graphs.get(key)
        if g is None:
            dev = self.Kp.device
            kvc.kvc_device_error()                   # error-word lookup outside capture
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            graph = torch.cuda.CUDAGraph()
            n0 = kvc.kvc_launch_count()
            with torch.cuda.graph(graph, stream=side):
                fn(side)
            torch.cuda.current_stream(dev).wait_stream(side)
            g = (graph, kvc.kvc_launch_count() - n0)
            self._graphs[key] = g
        g[0].replay()
        self.graph_launches = g[1]

    @staticmethod
    def _key(name, *tensors):
        return (name,) + tuple(t.data_ptr() if t is not None else 0 for t in tensors)

    def score(self, K, V, Qp, slot_bounds, n_slots, head_sens=None, stream=None, graph=False):
        def run(st):
            if self.curvature_trees:
                kvc.kvc_tree_cuts(self.p, self.ctx_len, K, self.rope_cos, self.rope_sin,
                                  slot_bounds, n_slots, self.tree_kappa, self.cuts, st)
            elif self.cuts is not None:              # midpoint trees: an all-zero table
                with torch.cuda.stream(torch.cuda.current_stream() if st is None else st):
                    self.cuts.zero_()
            kvc.kvc_score(self.p, self.ctx_len, K, V, Qp, self.rope_cos, self.rope_sin,
                          slot_bounds, n_slots, head_sens, self.lse, self.feats, self.relevance,
                          self.op_util, self.op_cost, self.ws_score, st)
        if graph:
            self._graphed(self._key("score", K, V, Qp, slot_bounds, n_slots, head_sens), run)
        else:
            run(stream)

    def select(self, slot_bounds, n_slots, head_sens=None, op_util=None, relevance=None,
               stream=None, graph=False):
        rel = self.relevance if relevance is None else relevance
        util = self.op_util if op_util is None else op_util

        def run(st):
            kvc.kvc_select(self.p, self.ctx_len, slot_bounds, n_slots, rel, head_sens, util,
                           self.op_cost, self.taken, self.len_lh, self.cap_lh, self.off_lh,
                           self.total, self.ws_select, st)
        if graph:
            self._graphed(self._key("select", slot_bounds, n_slots, head_sens, rel, util), run)
        else:
            run(stream)

    def merge_pack(self, K, V, slot_bounds, n_slots, taken=None, stream=None, graph=False):
        tk = self.taken if taken is None else taken

        def run(st):
            kvc.kvc_merge_pack(self.p, self.ctx_len, K, V, self.relevance, self.rope_cos,
                               self.rope_sin, slot_bounds, n_slots, tk, self.len_lh, self.off_lh,
                               self.Kp, self.Vp, self.logm, self.pos, self.ws_pack, st)
        if graph:
            self._graphed(self._key("pack", K, V, slot_bounds, n_slots, tk), run)
        else:
            run(stream)

    def compress(self, K, V, Qp, slot_bounds, n_slots, head_sens=None, stream=None, graph=False):
        self.score(K, V, Qp, slot_bounds, n_slots, head_sens, stream, graph)
        self.select(slot_bounds, n_slots, head_sens, stream=stream, graph=graph)
        self.merge_pack(K, V, slot_bounds, n_slots, stream=stream, graph=graph)

    def compress_from_host(self, h_K, h_V, h_Qp, K, V, Qp, slot_bounds, n_slots,
                           head_sens=None, chunks: int = 4, copy_stream=None, graph=False):
        """Batch 1, inputs in pinned host memory: copies K, V and the probes into the
        device buffers K, V, Qp one layer chunk at a time on `copy_stream` while the
        chunks already on the device are scored on the current stream (scoring has
        no coupling across layers; the budget couples them only in select), then
        selects and packs (as graph replays with graph=True).  The first chunk is
        about half the size of the others, so less of the copy is exposed.  Same
        results as copying everything, then compress().  Copies the caller queues
        on `copy_stream` afterwards run behind the chunks."""
        p = self.p
        if p.B != 1:
            raise ValueError("compress_from_host copies layer chunks of one sequence")
        L, H, n = p.L, p.H, self.ctx_host[0]
        dev = K.device
        cur = torch.cuda.current_stream(dev)
        cs = copy_stream if copy_stream is not None else torch.cuda.Stream(device=dev)
        cs.wait_stream(cur)                          # the buffers are free to overwrite
        # a small first chunk, so scoring starts early; the rest in equal parts
        chunks = max(1, min(chunks, L))
        first = max(1, -(-L // (2 * chunks))) if chunks > 1 else L
        cuts = [0] + [first + round(c * (L - first) / (chunks - 1)) for c in range(chunks)] \
            if chunks > 1 else [0, L]
        events = []
        for c in range(chunks):
            l0, l1 = cuts[c], cuts[c + 1]
            r0, r1 = l0 * H * n, l1 * H * n
            with torch.cuda.stream(cs):
                K[r0:r1].copy_(h_K[r0:r1], non_blocking=True)
                V[r0:r1].copy_(h_V[r0:r1], non_blocking=True)
                Qp[:, l0:l1].copy_(h_Qp[:, l0:l1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
            events.append(ev)
        for c in range(chunks):
            l0, l1 = cuts[c], cuts[c + 1]
            if l1 == l0:
                continue
            r0, r1 = l0 * H * n, l1 * H * n
            cur.wait_event(events[c])
            pc = kvc.kvc_params.from_buffer_copy(p)
            pc.L = l1 - l0
            if self.cuts is not None and not self.curvature_trees:
                pc.tree_cuts = self.cuts[:, l0:l1].data_ptr()
                with torch.cuda.stream(cur):
                    self.cuts[:, l0:l1].zero_()
            if self.curvature_trees:
                pc.tree_cuts = self.cuts[:, l0:l1].data_ptr()
                kvc.kvc_tree_cuts(pc, self.ctx_len, K[r0:r1], self.rope_cos, self.rope_sin,
                                  slot_bounds, n_slots, self.tree_kappa[r0:r1],
                                  self.cuts[:, l0:l1], cur)
            kvc.kvc_score(pc, self.ctx_len, K[r0:r1], V[r0:r1], Qp[:, l0:l1], self.rope_cos,
                          self.rope_sin, slot_bounds, n_slots,
                          None if head_sens is None else head_sens[l0:l1], self.lse[:, l0:l1],
                          self.feats[r0:r1], self.relevance[r0:r1], self.op_util[:, l0:l1],
                          self.op_cost[:, l0:l1], self.ws_score, cur)
        self.select(slot_bounds, n_slots, head_sens, graph=graph)
        self.merge_pack(K, V, slot_bounds, n_slots, graph=graph)

    # ---------------------------------------------------------------- packed-cache files
    def save_packed(self, path: str) -> None:
        """Writes this object's packed cache (after kvc_merge_pack and any
        decode steps) to an .npz file (write_packed)."""
        torch.cuda.synchronize(self.Kp.device)
        write_packed(path, self.p, {n: getattr(self, n) for n in _PACKED_ARRAYS})

    def load_packed(self, path: str) -> None:
        """Replaces this object's packed cache with a saved one, so decoding
        resumes where the saving process stopped.  The file's shape fields
        (B, L, H, G, d, dtype) must match this object's and its rows must fit
        the packed buffers."""
        params, t = read_packed(path)
        for k in ("B", "L", "H", "G", "d", "dtype"):
            if params[k] != getattr(self.p, k):
                raise ValueError(f"{path}: {k} = {params[k]}, this cache has {getattr(self.p, k)}")
        rows = t["Kp"].shape[0]
        if rows > self.Kp.shape[0]:
            raise ValueError(f"{path}: {rows} rows, the packed buffers hold {self.Kp.shape[0]}")
        for n in ("Kp", "Vp", "logm", "pos"):
            getattr(self, n)[:rows].copy_(t[n])
        for n in ("len_lh", "cap_lh", "off_lh"):
            getattr(self, n).copy_(t[n].view(getattr(self, n).shape))
        self.ws_decode.zero_()                       # fresh arrival counters
        torch.cuda.synchronize(self.Kp.device)

    def decode(self, q, k_new, v_new, out, pos_new=None, stream=None):
        kvc.kvc_decode_attn(self.p, q, k_new, v_new, pos_new, self.Kp, self.Vp, self.logm,
                            self.pos, self.len_lh, self.cap_lh, self.off_lh, out, self.ws_decode,
                            stream)

    def decode_many(self, q_all, kn_all, vn_all, out_all, pos_all=None, graph=True):
        """T = q_all.shape[0] decode steps back to back (step t reads q_all[t],
        kn_all[t], vn_all[t] and writes out_all[t]).  With graph=True the T calls
        are captured once per set of buffers into a CUDA graph and replayed, so
        the steps pay no per-launch host cost; the cache lengths advance on the
        device either way.  Returns the number of library kernels launched."""
        if not graph:
            n0 = kvc.kvc_launch_count()
            for t in range(q_all.shape[0]):
                self.decode(q_all[t], kn_all[t], vn_all[t], out_all[t],
                            None if pos_all is None else pos_all[t])
            return kvc.kvc_launch_count() - n0
        key = tuple(x.data_ptr() if x is not None else 0
                    for x in (q_all, kn_all, vn_all, out_all, pos_all)) + (q_all.shape[0],)
        g = self._graphs.get(key)
        if g is None:
            g = DecodeGraph(self.p, q_all, kn_all, vn_all, pos_all, self.Kp, self.Vp, self.logm,
                            self.pos, self.len_lh, self.cap_lh, self.off_lh, out_all,
                            self.ws_decode)
            self._graphs[key] = g
        g.replay()
        return g.launches


class DecodeGraph:
    """T kvc_decode_attn calls captured into one CUDA graph.

    The buffers are baked into the graph: replay() runs the T steps on the
    current stream over whatever the buffers then hold.  The library's one-time
    device lookups run before capture (a kvc_device_error call)."""

    def __init__(self, p, q_all, kn_all, vn_all, pos_all, Kp, Vp, logm, pos, len_lh, cap_lh,
                 off_lh, out_all, ws):
        dev = q_all.device
        kvc.kvc_device_error()                       # error-word lookup outside capture
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        self.graph = torch.cuda.CUDAGraph()
        n0 = kvc.kvc_launch_count()
        with torch.cuda.graph(self.graph, stream=side):
            for t in range(q_all.shape[0]):
                kvc.kvc_decode_attn(p, q_all[t], kn_all[t], vn_all[t],
                                    None if pos_all is None else pos_all[t], Kp, Vp, logm, pos,
                                    len_lh, cap_lh, off_lh, out_all[t], ws, side)
        self.launches = kvc.kvc_launch_count() - n0
        torch.cuda.current_stream(dev).wait_stream(side)
        # keep the baked buffers alive as long as the graph
        self._keep = (q_all, kn_all, vn_all, pos_all, Kp, Vp, logm, pos, len_lh, cap_lh, off_lh,
                      out_all, ws)

    def replay(self):
        self.graph.replay()


class EvictingCache:
    """NEXT f2: DistillCache per-step top-B eviction with the heuristic score
    (DistillCache Algorithm 1; the score is the attention feature alpha of 3.1.1).

    Every (b, l, h) holds the same tokens of sequence b (its prompt to start
    with) in the same rows of its `cap`-row range at off_lh = (b*L*H + l*H + h)
    * cap.  One step is kvc_decode_attn_lse (append + attend, base-2 LSE per
    query head and, with scores=True, every entry's score) -> kvc_token_alpha
    (from those scores, else recomputed from K) -> kvc_evict_topb (in place);
    every entry keeps log m = 0.  The class only allocates and marshals.
    """

    def __init__(self, p: kvc.kvc_params, K, V, ctx_len: Sequence[int], reserve: int,
                 ratio: float, b_min: int, tensor_cores: bool = True, scores: bool = True):
        B, L, H = p.B, p.L, p.H
        assert K.shape[:3] == (B, L, H) and K.shape == V.shape
        dev = K.device
        self.p, self.ratio, self.b_min = p, float(ratio), int(b_min)
        self.ctx = [int(n) for n in ctx_len]
        self.cap = max(self.ctx) + int(reserve)
        rows = B * L * H * self.cap
        p.packed_rows = rows if tensor_cores else 0
        dt = TORCH_DT[p.dtype]
        self.K = torch.zeros((rows, p.d), dtype=dt, device=dev)
        self.V = torch.zeros((rows, p.d), dtype=dt, device=dev)
        self.pos = torch.zeros((rows,), dtype=torch.float32, device=dev)
        self.logm = torch.zeros((rows,), dtype=torch.float32, device=dev)
        self._prompt = (K, V)
        self.len_lh = torch.zeros((B * L * H,), dtype=torch.int32, device=dev)
        self.cap_lh = torch.full((B * L * H,), self.cap, dtype=torch.int32, device=dev)
        self.off_lh = torch.arange(B * L * H, dtype=torch.int64, device=dev) * self.cap
        self.lse = torch.zeros((B * L * H, p.G), dtype=torch.float32, device=dev)
        # the decode's per-entry scores feed alpha (else alpha recomputes them from K)
        self.scores = (torch.zeros((rows, p.G), dtype=torch.float32, device=dev)
                       if scores else None)
        self.alpha = torch.zeros((B, self.cap), dtype=torch.float32, device=dev)
        self.ws_decode = torch.zeros(kvc.kvc_workspace_bytes(kvc.KVC_WS_DECODE, p),
                                     dtype=torch.uint8, device=dev)
        self.ws_evict = torch.empty(kvc.kvc_evict_workspace_bytes(p, self.cap),
                                    dtype=torch.uint8, device=dev)
        self._graphs = {}
        self.reset()

    def reset(self):
        """Back to the prompt: every (b, l, h) holds the prompt tokens in order."""
        p, (K, V) = self.p, self._prompt
        B, L, H = p.B, p.L, p.H
        Kc = self.K.view(B, L, H, self.cap, p.d)
        Vc = self.V.view(B, L, H, self.cap, p.d)
        Pc = self.pos.view(B, L, H, self.cap)
        for b, n in enumerate(self.ctx):
            assert n <= K.shape[3]
            Kc[b, :, :, :n] = K[b, :, :, :n]
            Vc[b, :, :, :n] = V[b, :, :, :n]
            Pc[b, :, :, :n] = torch.arange(n, dtype=torch.float32, device=K.device)
        lens = np.repeat(np.asarray(self.ctx, np.int32), L * H)
        self.len_lh.copy_(torch.from_numpy(lens))
        self.logm.zero_()

    def step(self, q, k_new, v_new, out, n_seen, pos_new=None, stream=None):
        """One decode step then one eviction; n_seen [B] int64 = tokens seen so far,
        this step's included."""
        kvc.kvc_decode_attn_lse(self.p, q, k_new, v_new, pos_new, self.K, self.V, self.logm,
                                self.pos, self.len_lh, self.cap_lh, self.off_lh, out, self.lse,
                                self.scores, self.ws_decode, stream)
        kvc.kvc_token_alpha(self.p, q, self.K, self.scores, self.len_lh, self.off_lh, self.lse,
                            self.alpha, self.ws_evict, stream)
        kvc.kvc_evict_topb(self.p, self.alpha, n_seen, self.ratio, self.b_min, self.K, self.V,
                           self.pos, self.logm, self.off_lh, self.len_lh, self.ws_evict, stream)

    def run_many(self, q_all, kn_all, vn_all, out_all, nseen_all, pos_all=None, graph=True):
        """T steps back to back (step t reads row t of every *_all tensor); with
        graph=True they are captured once per set of buffers into a CUDA graph
        and replayed.  Returns the library kernels launched."""
        T = q_all.shape[0]
        if not graph:
            n0 = kvc.kvc_launch_count()
            for t in range(T):
                self.step(q_all[t], kn_all[t], vn_all[t], out_all[t], nseen_all[t],
                          None if pos_all is None else pos_all[t])
            return kvc.kvc_launch_count() - n0
        key = tuple(x.data_ptr() if x is not None else 0
                    for x in (q_all, kn_all, vn_all, out_all, nseen_all, pos_all)) + (T,)
        g = self._graphs.get(key)
        if g is None:
            dev = q_all.device
            kvc.kvc_device_error()                   # error-word lookup outside capture
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            graph_ = torch.cuda.CUDAGraph()
            n0 = kvc.kvc_launch_count()
            with torch.cuda.graph(graph_, stream=side):
                for t in range(T):
                    self.step(q_all[t], kn_all[t], vn_all[t], out_all[t], nseen_all[t],
                              None if pos_all is None else pos_all[t], side)
            torch.cuda.current_stream(dev).wait_stream(side)
            g = (graph_, kvc.kvc_launch_count() - n0,
                 (q_all, kn_all, vn_all, out_all, nseen_all, pos_all))
            self._graphs[key] = g
        g[0].replay()
        return g[1]

    def entries(self, b: int, l: int, h: int):
        """(K, V, pos) rows the (b, l, h) currently holds, in row order (host copies)."""
        blh = (b * self.p.L + l) * self.p.H + h
        n = int(self.len_lh[blh])
        o = blh * self.cap
        return (self.K[o:o + n].float().cpu().numpy(), self.V[o:o + n].float().cpu().numpy(),
                self.pos[o:o + n].cpu().numpy())


def pad_bounds(bounds_list, S_max: int) -> np.ndarray:
    """[B, S_max + 1] int32 slot boundaries (rows padded with their last value)."""
    out = np.zeros((len(bounds_list), S_max + 1), dtype=np.int32)
    for b, bd in enumerate(bounds_list):
        bd = np.asarray(bd, dtype=np.int32)
        out[b, :len(bd)] = bd
        out[b, len(bd):] = bd[-1]
    return out
