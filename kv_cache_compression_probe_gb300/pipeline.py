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


class Compressor:
    def __init__(self, p: kvc.kvc_params, ctx_len: Sequence[int], device="cuda",
                 tensor_cores: bool = True):
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
        self._graphs = {}

    # ---------------------------------------------------------------- calls
    def score(self, K, V, Qp, slot_bounds, n_slots, head_sens=None, stream=None):
        kvc.kvc_score(self.p, self.ctx_len, K, V, Qp, self.rope_cos, self.rope_sin, slot_bounds,
                      n_slots, head_sens, self.lse, self.feats, self.relevance, self.op_util,
                      self.op_cost, self.ws_score, stream)

    def select(self, slot_bounds, n_slots, head_sens=None, op_util=None, relevance=None,
               stream=None):
        kvc.kvc_select(self.p, self.ctx_len, slot_bounds, n_slots,
                       self.relevance if relevance is None else relevance, head_sens,
                       self.op_util if op_util is None else op_util, self.op_cost, self.taken,
                       self.len_lh, self.cap_lh, self.off_lh, self.total, self.ws_select, stream)

    def merge_pack(self, K, V, slot_bounds, n_slots, taken=None, stream=None):
        kvc.kvc_merge_pack(self.p, self.ctx_len, K, V, self.relevance, self.rope_cos,
                           self.rope_sin, slot_bounds, n_slots,
                           self.taken if taken is None else taken, self.len_lh, self.off_lh,
                           self.Kp, self.Vp, self.logm, self.pos, self.ws_pack, stream)

    def compress(self, K, V, Qp, slot_bounds, n_slots, head_sens=None, stream=None):
        self.score(K, V, Qp, slot_bounds, n_slots, head_sens, stream)
        self.select(slot_bounds, n_slots, head_sens, stream=stream)
        self.merge_pack(K, V, slot_bounds, n_slots, stream=stream)

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


def pad_bounds(bounds_list, S_max: int) -> np.ndarray:
    """[B, S_max + 1] int32 slot boundaries (rows padded with their last value)."""
    out = np.zeros((len(bounds_list), S_max + 1), dtype=np.int32)
    for b, bd in enumerate(bounds_list):
        bd = np.asarray(bd, dtype=np.int32)
        out[b, :len(bd)] = bd
        out[b, len(bd):] = bd[-1]
    return out
