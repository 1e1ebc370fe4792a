"""Thin ctypes binding of libkvc (include/kvc.h).

Every function has the C name and only marshals arguments: torch CUDA tensors
become raw device pointers, the stream defaults to torch's current stream, and a
negative status raises KvcError.  All compute runs in libkvc's kernels; there
is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

KVC_OK, KVC_EINVAL, KVC_EBUDGET, KVC_ECAPACITY = 0, -1, -2, -3
KVC_ECUDA, KVC_ETIMEOUT, KVC_EWORKSPACE, KVC_EDEVICE, KVC_ESCRATCH = -4, -5, -6, -7, -8
KVC_F32, KVC_BF16 = 0, 1
KVC_WS_SCORE, KVC_WS_SELECT, KVC_WS_PACK, KVC_WS_DECODE, KVC_WS_PARTITION = range(5)
KVC_DECODE_STATIC_SCRATCH_BYTES = 48 << 20   # the allocation-free decode's array (kvc.h)

EXPORTED = ("kvc_status_string", "kvc_last_cuda_error", "kvc_device_error", "kvc_launch_count", "kvc_workspace_bytes",
            "kvc_rope_table", "kvc_score", "kvc_select", "kvc_merge_pack", "kvc_decode_attn",
            "kvc_partition", "kvc_decode_attn_noalloc", "kvc_decode_attn_lse", "kvc_token_alpha",
            "kvc_evict_workspace_bytes", "kvc_evict_topb", "kvc_set_phase_timing",
            "kvc_score_phase_ms", "kvc_decode_attn_layers", "kvc_tree_cuts", "kvc_set_wait_limit")


class kvc_params(ctypes.Structure):
    _fields_ = [
        ("B", c_int32), ("L", c_int32), ("H", c_int32), ("G", c_int32), ("d", c_int32),
        ("P", c_int32), ("W", c_int32), ("dtype", c_int32), ("n_max", c_int32),
        ("S_max", c_int32), ("rope_base", c_float), ("hop_weight", c_float),
        ("n_hops", c_int32), ("w_part", c_float), ("w_value", c_float), ("value_floor", c_float),
        ("budget_ratio", c_double), ("budget_entries_per_lh", c_int64),
        ("floor_cap_frac", c_double), ("floor_cap_tokens", c_int64), ("decode_reserve", c_int32),
        ("total_ctx", c_int64),
        ("packed_rows", c_int64),
        ("head_full_frac", c_double),
        ("tree_cuts", ctypes.c_void_p),
        ("salient_extract", c_int32),
    ]


class KvcError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = f"{what}: {kvc_status_string(status)} ({status})"
        if status == KVC_ECUDA:
            msg += f": {lib().kvc_last_cuda_error().decode()}"
        super().__init__(msg)
        self.status = status


_lib = None
_P = ctypes.POINTER(kvc_params)


def lib():
    """Load libkvc.so (after torch, so its CUDA runtime is shared).  Raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp = c_void_p
        L.kvc_status_string.argtypes = [c_int]; L.kvc_status_string.restype = ctypes.c_char_p
        L.kvc_last_cuda_error.argtypes = []; L.kvc_last_cuda_error.restype = ctypes.c_char_p
        L.kvc_device_error.argtypes = [vp, ctypes.POINTER(c_int32)]; L.kvc_device_error.restype = c_int
        L.kvc_launch_count.argtypes = []; L.kvc_launch_count.restype = c_int64
        L.kvc_set_wait_limit.argtypes = [ctypes.c_uint64, c_int32]
        L.kvc_set_wait_limit.restype = c_int
        L.kvc_workspace_bytes.argtypes = [c_int, _P]; L.kvc_workspace_bytes.restype = c_size_t
        L.kvc_rope_table.argtypes = [c_int32, c_float, c_int64, vp, vp, vp]
        L.kvc_rope_table.restype = c_int
        L.kvc_score.argtypes = [_P] + [vp] * 15 + [c_size_t, vp]; L.kvc_score.restype = c_int
        L.kvc_select.argtypes = [_P] + [vp] * 13 + [c_size_t, vp]; L.kvc_select.restype = c_int
        L.kvc_merge_pack.argtypes = [_P] + [vp] * 15 + [c_int64, vp, c_size_t, vp]
        L.kvc_merge_pack.restype = c_int
        L.kvc_decode_attn.argtypes = [_P] + [vp] * 13 + [c_size_t, vp]
        L.kvc_decode_attn.restype = c_int
        L.kvc_decode_attn_noalloc.argtypes = [_P] + [vp] * 13
        L.kvc_decode_attn_noalloc.restype = c_int
        L.kvc_decode_attn_layers.argtypes = [_P, c_int32, c_int32] + [vp] * 13 + [c_size_t, vp]
        L.kvc_decode_attn_layers.restype = c_int
        L.kvc_decode_attn_lse.argtypes = [_P] + [vp] * 15 + [c_size_t, vp]
        L.kvc_decode_attn_lse.restype = c_int
        L.kvc_token_alpha.argtypes = [_P] + [vp] * 7 + [c_int32, vp, c_size_t, vp]
        L.kvc_token_alpha.restype = c_int
        L.kvc_evict_workspace_bytes.argtypes = [_P, c_int32]
        L.kvc_evict_workspace_bytes.restype = c_size_t
        L.kvc_evict_topb.argtypes = [_P, vp, c_int32, vp, c_double, c_int32] + [vp] * 7 + [c_size_t, vp]
        L.kvc_evict_topb.restype = c_int
        L.kvc_set_phase_timing.argtypes = [c_int]; L.kvc_set_phase_timing.restype = None
        L.kvc_score_phase_ms.argtypes = [ctypes.POINTER(c_float), c_int32]
        L.kvc_score_phase_ms.restype = c_int
        L.kvc_partition.argtypes = [_P, vp, vp, c_int32, vp, vp, vp, vp, c_size_t, vp]
        L.kvc_partition.restype = c_int
        L.kvc_tree_cuts.argtypes = [_P] + [vp] * 9
        L.kvc_tree_cuts.restype = c_int
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors passed to libkvc must be contiguous CUDA tensors")
    return c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return c_void_p(stream.cuda_stream)
    return c_void_p(int(stream))


def _check(st: int, what: str):
    if st != KVC_OK:
        raise KvcError(st, what)


def _ws(t):
    return (_ptr(t), t.numel() * t.element_size()) if t is not None else (None, 0)


def make_params(**kw) -> kvc_params:
    p = kvc_params()
    defaults = dict(rope_base=10000.0, hop_weight=0.3, n_hops=2, w_part=0.25, w_value=0.75,
                    value_floor=0.1, budget_ratio=0.25, budget_entries_per_lh=0,
                    floor_cap_frac=0.6, floor_cap_tokens=-1, decode_reserve=0, total_ctx=0,
                    packed_rows=0, head_full_frac=0.0, tree_cuts=None)
    defaults.update(kw)
    for k, v in defaults.items():
        setattr(p, k, v)
    return p


# ------------------------------------------------------------------ calls
def kvc_status_string(st: int) -> str:
    return lib().kvc_status_string(st).decode()


def kvc_device_error(stream=None) -> int:
    code = c_int32(0)
    _check(lib().kvc_device_error(_stream(stream), ctypes.byref(code)), "kvc_device_error")
    return code.value


def kvc_launch_count() -> int:
    return int(lib().kvc_launch_count())


def kvc_set_wait_limit(first_wait_ns: int, withhold_copies: bool = False):
    _check(lib().kvc_set_wait_limit(int(first_wait_ns), 1 if withhold_copies else 0),
           "kvc_set_wait_limit")


def kvc_workspace_bytes(which: int, p: kvc_params) -> int:
    return int(lib().kvc_workspace_bytes(which, ctypes.byref(p)))


def kvc_rope_table(d: int, base: float, n_half: int, cos_tab, sin_tab, stream=None):
    _check(lib().kvc_rope_table(d, base, n_half, _ptr(cos_tab), _ptr(sin_tab), _stream(stream)),
           "kvc_rope_table")


def kvc_score(p, ctx_len, K, V, Qp, rope_cos, rope_sin, slot_bounds, n_slots, head_sens,
              lse, feats, relevance, op_util, op_cost, workspace, stream=None):
    w, wb = _ws(workspace)
    _check(lib().kvc_score(ctypes.byref(p), _ptr(ctx_len), _ptr(K), _ptr(V), _ptr(Qp),
                           _ptr(rope_cos), _ptr(rope_sin), _ptr(slot_bounds), _ptr(n_slots),
                           _ptr(head_sens), _ptr(lse), _ptr(feats), _ptr(relevance),
                           _ptr(op_util), _ptr(op_cost), w, wb, _stream(stream)), "kvc_score")


def kvc_select(p, ctx_len, slot_bounds, n_slots, relevance, head_sens, op_util, op_cost, taken,
               len_lh, cap_lh, off_lh, total_entries, workspace, stream=None):
    w, wb = _ws(workspace)
    _check(lib().kvc_select(ctypes.byref(p), _ptr(ctx_len), _ptr(slot_bounds), _ptr(n_slots),
                            _ptr(relevance), _ptr(head_sens), _ptr(op_util), _ptr(op_cost),
                            _ptr(taken), _ptr(len_lh), _ptr(cap_lh), _ptr(off_lh),
                            _ptr(total_entries), w, wb, _stream(stream)), "kvc_select")


def kvc_merge_pack(p, ctx_len, K, V, relevance, rope_cos, rope_sin, slot_bounds, n_slots, taken,
                   len_lh, off_lh, Kp, Vp, logm, pos, workspace, stream=None):
    w, wb = _ws(workspace)
    _check(lib().kvc_merge_pack(ctypes.byref(p), _ptr(ctx_len), _ptr(K), _ptr(V), _ptr(relevance),
                                _ptr(rope_cos), _ptr(rope_sin), _ptr(slot_bounds), _ptr(n_slots),
                                _ptr(taken), _ptr(len_lh), _ptr(off_lh), _ptr(Kp), _ptr(Vp),
                                _ptr(logm), _ptr(pos), Kp.shape[0], w, wb, _stream(stream)),
           "kvc_merge_pack")


def kvc_decode_attn(p, q, k_new, v_new, pos_new, Kp, Vp, logm, pos, len_lh, cap_lh, off_lh, out,
                    workspace, stream=None):
    w, wb = _ws(workspace)
    _check(lib().kvc_decode_attn(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new),
                                 _ptr(pos_new), _ptr(Kp), _ptr(Vp), _ptr(logm), _ptr(pos),
                                 _ptr(len_lh), _ptr(cap_lh), _ptr(off_lh), _ptr(out), w, wb,
                                 _stream(stream)), "kvc_decode_attn")


def kvc_decode_attn_layers(p, layer_begin, layer_end, q, k_new, v_new, pos_new, Kp, Vp, logm,
                           pos, len_lh, cap_lh, off_lh, out, workspace, stream=None):
    """kvc_decode_attn over layers [layer_begin, layer_end) (q, k_new, v_new, out
    cover the range; the per-(b,l,h) arrays are whole)."""
    w, wb = _ws(workspace)
    _check(lib().kvc_decode_attn_layers(ctypes.byref(p), int(layer_begin), int(layer_end), _ptr(q),
                                        _ptr(k_new), _ptr(v_new), _ptr(pos_new), _ptr(Kp),
                                        _ptr(Vp), _ptr(logm), _ptr(pos), _ptr(len_lh),
                                        _ptr(cap_lh), _ptr(off_lh), _ptr(out), w, wb,
                                        _stream(stream)), "kvc_decode_attn_layers")


def kvc_decode_attn_noalloc(p, q, k_new, v_new, pos_new, Kp, Vp, logm, pos, len_lh, cap_lh,
                            off_lh, out, stream=None):
    """kvc_decode_attn without a workspace: the library's fixed device scratch array
    is used instead (for callers that cannot allocate device memory)."""
    _check(lib().kvc_decode_attn_noalloc(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new),
                                         _ptr(pos_new), _ptr(Kp), _ptr(Vp), _ptr(logm),
                                         _ptr(pos), _ptr(len_lh), _ptr(cap_lh), _ptr(off_lh),
                                         _ptr(out), _stream(stream)), "kvc_decode_attn_noalloc")


def kvc_decode_attn_lse(p, q, k_new, v_new, pos_new, Kp, Vp, logm, pos, len_lh, cap_lh, off_lh,
                        out, lse_out, scores_out, workspace, stream=None):
    w, wb = _ws(workspace)
    _check(lib().kvc_decode_attn_lse(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new),
                                     _ptr(pos_new), _ptr(Kp), _ptr(Vp), _ptr(logm), _ptr(pos),
                                     _ptr(len_lh), _ptr(cap_lh), _ptr(off_lh), _ptr(out),
                                     _ptr(lse_out), _ptr(scores_out), w, wb, _stream(stream)),
           "kvc_decode_attn_lse")


def kvc_token_alpha(p, q, Kp, scores, len_lh, off_lh, lse_out, alpha, workspace, stream=None):
    w, wb = _ws(workspace)
    _check(lib().kvc_token_alpha(ctypes.byref(p), _ptr(q), _ptr(Kp), _ptr(scores), _ptr(len_lh),
                                 _ptr(off_lh), _ptr(lse_out), _ptr(alpha), alpha.shape[1], w, wb,
                                 _stream(stream)), "kvc_token_alpha")


def kvc_evict_workspace_bytes(p, alpha_cols: int) -> int:
    return int(lib().kvc_evict_workspace_bytes(ctypes.byref(p), alpha_cols))


def kvc_evict_topb(p, alpha, n_seen, ratio, b_min, K, V, pos, logm, off_lh, len_lh, workspace,
                   stream=None):
    w, wb = _ws(workspace)
    _check(lib().kvc_evict_topb(ctypes.byref(p), _ptr(alpha), alpha.shape[1], _ptr(n_seen),
                                float(ratio), int(b_min), _ptr(K), _ptr(V), _ptr(pos),
                                _ptr(logm), _ptr(off_lh), _ptr(len_lh), w, wb, _stream(stream)),
           "kvc_evict_topb")


def kvc_set_phase_timing(on: bool):
    lib().kvc_set_phase_timing(1 if on else 0)


def kvc_score_phase_ms(n: int = 5):
    """Durations (ms) of the phases of the last timed kvc_score call."""
    buf = (c_float * n)()
    st = lib().kvc_score_phase_ms(buf, n)
    if st < 0:
        raise KvcError(st, "kvc_score_phase_ms")
    return [float(buf[i]) for i in range(st)]


def kvc_partition(p, ctx_len, hidden, dh, kappa, slot_bounds, n_slots, workspace, stream=None):
    w, wb = _ws(workspace)
    _check(lib().kvc_partition(ctypes.byref(p), _ptr(ctx_len), _ptr(hidden), dh, _ptr(kappa),
                               _ptr(slot_bounds), _ptr(n_slots), w, wb, _stream(stream)),
           "kvc_partition")


def kvc_tree_cuts(p, ctx_len, K, rope_cos, rope_sin, slot_bounds, n_slots, kappa, cuts,
                  stream=None):
    _check(lib().kvc_tree_cuts(ctypes.byref(p), _ptr(ctx_len), _ptr(K), _ptr(rope_cos),
                               _ptr(rope_sin), _ptr(slot_bounds), _ptr(n_slots), _ptr(kappa),
                               _ptr(cuts), _stream(stream)), "kvc_tree_cuts")


def workspace(which: int, p: kvc_params, device="cuda", zero=False) -> torch.Tensor:
    """A 256-byte aligned workspace tensor for call `which` (torch's allocator
    returns 512-byte aligned blocks)."""
    n = max(kvc_workspace_bytes(which, p), 256)
    t = (torch.zeros if zero else torch.empty)(n, dtype=torch.uint8, device=device)
    assert t.data_ptr() % 256 == 0
    return t
