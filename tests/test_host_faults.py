"""Host-side fault injection: every entry point rejects a malformed parameter
block, a missing pointer, and a workspace that is missing, too small or
misaligned, with its status code and before it touches the device (no GPU
needed: the fake pointers are never dereferenced)."""
import ctypes

import pytest

from kv_cache_compression_probe_gb300 import kvc

VP = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    from kv_cache_compression_probe_gb300 import build
    build.build()
    return kvc.lib()


def _params(**over):
    kw = dict(B=1, L=2, H=2, G=4, d=128, P=16, W=32, dtype=kvc.KVC_BF16, n_max=1024, S_max=16,
              decode_reserve=4)
    kw.update(over)
    return kvc.make_params(**kw)


def _fake(k):
    return [VP(4096 * (i + 1)) for i in range(k)]


# name, pointer arguments before the workspace, workspace kind, extra scalar
# arguments (inserted at the given index)
CALLS = {
    "kvc_score": (14, kvc.KVC_WS_SCORE, {}),
    "kvc_select": (12, kvc.KVC_WS_SELECT, {}),
    "kvc_merge_pack": (15, kvc.KVC_WS_PACK, {15: ctypes.c_int64(1 << 20)}),
    "kvc_decode_attn": (12, kvc.KVC_WS_DECODE, {}),
    "kvc_partition": (5, kvc.KVC_WS_PARTITION, {2: ctypes.c_int32(256)}),
}
# pointers the header lets be NULL (head_sens, pos_new): never left out here,
# since the call would then go on to the device with the fake pointers
OPTIONAL = {"kvc_score": {8}, "kvc_select": {4}, "kvc_decode_attn": {3}}


def _args(name, ptrs, ws, ws_bytes):
    n, _, extra = CALLS[name]
    args = list(ptrs)
    for i in sorted(extra):
        args.insert(i, extra[i])
    return args + [ws, ctypes.c_size_t(ws_bytes), None]


def _call(lib, name, p, ptrs, ws, ws_bytes):
    return getattr(lib, name)(ctypes.byref(p), *_args(name, ptrs, ws, ws_bytes))


BAD_PARAMS = [dict(B=0), dict(L=0), dict(H=-1), dict(G=3), dict(d=96), dict(P=0),
              dict(G=8, P=64), dict(W=8), dict(dtype=7), dict(n_max=40), dict(S_max=0),
              dict(decode_reserve=-1), dict(packed_rows=-5), dict(head_full_frac=1.5)]


@pytest.mark.parametrize("name", list(CALLS))
@pytest.mark.parametrize("bad", BAD_PARAMS, ids=[next(iter(b)) + "=" + str(next(iter(b.values())))
                                                 for b in BAD_PARAMS])
def test_malformed_parameters_are_rejected(lib, name, bad):
    p = _params(**bad)
    n, which, _ = CALLS[name]
    assert _call(lib, name, p, _fake(n), VP(1 << 20), 1 << 40) == kvc.KVC_EINVAL


@pytest.mark.parametrize("name", list(CALLS))
def test_missing_pointers_are_rejected(lib, name):
    p = _params()
    n, which, _ = CALLS[name]
    need = lib.kvc_workspace_bytes(which, ctypes.byref(p))
    assert need > 0
    for i in range(n):
        if i in OPTIONAL.get(name, ()):
            continue
        ptrs = _fake(n)
        ptrs[i] = None
        assert _call(lib, name, p, ptrs, VP(1 << 20), need) == kvc.KVC_EINVAL, (name, i)


@pytest.mark.parametrize("name", list(CALLS))
def test_bad_workspaces_are_rejected(lib, name):
    p = _params()
    n, which, _ = CALLS[name]
    need = lib.kvc_workspace_bytes(which, ctypes.byref(p))
    ptrs = _fake(n)
    assert _call(lib, name, p, ptrs, None, need) == kvc.KVC_EWORKSPACE
    assert _call(lib, name, p, ptrs, VP(1 << 20), need - 1) == kvc.KVC_EWORKSPACE
    assert _call(lib, name, p, ptrs, VP((1 << 20) + 16), need) == kvc.KVC_EWORKSPACE


def test_budget_below_the_window_is_reported(lib):
    p = _params(budget_entries_per_lh=8)                  # W = 32
    need = lib.kvc_workspace_bytes(kvc.KVC_WS_SELECT, ctypes.byref(p))
    assert _call(lib, "kvc_select", p, _fake(12), VP(1 << 20), need) == kvc.KVC_EBUDGET


def test_workspace_size_of_a_malformed_block_is_zero(lib):
    for which in range(5):
        assert lib.kvc_workspace_bytes(which, ctypes.byref(_params(d=96))) == 0


def test_tree_cuts_rejects_bad_arguments(lib):
    """kvc_tree_cuts (no workspace): a malformed block, each missing pointer
    and a key pointer off a 16-byte boundary (the key rows are read with
    vector loads) are rejected before any launch."""
    args = _fake(8)                      # ctx_len, K, cos, sin, bounds, n_slots, kappa, cuts
    assert lib.kvc_tree_cuts(ctypes.byref(_params(B=0)), *args, None) == kvc.KVC_EINVAL
    for i in range(8):
        a = list(args)
        a[i] = None
        assert lib.kvc_tree_cuts(ctypes.byref(_params()), *a, None) == kvc.KVC_EINVAL, i
    a = list(args)
    a[1] = VP(4096 + 8)
    assert lib.kvc_tree_cuts(ctypes.byref(_params()), *a, None) == kvc.KVC_EINVAL


@pytest.mark.parametrize("name,idx", [("kvc_score", 1), ("kvc_score", 2), ("kvc_score", 3),
                                      ("kvc_merge_pack", 1), ("kvc_merge_pack", 2),
                                      ("kvc_merge_pack", 11), ("kvc_merge_pack", 12)])
def test_row_arrays_off_a_16_byte_boundary_are_rejected(lib, name, idx):
    """K, V, Qp (score) and K, V, Kp, Vp (pack) are read or written as whole
    16-byte vectors and prefetched in bulk: an array off a 16-byte boundary is
    rejected before any launch (the workspace is valid, so the status can only
    come from the pointer)."""
    p = _params()
    n, kind, _ = CALLS[name]
    need = kvc.kvc_workspace_bytes(kind, p)
    ptrs = _fake(n)
    ptrs[idx] = VP(4096 * (idx + 1) + 8)
    assert _call(lib, name, p, ptrs, VP(1 << 30), need) == kvc.KVC_EINVAL
