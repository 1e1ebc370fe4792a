"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/kvc.h declares (host-only calls; no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from kv_cache_compression_probe_gb300 import build as B
    B.build()
    from kv_cache_compression_probe_gb300 import kvc
    return kvc.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    from kv_cache_compression_probe_gb300 import kvc
    assert set(names) == set(kvc.EXPORTED)


def test_host_only_calls(lib):
    from kv_cache_compression_probe_gb300 import kvc
    assert kvc.kvc_status_string(0) == "ok"
    assert "budget" in kvc.kvc_status_string(kvc.KVC_EBUDGET)
    assert kvc.kvc_launch_count() >= 0
    p = kvc.make_params(B=1, L=32, H=8, G=4, d=128, P=64, W=128, dtype=kvc.KVC_BF16, n_max=16384,
                        S_max=300, decode_reserve=256)
    for w in range(5):
        assert kvc.kvc_workspace_bytes(w, p) > 0
    bad = kvc.make_params(B=1, L=1, H=1, G=3, d=128, P=64, W=128, dtype=1, n_max=1000, S_max=4)
    assert kvc.kvc_workspace_bytes(kvc.KVC_WS_DECODE, bad) == 0


def test_params_struct_layout_matches_header():
    from kv_cache_compression_probe_gb300 import kvc
    assert ctypes.sizeof(kvc.kvc_params) == 144
    assert kvc.kvc_params.tree_cuts.offset == 128
    assert kvc.kvc_params.salient_extract.offset == 136
    assert kvc.kvc_params.total_ctx.offset == 104
    assert kvc.kvc_params.packed_rows.offset == 112
    assert kvc.kvc_params.head_full_frac.offset == 120
    assert kvc.kvc_params.budget_ratio.offset == 64
    assert kvc.kvc_params.floor_cap_tokens.offset == 88
    assert kvc.kvc_params.decode_reserve.offset == 96


def test_binding_argument_counts_match_header(lib):
    """Each ctypes prototype has as many arguments as the header declaration."""
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for name, args in re.findall(r"\b(kvc_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", src):
        n = 0 if args.strip() in ("", "void") else len(args.split(","))
        assert len(getattr(lib, name).argtypes) == n, name


def test_tree_cuts_rejects_bad_arguments_on_the_host(lib):
    """kvc_tree_cuts checks its arguments before touching the device: missing
    pointers and more than 65535 (b,l,h) give KVC_EINVAL (no GPU needed)."""
    from kv_cache_compression_probe_gb300 import kvc
    p = kvc.make_params(B=1, L=2, H=2, G=4, d=128, P=64, W=128, dtype=kvc.KVC_BF16, n_max=4096,
                        S_max=64)
    fake = [ctypes.c_void_p(256 * (k + 1)) for k in range(8)]   # never dereferenced
    assert lib.kvc_tree_cuts(ctypes.byref(p), None, *fake[1:], None) == kvc.KVC_EINVAL
    assert lib.kvc_tree_cuts(ctypes.byref(p), *fake[:7], None, None) == kvc.KVC_EINVAL
    big = kvc.make_params(B=1, L=300, H=256, G=1, d=128, P=64, W=128, dtype=kvc.KVC_BF16,
                          n_max=4096, S_max=64)
    assert lib.kvc_tree_cuts(ctypes.byref(big), *fake, None) == kvc.KVC_EINVAL


def test_binding_constants_match_header():
    """Status codes and the allocation-free decode's scratch size agree with kvc.h."""
    from kv_cache_compression_probe_gb300 import kvc
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    defs = dict(re.findall(r"#define\s+(KVC_[A-Z_0-9]+)\s+(\S.*?)\s*(?:/\*.*)?$", src, flags=re.M))
    for name in ("KVC_OK", "KVC_EINVAL", "KVC_EBUDGET", "KVC_ECAPACITY", "KVC_ECUDA",
                 "KVC_ETIMEOUT", "KVC_EWORKSPACE", "KVC_EDEVICE", "KVC_ESCRATCH"):
        assert int(defs[name]) == getattr(kvc, name), name
    m = re.fullmatch(r"\((\d+)u\s*<<\s*(\d+)\)", defs["KVC_DECODE_STATIC_SCRATCH_BYTES"])
    assert int(m.group(1)) << int(m.group(2)) == kvc.KVC_DECODE_STATIC_SCRATCH_BYTES
