"""Host-side pieces of bench.py's records (CPU only): the select byte model
and the parity record's staleness check."""
import json
import os

import bench


def test_select_roofline_byte_model():
    class Cfg:
        L, H = 2, 3
    # (n, slot bounds): 40 tokens in 3 slots, 24 tokens in 2 slots
    seqs = [(40, [0, 10, 25, 40]), (24, [0, 12, 24])]
    r = bench.select_roofline(Cfg, seqs, sel_ms=1.0, hbm=1000.0)
    ops = 6 * (3 + 2) * 16
    toks = 6 * (40 + 24)
    assert r["algorithmic_bytes"] == 8 * (ops * 12 + toks * 5)
    assert abs(r["achieved"] - r["algorithmic_bytes"] / 1e-3 / 1e9) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 1000.0) < 1e-12


def test_parity_record_is_current_only_for_the_recorded_sources(tmp_path, monkeypatch):
    root = tmp_path
    (root / "profiles").mkdir()
    srcs = []
    for k in range(2):
        f = root / f"src{k}.cu"
        f.write_bytes(b"kernel %d" % k)
        srcs.append(f.name)
    import hashlib
    h = hashlib.sha256()
    for f in srcs:
        h.update((root / f).read_bytes())
    rec = {"tie_band_rel": 1e-6, "source_sha256": h.hexdigest(),
           "sequences": [{"ops": 10, "ties_reported": 0, "tie_runs_reordered": 1,
                          "util_max_abs_err": 1e-9, "util_max_rel_err": 1e-3,
                          "util_within_1e5_rel": 9, "util_within_scale_term_only": 1,
                          "util_worst_err_over_bound": 0.5}]}
    (root / "profiles" / "parity_w.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(root))
    monkeypatch.setattr(bench, "PARITY_SOURCES", srcs)
    r = bench.parity_record("w")
    assert r["current"] and r["ops"] == 10 and r["util_within_scale_term_only"] == 1
    (root / srcs[0]).write_bytes(b"changed")
    assert not bench.parity_record("w")["current"]
    assert bench.parity_record("missing") is None
