"""Host logic of bench.py that decides what its JSON line reports: the
stored DRAM traffic is used only for the kernel source it was taken on, and
the source hash covers every kernel file and the C header.  No GPU."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _copy_sources(dst):
    src = os.path.join(ROOT, "activation_sparse_decode_rank_gb300", "csrc")
    os.makedirs(os.path.join(dst, "activation_sparse_decode_rank_gb300"))
    shutil.copytree(src, os.path.join(dst, "activation_sparse_decode_rank_gb300", "csrc"),
                    ignore=shutil.ignore_patterns("*.o", "*.so"))
    os.makedirs(os.path.join(dst, "include"))
    shutil.copy(os.path.join(ROOT, "include", "pi.h"), os.path.join(dst, "include", "pi.h"))


def test_source_hash_follows_kernels_and_header(tmp_path, monkeypatch):
    _copy_sources(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.csrc_hash()
    assert len(h0) == 16 and int(h0, 16) >= 0
    # a file that is not a kernel source leaves it alone
    (tmp_path / "activation_sparse_decode_rank_gb300" / "csrc" / "notes.txt").write_text("x")
    assert bench.csrc_hash() == h0
    # one byte more in a kernel source, or in the header, changes it
    cu = sorted(p for p in (tmp_path / "activation_sparse_decode_rank_gb300" / "csrc").iterdir()
                if p.suffix in (".cu", ".cuh"))[0]
    cu.write_bytes(cu.read_bytes() + b"\n")
    h1 = bench.csrc_hash()
    assert h1 != h0
    hp = tmp_path / "include" / "pi.h"
    hp.write_bytes(hp.read_bytes() + b"\n")
    assert bench.csrc_hash() not in (h0, h1)


def test_stored_traffic_only_for_the_current_source(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(f))
    key = "seq_kernel:some_stack:4"
    assert bench.stored_traffic(key) is None  # no file
    f.write_text("{not json")
    assert bench.stored_traffic(key) is None  # unreadable file
    entry = {"csrc_hash": bench.csrc_hash(), "dram_bytes_per_step": 1234.0,
             "algorithmic_bytes_per_step": 1000.0}
    f.write_text(json.dumps({key: entry}))
    assert bench.stored_traffic(key) == (1234.0, 1000.0)
    assert bench.stored_traffic("seq_kernel:other:4") is None  # another workload
    f.write_text(json.dumps({key: dict(entry, csrc_hash="0" * 16)}))
    assert bench.stored_traffic(key) is None  # taken on other kernel source
    f.write_text(json.dumps({key: {"csrc_hash": bench.csrc_hash()}}))
    assert bench.stored_traffic(key) is None  # no per-step figure


def test_committed_traffic_entries_are_well_formed():
    # every committed entry names its source hash, the command that made it
    # and per-step (or per-launch) byte counts that add up
    j = json.load(open(bench.PROFILE_TRAFFIC))
    assert j
    for key, e in j.items():
        assert len(e["csrc_hash"]) == 16 and e["source"].startswith(("ncu ", "python "))
        assert "--clock-control none" in e["source"]
        for unit in ("per_step", "per_launch"):
            rd, wr = e.get(f"dram_bytes_read_{unit}"), e.get(f"dram_bytes_write_{unit}")
            if rd is not None and f"dram_bytes_{unit}" in e:
                assert e[f"dram_bytes_{unit}"] == pytest.approx(rd + wr, rel=1e-9)


def test_aggregate_is_all_units_over_the_slowest_time():
    v, t = bench.aggregate([10.0, 12.5], [100, 100], 2)
    assert t == 12.5 and v == pytest.approx(200 / 0.0125)
    assert bench.aggregate([0.0], [5], 1)[0] == 0.0
