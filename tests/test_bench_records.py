"""The committed measurement records bench.py reads, checked on the CPU.

`profiles/traffic.json` holds one ncu DRAM-traffic figure per (kernel, workload) with the SHA-256
of the kernel's source at capture time; bench.py reports the figure only while the source still
has that hash (a changed kernel reports null until it is captured again).  Every record must
resolve for the committed sources, name a workload that bench.py runs, and stop resolving when
its source changes.  `profiles/launch_shares.json` (the ncu launch list of the default bench
command) must have shares that sum to one.
"""
import hashlib
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _records():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_traffic_records_match_the_committed_sources():
    recs = _records()
    assert recs
    for r in recs:
        got = bench.traffic_record(r["kernel"], r["workload"])
        assert got == r["dram_bytes_per_launch"], (r["kernel"], r["workload"], "source changed since capture")
        assert got > 0
        assert "--clock-control none" in r["command"]


def test_traffic_records_name_benchmarked_workloads():
    names = {synth.config(n).name for n in range(1, 6)}
    names |= set(bench.TOPK_WORKLOADS.values())
    names |= {bench.COMBINE_COMPRESSED_WORKLOAD, bench.INSERT_WORKLOAD}
    assert set(bench.TOPK_WORKLOADS) == {"long-batch", "long-decode"}
    for r in _records():
        assert r["workload"] in names, r["workload"]


def test_traffic_record_is_null_once_the_source_changes(tmp_path, monkeypatch):
    # a copy of the repository layout bench.traffic_record reads, with one kernel source edited
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    recs = _records()
    r = recs[0]
    shutil.copy(os.path.join(ROOT, "profiles", "traffic.json"), root / "profiles" / "traffic.json")
    src = root / r["source"]
    src.parent.mkdir(parents=True)
    text = open(os.path.join(ROOT, r["source"]), "rb").read()
    src.write_bytes(text)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.traffic_record(r["kernel"], r["workload"]) == r["dram_bytes_per_launch"]
    src.write_bytes(text + b"\n// edited\n")
    assert hashlib.sha256(src.read_bytes()).hexdigest() != r["source_sha256"]
    assert bench.traffic_record(r["kernel"], r["workload"]) is None
    assert bench.traffic_record(r["kernel"], "a workload nobody captured") is None


def test_launch_shares_sum_to_one():
    with open(os.path.join(ROOT, "profiles", "launch_shares.json")) as f:
        d = json.load(f)
    shares = [k["share"] for k in d["kernels"].values()]
    assert abs(sum(shares) - 1.0) < 1e-6
    assert all(k["launches"] > 0 and k["avg_ns"] > 0 for k in d["kernels"].values())
    assert "--clock-control none" in d["command"]
