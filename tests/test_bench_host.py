"""Host logic of bench.py that needs no GPU: the per-kernel source hash and
the lookup of committed ncu traffic records."""
import json
import os
import sys

from tests.conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402

CSRC = os.path.join(ROOT, "tensor_transformer_linear_tma_b300", "csrc")


def test_source_hash_covers_the_named_files_only():
    every = sorted(os.listdir(CSRC))
    assert bench.kernel_source_sha() == bench.kernel_source_sha(every)
    some = ["tp_gemm.cuh", "tp_ptx.cuh"]
    assert bench.kernel_source_sha(some) == bench.kernel_source_sha(list(reversed(some)))  # order-free
    assert bench.kernel_source_sha(some) != bench.kernel_source_sha(every)
    assert len(bench.kernel_source_sha(some)) == 16


def test_traffic_records_are_well_formed():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    records = {k: v for k, v in d.items() if isinstance(v, dict)}
    assert records
    for key, rec in records.items():
        assert ":" in key
        assert all(os.path.exists(os.path.join(CSRC, f)) for f in rec["source_files"]), key
        assert len(rec["source_sha"]) == 16 and rec["T"] >= 1 and rec["dram_bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(ROOT, "profiles", rec["summary"])), key


def test_traffic_lookup_needs_the_same_token_count_and_sources():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    key, rec = next((k, v) for k, v in d.items() if isinstance(v, dict))
    workload, kernel = key.split(":", 1)
    assert bench.ncu_traffic(kernel, workload, rec["T"] + 1) is None
    assert bench.ncu_traffic("no such kernel", workload, rec["T"]) is None
    fresh = rec["source_sha"] == bench.kernel_source_sha(rec["source_files"])
    assert (bench.ncu_traffic(kernel, workload, rec["T"]) == rec["dram_bytes_per_launch"]) == fresh
