"""bench.py host logic: committed DRAM-traffic figures are reported only for the kernel
sources they were measured on; NUMA placement of host buffers.  No GPU."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_every_timed_kernel_lists_existing_sources():
    for kernel in bench.KERNEL_SOURCES:
        files = bench.kernel_sources(kernel)
        assert files[-1] == "include/kvo.h"
        for rel in files:
            assert os.path.isfile(os.path.join(ROOT, rel)), rel


def test_traffic_is_reported_only_for_the_measured_sources(tmp_path, monkeypatch):
    path = tmp_path / "traffic.json"
    entry = {"bytes_per_launch": 123456, "workload": "w",
             "source_hash": bench.kernel_source_hash("attend")}
    path.write_text(json.dumps({"attend": entry}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.load_traffic("attend", "w") == 123456.0
    assert bench.load_traffic("attend", "other workload") is None
    assert bench.load_traffic("fused", "w") is None  # no entry
    entry["source_hash"] = "0" * 16  # taken on other sources
    path.write_text(json.dumps({"attend": entry}))
    assert bench.load_traffic("attend", "w") is None


def test_a_kernel_hash_follows_only_its_own_sources():
    # the attention kernel's hash does not cover the step kernels' files
    assert "top_cache_gb300/csrc/kvo_fused.cuh" not in bench.kernel_sources("attend")
    assert "top_cache_gb300/csrc/kvo_attend.cu" not in bench.kernel_sources("fused")
    # kernels built from different files have different hashes (the append and gather
    # kernels share one translation unit, hence one hash)
    hashes = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    for a in hashes:
        for b in hashes:
            if sorted(bench.KERNEL_SOURCES[a]) != sorted(bench.KERNEL_SOURCES[b]):
                assert hashes[a] != hashes[b], (a, b)


def test_committed_entries_name_their_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for kernel, e in t.items():
        if kernel.startswith("_"):
            continue
        assert e["sources"] == bench.kernel_sources(kernel)
        assert e["bytes_per_launch"] > 0 and len(e["source_hash"]) == 16


def test_numa_spread_of_a_host_buffer():
    import numpy as np
    buf = np.ones(1 << 20, dtype=np.uint8)
    spread = bench.numa_spread(buf.ctypes.data)
    if spread is not None:  # /proc/self/numa_maps readable
        assert all(k.startswith("N") for k in spread)
        assert abs(sum(spread.values()) - 1.0) < 1e-3


def test_timed_region_profiles_the_roofline_kernels_only():
    # the kinds bracketed with events inside the timed region are names the library
    # profiles, and the mask passed to KVO_OPT_PROFILE_KINDS has exactly their bits
    from top_cache_gb300 import kvo as K
    for name in bench.TIMED_KINDS:
        assert name in K.PROF_KINDS
    mask = bench._kinds_mask(bench.TIMED_KINDS)
    assert mask == sum(1 << K.PROF_KINDS.index(n) for n in ("score", "gather", "fused"))
    assert 0 < mask < (1 << len(K.PROF_KINDS))
    # the committed figures cover the default workload's dominant kernels
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for kernel in ("score", "gather"):
        assert t[kernel]["workload"] == bench.DEFAULT_WORKLOAD
