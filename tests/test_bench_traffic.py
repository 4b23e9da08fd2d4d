"""The `traffic` of bench.py's roofline comes from a recorded ncu capture
(profiles/traffic_<workload>.txt) only while the persistent kernel's sources
and the launch knobs are the ones the capture was taken with; otherwise the
line reports null rather than a stale figure."""
import os
import sys

import bench

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
import moe_inputs as mi  # noqa: E402


def _record(key):
    rec = {}
    with open(os.path.join(os.path.dirname(HERE), "profiles", f"traffic_{key}.txt")) as fh:
        for line in fh:
            parts = line.split(None, 1)
            if len(parts) == 2 and not line.startswith("#"):
                rec[parts[0]] = parts[1].strip()
    return rec


def _default_cfg(name, monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    return bench.workload_config(mi.CONFIGS[name], bench.parse_args())


def test_records_describe_the_default_launch(monkeypatch):
    for name, key in (("dsv3", "dsv3_bf16"), ("dsv3_mxfp8", "dsv3_mxfp8_mxfp8")):
        rec = _record(key)
        cfg = _default_cfg(name, monkeypatch)
        for k in ("minibatch", "ring_slots", "gather_ctas", "mma_pair", "raster", "dispatch", "pad_odd_tiles",
                  "gemm_ctas"):
            assert rec[k] == str(cfg[k]), (key, k)
        assert int(rec["dram_bytes_per_launch"]) == int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])


def test_figure_only_for_the_recorded_sources_and_knobs(monkeypatch):
    rec = _record("dsv3_bf16")
    cfg = _default_cfg("dsv3", monkeypatch)
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: rec["sources_sha256"])
    traffic, _ = bench.recorded_traffic("dsv3_bf16", cfg)
    assert traffic == float(rec["dram_bytes_per_launch"])
    # another launch configuration
    assert bench.recorded_traffic("dsv3_bf16", {**cfg, "minibatch": 4096}) == (None, None)
    assert bench.recorded_traffic("dsv3_bf16", {**cfg, "pad_odd_tiles": 1}) == (None, None)
    # other kernel sources
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: "0" * 64)
    assert bench.recorded_traffic("dsv3_bf16", cfg) == (None, None)
    # no record at all
    assert bench.recorded_traffic("no_such_workload", cfg) == (None, None)


def test_source_hash_covers_the_persistent_kernel_only():
    # the hash reads exactly TRAFFIC_SOURCES and the C header, in that order
    import hashlib
    root = os.path.dirname(HERE)
    h = hashlib.sha256()
    for f in [os.path.join(root, "routing_grouped_expert_gemm_gb300", "csrc", s) for s in bench.TRAFFIC_SOURCES] + \
            [os.path.join(root, "include", "moe.h")]:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    assert bench.kernel_sources_hash() == h.hexdigest()
    assert "megakernel.cu" in bench.TRAFFIC_SOURCES and "router.cu" not in bench.TRAFFIC_SOURCES
