"""The bench's roofline.traffic comes from the committed ncu record only while
the prefill kernels' sources are the ones it was measured on."""

import json
import os

import bench


def test_traffic_record_is_used_only_for_the_sources_it_was_measured_on(monkeypatch):
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["prefill_T16384"]
    assert rec["dram_bytes_per_launch"] > 0
    monkeypatch.setattr(bench, "prefill_source_digest", lambda: rec["source_sha256_16"])
    assert bench.traffic_record() == rec["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "prefill_source_digest", lambda: "0" * 16)
    assert bench.traffic_record() is None


def test_the_source_digest_covers_every_prefill_kernel_source():
    csrc = os.path.join(bench.ROOT, "gated_deltanet_scan_gb300", "csrc")
    for name in bench.PREFILL_SOURCES:
        assert os.path.isfile(os.path.join(csrc, name)), name
    assert {"gdr_factor.cu", "gdr_prefill_tc.cu"} <= set(bench.PREFILL_SOURCES)
    assert len(bench.prefill_source_digest()) == 16
