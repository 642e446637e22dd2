"""The benchmark's recorded DRAM traffic (CPU only): each record is keyed to
the hash of the sources of the kernels it names, so an edit to one kernel's
file orphans only the records that cover that kernel."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def names(paths):
    return [os.path.basename(p) for p in paths]


def test_sources_follow_the_kernels_named():
    headers = ["decode_page.cuh", "pkv_device.cuh", "pkv_internal.h"]
    assert names(bench.kernel_sources("paged_decode_pagebox_kernel (fused step)")) == \
        ["decode_pagebox.cu"] + headers
    assert names(bench.kernel_sources("paged_decode_kernel+merge_plan_kernel (fused step)")) == \
        ["decode_attention.cu"] + headers
    assert names(bench.kernel_sources(
        "paged_decode_shared_kernel+paged_decode_pagebox_kernel+merge_plan_kernel")) == \
        ["decode_attention.cu", "decode_pagebox.cu", "decode_shared.cu"] + headers
    assert names(bench.kernel_sources(
        "paged_decode_shared_kernel+paged_decode_segments_kernel+merge_plan_kernel")) == \
        ["decode_attention.cu", "decode_segments.cu", "decode_shared.cu"] + headers
    assert set(names(bench.kernel_sources())) >= {"decode_attention.cu", "decode_pagebox.cu",
                                                   "decode_shared.cu", "decode_segments.cu"}


def test_hash_ignores_comments_and_separates_kernels(tmp_path, monkeypatch):
    for f in ("decode_attention.cu", "decode_pagebox.cu", "decode_shared.cu",
              "decode_segments.cu", "decode_page.cuh", "pkv_device.cuh", "pkv_internal.h"):
        (tmp_path / f).write_text(f"// {f}\nint {f.split('.')[0]}_x = 1;\n")
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES",
                        [str(tmp_path / f) for f in sorted({f for fs in bench.KERNEL_FILES.values()
                                                            for f in fs})])
    pagebox = "paged_decode_pagebox_kernel (fused step)"
    shared = "paged_decode_shared_kernel+paged_decode_pagebox_kernel+merge_plan_kernel (fused step)"
    h_pb, h_sh = bench.kernel_sha(pagebox), bench.kernel_sha(shared)
    (tmp_path / "decode_shared.cu").write_text("/* a comment */ int decode_shared_x = 1; // more\n")
    assert bench.kernel_sha(pagebox) == h_pb and bench.kernel_sha(shared) == h_sh
    (tmp_path / "decode_shared.cu").write_text("int decode_shared_x = 2;\n")
    assert bench.kernel_sha(pagebox) == h_pb     # another kernel's edit
    assert bench.kernel_sha(shared) != h_sh      # this record's kernel changed


def test_committed_records_are_well_formed():
    # a record whose kernel changed since its counters were taken reads as
    # null in the benchmark line (not an error): it resolves to its bytes or
    # to None, never to another record's
    with open(bench.TRAFFIC_FILE) as f:
        recs = json.load(f)
    assert {r["workload"] for r in recs} >= {"peak", "mix"}
    for r in recs:
        assert set(r) >= {"workload", "kernel", "kernel_sha", "dram_bytes_per_launch", "source"}
        assert r["dram_bytes_per_launch"] > 0 and len(r["kernel_sha"]) == 64
        assert bench.recorded_traffic(r["workload"], r["kernel"]) in (
            r["dram_bytes_per_launch"], None)
