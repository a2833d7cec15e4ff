"""The DRAM traffic the benchmark reports beside its rooflines comes from a
table of one ncu capture per kernel; every entry must match the recorded
capture (the profile summary's table, scaled to the full layer) and carry
the digest of the kernel source it was taken on, so that a changed kernel
reports no traffic instead of a stale one (no GPU needed)."""
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUMMARY = os.path.join(ROOT, "profiles", "dram_traffic_qwen3_8b_16k.md")
KERNELS = {"attention": "attn_kernel", "summary_scan": "scan_kernel",
           "topk_select": "select_kernel", "prefetch": "gather_kernel"}


def summary_rows():
    rows = {}
    for line in open(SUMMARY):
        m = re.match(r"\| `(\w+)[^`]*` \| ([\d,]+) B \| ([\d,]+) B \|.*\| ([\d,]+) B \|", line)
        if m:
            rd, wr, full = (int(x.replace(",", "")) for x in m.group(2, 3, 4))
            rows[m.group(1)] = (rd, wr, full)
    return rows


def test_table_matches_the_recorded_capture():
    rows = summary_rows()
    table = bench.PROFILED_TRAFFIC["qwen3_8b_16k"]
    assert set(table) == set(KERNELS)
    for name, (nbytes, digest) in table.items():
        rd, wr, full = rows[KERNELS[name]]
        assert full == 2 * (rd + wr)          # 64 requests captured, 128 reported
        assert nbytes == full
        assert digest in open(SUMMARY).read()


def test_traffic_is_null_once_the_kernel_source_changes(monkeypatch):
    table = bench.PROFILED_TRAFFIC["qwen3_8b_16k"]
    for name, (nbytes, digest) in table.items():
        current = bench.source_digest(bench.KERNEL_SOURCES[name])
        want = nbytes if current == digest else None
        assert bench.profiled_traffic("qwen3_8b_16k", name) == want
    monkeypatch.setattr(bench, "source_digest", lambda _: "0" * 16)
    assert all(bench.profiled_traffic("qwen3_8b_16k", n) is None for n in table)
    assert bench.profiled_traffic("llama31_8b_32k", "attention") is None
