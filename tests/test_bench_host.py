"""Host-side logic of bench.py: the DRAM-traffic figure of the roofline
object comes from a committed ncu capture only while the captured kernel
source is the current one.

The source hash must cover every header the forward kernel is built from
(a change in any of them makes a new kernel); these tests follow the
kernel's quoted includes and check each is hashed, and check the three
outcomes of reading the capture data: current, stale, missing.
"""
import json
import os
import re

import bench

CSRC = os.path.join(bench.ROOT, "attention_attn_fwd_gb300", "csrc")


def local_includes(path, seen=None):
    """Quoted #include files reachable from `path` inside csrc."""
    seen = set() if seen is None else seen
    with open(path) as f:
        for name in re.findall(r'^#include "([^"]+)"', f.read(), re.M):
            inc = os.path.normpath(os.path.join(os.path.dirname(path), name))
            if os.path.dirname(inc) == CSRC and inc not in seen:
                seen.add(inc)
                local_includes(inc, seen)
    return seen


def test_hash_covers_every_kernel_header():
    kernel = os.path.join(CSRC, "attn_fwd_kernel.cuh")
    hashed = {os.path.normpath(os.path.join(bench.ROOT, rel))
              for rel in bench.KERNEL_SOURCES}
    needed = local_includes(kernel) | {kernel}
    assert needed <= hashed, sorted(needed - hashed)


def test_hash_changes_with_any_source(tmp_path, monkeypatch):
    copies = []
    for rel in bench.KERNEL_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        with open(os.path.join(bench.ROOT, rel), "rb") as f:
            dst.write_bytes(f.read())
        copies.append(dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    for dst in copies:
        data = dst.read_bytes()
        dst.write_bytes(data + b"\n")
        assert bench.kernel_source_hash() != h0, dst
        dst.write_bytes(data)
    assert bench.kernel_source_hash() == h0


def write_capture(path, source_hash, nbytes):
    path.write_text(json.dumps({"kernel_source_hash": source_hash,
                                "dram_bytes_per_launch": nbytes}))


def test_traffic_of_current_capture(tmp_path, monkeypatch):
    cap = tmp_path / "capture.json"
    write_capture(cap, bench.kernel_source_hash(), 123456)
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(cap))
    nbytes, source = bench.measured_traffic()
    assert nbytes == 123456
    assert bench.kernel_source_hash() in source


def test_stale_capture_gives_no_traffic(tmp_path, monkeypatch):
    cap = tmp_path / "capture.json"
    write_capture(cap, "0123456789abcdef", 123456)
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(cap))
    nbytes, reason = bench.measured_traffic()
    assert nbytes is None
    assert "0123456789abcdef" in reason


def test_missing_capture_gives_no_traffic(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE",
                        str(tmp_path / "absent.json"))
    assert bench.measured_traffic() == (None, "no capture data")


def test_committed_capture_is_well_formed():
    with open(bench.TRAFFIC_PROFILE) as f:
        d = json.load(f)
    assert d["dram_bytes_per_launch"] == (d["dram_bytes_read"] +
                                          d["dram_bytes_write"])
    assert re.fullmatch(r"[0-9a-f]{16}", d["kernel_source_hash"])
