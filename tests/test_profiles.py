"""The committed ncu summaries: every JSON block that bench.py may read for
its roofline traffic parses and names a known workload, a source hash and a
positive byte count. (Whether an entry is current -- its hash equal to the
sources' hash now -- is bench.py's business: a stale entry gives null
traffic there, never a wrong number.)"""
import glob
import json
import os
import re

import pytest

import bench
from exact_attention_forward_14_b300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _entries():
    out = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            text = f.read()
        for block in re.findall(r"```json\n(.*?)```", text, flags=re.S):
            # traffic entries only (other summaries keep other JSON)
            if "dram_bytes_per_launch" in block:
                out.append((os.path.basename(path), block))
    return out


def test_profiles_hold_traffic_entries():
    assert len(_entries()) >= 8


@pytest.mark.parametrize("name,block", _entries(), ids=lambda x: x if isinstance(x, str) and x.endswith(".md") else "")
def test_traffic_entry_is_well_formed(name, block):
    entry = json.loads(block)
    assert entry["workload"] in inputs.WORKLOADS, name
    assert re.fullmatch(r"[0-9a-f]{16}", entry["kernel_hash"]), name
    assert isinstance(entry["dram_bytes_per_launch"], int) and entry["dram_bytes_per_launch"] > 0, name


def test_no_workload_has_two_entries_for_one_hash():
    seen = set()
    for name, block in _entries():
        entry = json.loads(block)
        key = (entry["workload"], entry["kernel_hash"])
        assert key not in seen, f"{name}: a second entry for {key}"
        seen.add(key)


def test_backward_and_d256_entries_use_their_own_source_lists():
    """bench.py hashes the backward over its kernels plus the host file that
    launches them side by side, and d = 256 over its kernel plus the main
    kernel's helpers: entries for those workloads must carry hashes of those
    source lists (checked by recomputing the hash of the current sources for
    the entries that are current, and by format for the rest)."""
    now = {
        "bwd": bench.kernel_source_hash(bench.KERNEL_SOURCES_BWD),
        "d256": bench.kernel_source_hash(bench.KERNEL_SOURCES_D256),
        "fwd": bench.kernel_source_hash(bench.KERNEL_SOURCES),
    }
    for name, block in _entries():
        entry = json.loads(block)
        w = entry["workload"]
        kind = "bwd" if w.startswith("bwd_") else ("d256" if w.startswith("d256") else "fwd")
        others = {k: v for k, v in now.items() if k != kind}
        assert entry["kernel_hash"] not in others.values(), (
            f"{name}: {w} carries the hash of another kernel's sources")
