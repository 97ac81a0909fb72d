"""The committed profile summaries stay what they claim to be.

Each summary under profiles/ is short text naming the command that made it;
every ncu command in it leaves the GPU clocks alone (--clock-control none)
and runs a committed entry point.  traffic.json holds per-launch DRAM
bytes only for kernels whose device code still hashes as recorded (bench.py
would report a stale record as null; here a stale record fails, so it is
re-captured or removed with the kernel change).
"""
import json
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
SUMMARIES = sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def test_profiles_hold_only_short_text():
    for f in os.listdir(PROFILES):
        assert f.endswith((".md", ".txt", ".json")), f
        assert os.path.getsize(os.path.join(PROFILES, f)) < 64 * 1024, f


@pytest.mark.parametrize("name", SUMMARIES)
def test_summary_names_its_command(name):
    with open(os.path.join(PROFILES, name), encoding="utf-8") as f:
        text = f.read()
    blocks = re.findall(r"```[a-z]*\n(.*?)```", text, flags=re.S)
    commands = [l.strip() for b in blocks for l in b.splitlines() if re.match(r"\s*ncu\s", l)]
    assert commands, "no ncu command in " + name
    for c in commands:
        assert "--clock-control none" in c, c
    # the profiled program is a committed entry point of the repository
    assert "python bench.py" in text
    assert "_work/" not in text


def test_traffic_records_are_current_and_per_launch():
    with open(os.path.join(PROFILES, "traffic.json")) as f:
        records = json.load(f)
    assert records
    for kernel, per_workload in records.items():
        assert kernel in bench.KERNEL_SOURCES, kernel
        for workload, r in per_workload.items():
            assert r["source_hash"] == bench.kernel_source_hash(kernel), (kernel, workload)
            assert r["dram_bytes_per_launch"] > 0
            assert "--clock-control none" in r["captured_with"]
