"""The committed profiling evidence (profiles/) is consistent with itself and
with the rules it was taken under: every ncu command leaves the GPU clocks
alone (--clock-control none), and every recorded DRAM traffic figure is the
algorithmic traffic of its workload (W and h read once, outputs written)
within 2%, i.e. no kernel re-reads W from HBM.  Host-only: reads text files.
"""

import glob
import json
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
SHAPES = {"llama3_8b": (4096, 128256)}


def _ncu_commands(text):
    """ncu command lines (a trailing backslash continues a command)."""
    out, cur = [], None
    for line in text.splitlines():
        s = line.strip()
        if cur is not None:
            cur += " " + s.rstrip("\\")
            if not s.endswith("\\"):
                out.append(cur)
                cur = None
            continue
        m = re.search(r"(?:^|\s|`)(ncu\s+--|ncu\s+-)", s)
        if m and ("--metrics" in s or "--set" in s or "--section" in s or "(same sections)" in s):
            if s.endswith("\\"):
                cur = s.rstrip("\\")
            else:
                out.append(s)
    return out


def test_every_ncu_command_keeps_the_clocks():
    files = sorted(glob.glob(os.path.join(PROFILES, "*.md")))
    assert files, "no profile summaries"
    seen = 0
    for path in files:
        for cmd in _ncu_commands(open(path).read()):
            seen += 1
            assert "--clock-control none" in cmd, (os.path.basename(path), cmd)
    assert seen >= 5


def test_recorded_traffic_is_the_algorithmic_traffic():
    records = json.load(open(os.path.join(PROFILES, "traffic.json")))
    assert set(k.split("@")[0] for k in records) == set(bench.KERNEL_SOURCES)
    for key, rec in records.items():
        kernel, workload = key.split("@")
        m = re.fullmatch(r"(\w+?)_B(\d+)", workload)
        assert m and m.group(1) in SHAPES, key
        d, V = SHAPES[m.group(1)]
        B = int(m.group(2))
        algo = bench.algorithmic_bytes(B, d, V)
        assert rec["dram_bytes_per_launch"] == rec["dram_read"] + rec["dram_write"], key
        assert abs(rec["dram_bytes_per_launch"] / algo - 1) < 0.02, (key, rec["dram_bytes_per_launch"], algo)
        assert "--clock-control none" in rec["command"], key
        assert re.fullmatch(r"[0-9a-f]{64}", rec["source_sha256"]), key


@pytest.mark.parametrize("kernel", sorted(bench.KERNEL_SOURCES))
def test_kernel_source_lists_exist(kernel):
    """The files whose hash keys a kernel's traffic record all exist (a renamed
    header would otherwise silently drop out of the key)."""
    for f in bench.KERNEL_SOURCES[kernel]:
        assert os.path.exists(os.path.join(bench._CSRC, f)), (kernel, f)
