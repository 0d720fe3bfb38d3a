"""The committed ncu summaries that bench.py reads its DRAM traffic from were
taken on the current kernel sources (no GPU needed).

bench.py reports a scoring kernel's DRAM traffic per launch only while the
sha of that kernel's sources matches the one recorded in its summary under
profiles/; this test keeps the summaries from falling behind the sources
unnoticed, and checks that each summary gives the full command that made it.
"""
import os
import re

import bench


def test_every_profiled_workload_has_current_traffic():
    for workload, (name, sources) in bench.PROFILES.items():
        traffic, where = bench.profiled_traffic(workload)
        assert traffic is not None, f"{workload}: {where}"
        assert traffic > 0
        text = open(os.path.join(bench.ROOT, "profiles", name)).read()
        assert "--clock-control none" in text, name
        assert re.search(r"python bench\.py[^\n]*&& ncu ", text), name


def test_profiles_are_text_summaries_with_commands():
    pdir = os.path.join(bench.ROOT, "profiles")
    for name in os.listdir(pdir):
        assert name.endswith((".md", ".txt")), name
        text = open(os.path.join(pdir, name)).read()
        assert len(text) < 64 * 1024, name
        for cmd in re.findall(r"\bncu [^\n]*", text):
            if "--metrics" in cmd or "--set" in cmd:
                assert "--clock-control none" in cmd, (name, cmd)
