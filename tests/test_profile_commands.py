"""Every ncu summary under profiles/ states the command that produced it; those commands must
still run committed files with options the benchmark accepts (checked here without running them)."""
import glob
import os
import re
import shlex

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _bench_commands(path):
    cmds = []
    for line in open(path):
        m = re.search(r"python (bench\.py[^&\\]*)", line)
        if m:
            cmds.append(shlex.split(m.group(1))[1:])
    return cmds


def test_there_are_profiles():
    assert len(PROFILES) >= 4


@pytest.mark.parametrize("path", PROFILES, ids=[os.path.basename(p) for p in PROFILES])
def test_profile_commands_parse(path):
    import bench
    cmds = _bench_commands(path)
    assert cmds, f"{os.path.basename(path)} gives no bench.py command"
    for argv in cmds:
        bench.parse_args(argv)  # exits (SystemExit) on an unknown or invalid option
    text = open(path).read()
    assert "--clock-control none" in text, "every ncu command must leave the GPU clocks alone"
