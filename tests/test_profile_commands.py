"""The ncu summaries under profiles/ each give the command that produced them; those commands must
keep running the committed bench.py (every flag still accepted) and must leave the GPU clocks
alone (`--clock-control none`)."""
import glob
import os
import re
import shlex
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _commands():
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for block in re.findall(r"```\n(.*?)```", open(path).read(), re.S):
            cmd = " ".join(block.replace("\\\n", " ").split())
            if cmd.startswith("ncu "):
                yield os.path.basename(path), cmd


def test_every_summary_records_its_command():
    names = {name for name, _ in _commands()}
    assert names == {os.path.basename(p) for p in glob.glob(os.path.join(ROOT, "profiles", "*.md"))}


def test_profile_commands_leave_clocks_alone():
    for name, cmd in _commands():
        assert "--clock-control none" in cmd, name


def test_profile_commands_parse_with_the_committed_bench(monkeypatch):
    n = 0
    for name, cmd in _commands():
        assert "python bench.py" in cmd, name
        args = shlex.split(cmd.split("python bench.py", 1)[1])
        monkeypatch.setattr(sys, "argv", ["bench.py"] + args)
        bench.parse()   # an unknown flag exits here
        n += 1
    assert n >= 5
