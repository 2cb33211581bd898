"""The ncu summaries under profiles/ name the command that made each of them,
and that command must run committed files only: every ncu line keeps the GPU
clocks as found (--clock-control none) and every bench.py invocation parses
with the current bench.py arguments."""
import glob
import os
import re
import shlex
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*")))


def _commands(text):
    """Shell commands inside fenced blocks, continuation lines joined."""
    cmds = []
    for block in re.findall(r"```[a-z]*\n(.*?)```", text, re.S):
        for cmd in block.replace("\\\n", " ").splitlines():
            if cmd.strip():
                cmds.append(cmd.strip())
    return cmds


def test_profiles_are_short_text_summaries():
    assert PROFILES, "no profile summaries"
    for p in PROFILES:
        assert p.endswith((".md", ".txt")), p
        assert os.path.getsize(p) < 16 * 1024, p


@pytest.mark.parametrize("path", PROFILES, ids=os.path.basename)
def test_profile_commands_run_committed_files(path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    text = open(path).read()
    cmds = [c for c in _commands(text) if c.startswith("ncu ")]
    assert cmds, f"{path}: no ncu command recorded"
    for cmd in cmds:
        argv = shlex.split(cmd)
        assert "--clock-control" in argv and argv[argv.index("--clock-control") + 1] == "none", cmd
        assert "_work" not in cmd and "/root/" not in cmd, cmd
        i = argv.index("bench.py")
        assert argv[i - 1] == "python", cmd
        monkeypatch.setattr(sys, "argv", ["bench.py"] + argv[i + 1:])
        bench.parse()                                  # exits (SystemExit) on an unknown flag or choice
