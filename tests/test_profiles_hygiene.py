"""The committed ncu summaries: short text, each with the command that made
it, and that command runs committed files only (with the argument choices
those files accept)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROF = os.path.join(ROOT, "profiles")


def _tracked():
    try:
        out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True,
                             check=True).stdout
    except (OSError, subprocess.CalledProcessError):
        pytest.skip("not a git checkout")
    return set(out.split())


def _summaries():
    return sorted(f for f in os.listdir(PROF) if not f.startswith("."))


def test_profiles_are_short_text():
    for f in _summaries():
        assert f.endswith((".md", ".txt")), f
        assert os.path.getsize(os.path.join(PROF, f)) < 32 * 1024, f


def test_every_capture_names_its_command_and_runs_committed_files():
    tracked = _tracked()
    cases = {"lm_head", "step", "target", "sampling"}
    for f in _summaries():
        txt = open(os.path.join(PROF, f)).read()
        scripts = re.findall(r"python ([\w./-]+\.py)", txt)
        joined = re.sub(r"\\\n\s*", " ", txt)  # shell line continuations
        # commands sit in indented blocks (prose may name ncu options too)
        ncu_cmds = re.findall(r"^\s+(?:.*&&\s*)?ncu\s+-[^\n]*", joined, re.M)
        if ncu_cmds:
            assert scripts, f"{f}: no command"
        for cmd in ncu_cmds:
            assert "--clock-control none" in cmd, f"{f}: ncu without --clock-control none"
        for s in scripts:
            assert s in tracked, f"{f}: {s} is not a committed file"
        for case in re.findall(r"python profile_cases\.py (\w+)", txt):
            assert case in cases, f"{f}: unknown case {case}"
