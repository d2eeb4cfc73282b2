"""The ncu summaries under profiles/ are short text files, each naming the
command that produced it; those commands run committed files only (the
benchmark), never scratch scripts or a profiler's raw output folder."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _summaries():
    return sorted(os.path.join(PROFILES, f) for f in os.listdir(PROFILES))


def test_profiles_are_short_text():
    for p in _summaries():
        assert p.endswith((".md", ".txt")), p
        assert os.path.getsize(p) < 16 * 1024, p


def test_each_summary_names_its_command_and_runs_committed_files():
    for p in _summaries():
        text = open(p).read()
        cmds = re.findall(r"^\s*#?\s*(?:ncu|python) .*$", text, flags=re.M)
        assert any("ncu " in c for c in cmds), f"{p}: no ncu command"
        assert any("bench.py" in c for c in cmds), f"{p}: no benchmark command"
        for c in cmds:
            assert "_work" not in c, f"{p}: {c}"
            m = re.search(r"python (\S+\.py)", c)
            if m:
                assert os.path.exists(os.path.join(ROOT, m.group(1))), f"{p}: {m.group(1)}"
