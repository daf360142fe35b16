"""Every ncu summary under profiles/ states the command that produced it; the
bench.py invocations in those commands must still parse with bench.py's
current options, so a summary never points at a flag that no longer exists."""
import glob
import os
import re
import shlex

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench_invocations(text: str):
    joined = re.sub(r"\\\n\s*", " ", text)  # shell line continuations
    for m in re.finditer(r"python bench\.py([^>`\n]*)", joined):
        yield shlex.split(m.group(1).replace("&&", " "))


def test_profile_commands_parse():
    found = 0
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            text = f.read()
        invocations = list(_bench_invocations(text))
        assert invocations, f"{os.path.basename(path)} names no bench.py command"
        for argv in invocations:
            bench.build_parser().parse_args(argv)
            found += 1
    assert found >= 5
