"""Every bench command that a summary under profiles/ says it was made with
still runs (the plain run before each ncu capture), so the summaries can be
reproduced from the committed files."""

import glob
import json
import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _commands():
    cmds = set()
    for f in glob.glob(os.path.join(ROOT, "profiles", "*")):
        text = open(f).read()
        for m in re.finditer(r"python bench\.py ([^>\\&\"\n]*)", text):
            cmds.add(m.group(1).strip())
    return sorted(cmds)


COMMANDS = _commands()


def test_profiles_name_commands():
    assert len(COMMANDS) >= 10


@pytest.mark.parametrize("args", COMMANDS)
def test_profile_command_runs(args):
    r = subprocess.run([sys.executable, "bench.py", *args.split()], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert lines, r.stdout[-2000:]
    json.loads(lines[-1])
