"""The checked build (FORK_ATTN_CHECKED): an out-of-range page id in an uploaded plan is
reported through the device error word and never dereferenced.  Run in a child process so
that this process keeps the plain library; only the checked library ever sees the
corrupted plan."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_corrupted_page_id_is_caught_by_the_checked_build():
    from shared_prefix_paged_attn_b300 import build
    build.build(checked=True)
    env = dict(os.environ, FORK_ATTN_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_plan_corruption.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [x for x in r.stdout.splitlines() if x.startswith("ok")]
    assert len(lines) == 2, r.stdout
