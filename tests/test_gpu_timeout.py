"""A bounded device-side wait that gives up is reported as a timeout, not as bad data.

The staged walk has a test hook, off unless SPEC_VERIFY_TEST_STALL names a batch row:
that row's first bulk copy is announced on its mbarrier (expect_tx) but never issued,
and its wait is bounded to 50 us instead of a quarter of a second.  With one CTA per
row (SPEC_VERIFY_CLUSTER=1) no copy is in flight for that row and no cluster peer is
involved, so the wait simply runs out and the kernel returns: the row gets count -1
and the call's row status is SV_ERR_TIMEOUT, while the other rows are unaffected.
The library reads these variables once, so each case runs in a child process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("row", [1, 2])  # a sampling row, a greedy row
def test_stalled_copy_reports_timeout(row):
    env = dict(os.environ, SPEC_VERIFY_PATH="staged", SPEC_VERIFY_CLUSTER="1", SPEC_VERIFY_TEST_STALL=str(row))
    res = subprocess.run([sys.executable, os.path.join(HERE, "_stall_check.py")], env=env, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert res.stdout.strip().endswith("ok")
