"""The bounded waits of the tensor-core attention kernels, run out on purpose.

Every pipeline wait of those kernels gives up after a time limit, sets
TV_DEV_TIMEOUT in the status word, lets its MMAs and TMA loads complete,
frees TMEM and returns.  The development build of the library
(-DTV_TEST_HOOKS, built here into _build/dev) lets a test shorten that limit
and have CTA 0 withhold the TMA loads of one ring tile, so that the waits on
that tile run out: no fault, no trap, nothing left waiting.  The calls run in
a child process that loads the development build in place of the product
library; the test checks that each kernel shape reported the timeout and that
the next call on the same stream, hook off, matches the oracle.
"""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_timeout_exit_reports_and_leaves_the_context_usable():
    from speculative_decoding_tree_attn_gb300 import build as B
    from speculative_decoding_tree_attn_gb300 import capi

    lib = B.build(dev=True)
    env = dict(os.environ, TREEVERIFY_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "timeout_child.py")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert [x["shape"] for x in lines] == ["one_m_tile", "two_m_tiles", "tail_rows"], r.stdout
    for x in lines:
        assert x["status"] & capi.TV_DEV_TIMEOUT, x
        assert x["err_after"] <= x["tol"], x
