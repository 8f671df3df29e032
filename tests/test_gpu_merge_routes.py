"""Split units whose rows are merged by different routes within one M tile.

A unit split between two CTAs is merged in the epilogue of the piece that
finishes last: straight from its TMEM accumulator when the other piece has
already published (directly, or through shared memory at the end of a
slice), else by publishing and, if its arrival completes the row's count,
merging from memory.  Each warp decides from its own rows' arrival counters,
so the warps of one M tile can take different routes when the other piece is
still publishing.  The development build (-DTV_TEST_HOOKS) can keep the warps
of chosen TMEM quarters off the direct merge, which makes that mix happen on
every split row; the results must be the same bits as with the normal routes
and match the oracle.  At the end of a slice the last piece stages the
other piece's rows through the idle K/V ring; with four tail warps, whose
two pairs take tiles in turn, the ring is idle only once both pairs have
read their last tiles: the development build can slow the first pair down
(it sleeps before each of its tiles), and the results must again be the same
bits.  The calls run in a child process that loads the development build in
place of the product library.
"""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_mixed_merge_routes_give_the_same_bits():
    from speculative_decoding_tree_attn_gb300 import build as B

    lib = B.build(dev=True)
    env = dict(os.environ, TREEVERIFY_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "route_child.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert {x["shape"] for x in lines} == {"one_m_tile", "two_m_tiles", "tail_rows", "tail_rows_slow_pair"}, r.stdout
    assert len(lines) == 16, r.stdout
    for x in lines:
        assert x["bit_identical"], x
        assert x["err"] <= x["tol"], x
