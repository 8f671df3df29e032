"""Library checks that need no GPU: the shared library loads, exports every
symbol include/treeverify.h declares, the host tree builder matches the
oracle bit for bit, and argument errors are reported without touching a
device."""

import os
import re

import numpy as np
import pytest

from oracle import tree as T
from speculative_decoding_tree_attn_gb300 import build as B
from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "treeverify.h")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not os.path.exists(capi.LIB_PATH):
        B.build()
    return capi.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    syms = declared_symbols()
    assert len(syms) >= 10
    h = capi.lib()
    for s in syms:
        assert hasattr(h, s), s
    assert set(syms) == set(capi.SIGNATURES), "binding and header disagree"


def test_version():
    assert capi.tv_version() >= 100


def test_tree_build_matches_oracle():
    rng = np.random.default_rng(30)
    cases = [W.PAGE_TREE_PATHS, [], [(0,), (0,), (1,)]]
    for _ in range(60):
        n = int(rng.integers(1, 65))
        paths = W.random_rank_paths(n, int(rng.integers(1, 10)), rng)
        order = rng.permutation(len(paths))
        cases.append([paths[i] for i in order])
    for paths in cases:
        parent, depth, mask, p2n, n = capi.tv_tree_build(paths)
        op, od, orows, onode = T.build_tree(paths)
        assert n == op.size
        np.testing.assert_array_equal(parent, op)
        np.testing.assert_array_equal(depth, od)
        np.testing.assert_array_equal(mask, np.array(orows, dtype=np.uint64))
        np.testing.assert_array_equal(p2n, [onode[tuple(p)] for p in paths])


def test_tree_build_errors():
    with pytest.raises(capi.TVError) as e:
        capi.tv_tree_build([(0,), (1, 1)])
    assert e.value.code == -2
    with pytest.raises(capi.TVError) as e:
        capi.tv_tree_build([(k,) for k in range(64)])
    assert e.value.code == -3
    with pytest.raises(capi.TVError) as e:
        capi.tv_tree_build([(0,), (-1,)])
    assert e.value.code == -1
    parent, depth, mask, p2n, n = capi.tv_tree_build([(k,) for k in range(63)])
    assert n == 64 and int(mask[63]) == (1 << 63) | 1


def test_device_entry_points_reject_bad_sizes_on_host():
    h = capi.lib()
    assert h.tv_tree_mask(None, 0, None, None, 1, 65, None, None, None, None, None) == -1
    assert h.tv_tree_mask(None, 0, None, None, 0, 10, None, None, None, None, None) == 0
    assert h.tv_rope_apply(None, None, None, None, 10, 1, 1, 1, 1, 60, 1, None, None) == -1
    assert h.tv_tree_accept_greedy(None, None, None, None, 0, None, 1, 65, 10, None, None, None, 4, None, None) == -1
    assert h.tv_tree_accept_sample(None, None, None, None, 0, None, None, None, 0, 10, 10, None, None, None, 4,
                                   0, None, 0, None, None) == 0
    assert b"bad sizes" in h.tv_last_error() or h.tv_last_error() == b""
    assert h.tv_tree_accept_sample(None, None, None, None, 0, None, None, None, 0, 10, 10, None, None, None, 4,
                                   5, None, 0, None, None) == -1
    assert b"unknown flags" in h.tv_last_error()
    assert h.tv_chain_accept_sample(None, None, None, None, None, None, 0, 3, 10, None, None, 4, 5, None, 0, None,
                                    None) == -1
    assert b"unknown flags" in h.tv_last_error()
    # the grid sampler's workspace: a 16-byte state per request, and 16 bytes per request and
    # 4096-entry chunk
    assert h.tv_accept_sample_workspace_size(256, 10, 128000) == 16 * 256 + 16 * 256 * 32
    assert h.tv_accept_sample_workspace_size(3, 2, 4097) == 16 * 3 + 16 * 3 * 2
    assert h.tv_accept_sample_workspace_size(0, 2, 100) == 0


def test_tree_prepare_rejects_bad_arguments_on_host():
    """tv_tree_prepare checks its sizes, rotation arguments and head_dim
    before any launch (fake non-null pointers are never touched)."""
    import ctypes
    h = capi.lib()
    fake = ctypes.c_void_p(256)
    tb = fake  # stands for every device buffer
    # N past the 64-node limit; B = 0 is a no-op
    assert h.tv_tree_prepare(None, 0, None, None, 1, 65, None, None, None, None, 0, None, 0, 128, 1, None, 16,
                             None, None) == -1
    assert b"bad sizes" in h.tv_last_error()
    assert h.tv_tree_prepare(None, 0, None, None, 0, 10, None, None, None, None, 0, None, 0, 128, 1, None, 16,
                             None, None) == 0
    # Q given without query heads, or without a table
    assert h.tv_tree_prepare(tb, 10, tb, None, 2, 10, tb, tb, tb, fake, 0, None, 0, 128, 1, tb, 16, None,
                             None) == -1
    assert b"rotation needs" in h.tv_last_error()
    assert h.tv_tree_prepare(tb, 10, tb, None, 2, 10, tb, tb, tb, fake, 4, fake, 2, 128, 1, None, 16, None,
                             None) == -1
    assert b"rotation needs" in h.tv_last_error()
    # a head_dim the rotation does not take
    assert h.tv_tree_prepare(tb, 10, tb, None, 2, 10, tb, tb, tb, fake, 4, fake, 2, 48, 1, tb, 16, None,
                             None) == -4  # TV_ERR_UNSUPPORTED
    assert b"head_dim 48" in h.tv_last_error()

