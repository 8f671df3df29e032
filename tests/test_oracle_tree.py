"""Pins for the oracle's tree structure (CPU only).

Each test ties ``oracle.tree`` to something other than itself: rows printed
on the mask page, the page's per-depth path products, the empty tree, the
missing-parent rejection, and a brute-force characterisation of ancestry
(node j is an ancestor-or-self of node i exactly when j's rank path is a
prefix of i's)."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import tree as T
from speculative_decoding_tree_attn_gb300 import workloads as W


def test_page_mask_rows(mask_facts):
    parent, depth, rows, _ = T.build_tree(W.PAGE_TREE_PATHS)
    assert parent.size == int(mask_facts["tree_verified"][0][0])
    for vals in mask_facts["mask_row"]:
        i, cols = int(vals[0]), {int(c) for c in vals[1:]}
        got = {j for j in range(parent.size) if (rows[i] >> j) & 1}
        assert got == cols, (i, got, cols)


def test_page_tree_depth_terms(mask_facts):
    """The example tree's per-depth path products are exactly the page's."""
    parent, depth, rows, node_of = T.build_tree(W.PAGE_TREE_PATHS)
    r = [float(x) for x in mask_facts["rank_probs"][0]]
    by_depth = {}
    for path in W.PAGE_TREE_PATHS:
        by_depth.setdefault(len(path), []).append(W.path_value(path, r))
    for vals in mask_facts["tree_depth_terms"]:
        d = int(vals[0])
        want = sorted(Fraction(v) for v in vals[1:])
        assert sorted(by_depth[d]) == want
    total = 1 + sum(sum(v) for v in by_depth.values())
    assert round(float(total), 2) == float(mask_facts["tree_expected_tokens"][0][0])
    chain = 1 + sum(Fraction(r[0]).limit_denominator(10**6) ** k for k in range(1, 5))
    assert round(float(chain), 2) == float(mask_facts["chain_expected_tokens"][0][0])


def test_empty_tree_is_one_node(mask_facts):
    parent, depth, rows, node_of = T.build_tree([])
    assert parent.tolist() == [-1] and depth.tolist() == [0]
    assert T.dense_mask(rows, 1).tolist() == [[True]]
    assert parent.size == int(mask_facts["empty_tree_nodes"][0][0])


@pytest.mark.parametrize("paths", [[(0, 1)], [(0,), (1, 1)], [(0,), (0, 0, 0)]])
def test_missing_parent_rejected(paths):
    with pytest.raises(T.MissingParentError):
        T.build_tree(paths)


def test_negative_rank_rejected():
    with pytest.raises(ValueError):
        T.build_tree([(0,), (-1,)])


def test_duplicates_and_order():
    parent, depth, rows, node_of = T.build_tree([(1, 0), (0,), (1,), (0,), (0, 0), ()])
    assert T.canonical_paths([(1, 0), (0,), (1,), (0, 0)]) == [(0,), (1,), (0, 0), (1, 0)]
    assert parent.tolist() == [-1, 0, 0, 1, 2]
    assert node_of[(0,)] == 1 and node_of[(1, 0)] == 4


def test_ancestry_is_prefix_relation():
    rng = np.random.default_rng(0)
    for trial in range(40):
        n = int(rng.integers(1, 65))
        paths = W.random_rank_paths(n, int(rng.integers(1, 9)), rng)
        parent, depth, rows, node_of = T.build_tree(paths)
        by_node = {v: k for k, v in node_of.items()}
        m = T.dense_mask(rows, parent.size)
        for i in range(parent.size):
            pi = by_node[i]
            for j in range(parent.size):
                pj = by_node[j]
                assert m[i, j] == (pi[:len(pj)] == pj)
            assert bin(rows[i]).count("1") == depth[i] + 1
            assert depth[i] == len(pi)


def test_siblings_share_positions():
    parent, depth, rows, node_of = T.build_tree(W.PAGE_TREE_PATHS)
    pos = T.positions(depth, 37)
    assert pos[0] == 37 and pos[1] == pos[2] == 38
    for i in range(1, parent.size):
        for j in range(1, parent.size):
            if parent[i] == parent[j]:
                assert pos[i] == pos[j]
        assert pos[i] == pos[parent[i]] + 1


def test_topology_checks():
    with pytest.raises(T.TopologyError):
        T.check_topology([0, 0])
    with pytest.raises(T.TopologyError):
        T.check_topology([-1, 1])
    with pytest.raises(T.TopologyError):
        T.check_topology([-1, 0, 3, 1])
    rows, depth, pos, ok = T.tree_mask_batch(np.array([[-1, 0, 1], [-1, 2, 0]]), [5, 6])
    assert ok.tolist() == [True, False]
    assert rows[0].tolist() == [1, 3, 7] and pos[0].tolist() == [5, 6, 7]
    assert rows[1].tolist() == [0, 0, 0]


def test_path_to_root():
    parent, depth, rows, node_of = T.build_tree(W.PAGE_TREE_PATHS)
    assert T.path_to_root(parent, 9) == [0, 1, 3, 6, 9]
    assert T.path_to_root(parent, 5) == [0, 2, 5]
    assert T.path_to_root(parent, 0) == [0]


def test_ragged_mask_equals_truncated_trees():
    """Ragged trees in a bucket: a request's valid rows are those of its tree
    alone (its first n_b nodes), absent rows are 0 with position -1, and the
    parent entries of absent nodes are never read."""
    rng = np.random.default_rng(77)
    N, B = 20, 12
    par = np.stack([T.build_tree(W.random_rank_paths(N, 5, rng))[0] for _ in range(B)])
    n = rng.integers(1, N + 1, size=B)
    n[0], n[1] = 1, N
    lens = rng.integers(0, 500, size=B)
    garbage = par.copy()
    for b in range(B):
        garbage[b, n[b]:] = 999
    rows, depth, pos, ok = T.tree_mask_batch(garbage, lens, n)
    assert ok.all()
    for b in range(B):
        r1, d1, p1, ok1 = T.tree_mask_batch(par[b:b + 1, :n[b]], lens[b:b + 1])
        assert ok1.all()
        np.testing.assert_array_equal(rows[b, :n[b]], r1[0])
        np.testing.assert_array_equal(pos[b, :n[b]], p1[0])
        assert (rows[b, n[b]:] == 0).all() and (pos[b, n[b]:] == -1).all() and (depth[b, n[b]:] == 0).all()
    # a bad parent among the valid nodes is still caught
    bad = garbage.copy()
    bad[1, 5] = 7
    assert not T.tree_mask_batch(bad, lens, n)[3][1]
