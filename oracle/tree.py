"""Oracle: draft-tree structure (test infrastructure, see ``oracle/__init__``).

Sources
-------
* "Build the tree attention mask that verifies a draft tree in one pass"
  (inferenceinterviews.com), "A strong answer": *The tree.* (candidates are
  rank paths, node 0 is the root = last accepted token) and *The mask.*
  (duplicates removed, order by length then lexicographically, parent
  pointers and depth, missing parent rejected, a node attends to itself and
  its ancestors, position id = prefix length + depth).
* "Encode branch histories in masks and positions" (study.greatitself.com),
  first two paragraphs: first proposed tokens have depth one; siblings share
  a sequence position.
* "Tree Verification" (stable-lab), *Tree Attention*: any parent-before-child
  flattening is valid, a node sees the context, its root-path ancestors and
  itself, nothing else.

The ancestor set of a node is represented as an integer bit row (bit j set
<=> node j is the node itself or one of its ancestors); ``dense_mask`` turns
the rows into the page's boolean N x N matrix.
"""

from __future__ import annotations

import numpy as np


class MissingParentError(ValueError):
    """A candidate path whose one-shorter prefix is not itself a candidate."""


class TopologyError(ValueError):
    """A parent array that is not parent-before-child with a single root."""


def canonical_paths(paths):
    """Distinct non-empty rank paths in the node order of the mask page.

    The order is by path length first and lexicographically within a length
    ("The mask.", tree-attention-mask page).  The empty path is the root and
    is not a candidate.  Negative ranks are rejected.
    """
    distinct = set()
    for raw in paths:
        t = tuple(int(r) for r in raw)
        if any(r < 0 for r in t):
            raise ValueError(f"negative rank in path {t}")
        if t:
            distinct.add(t)
    return sorted(distinct, key=lambda t: (len(t), t))


def build_tree(paths):
    """Rank paths -> (parent, depth, ancestor_rows, node_of).

    ``parent[0] = -1`` and ``depth[0] = 0`` describe the root; candidate k of
    the canonical order becomes node k + 1 with depth = its path length and
    parent = the node of the path with its last rank removed.  A missing
    prefix raises :class:`MissingParentError` (mask page, "The mask.": the
    missing-parent case is rejected).  ``node_of`` maps every input path
    (duplicates included) to its node id.
    """
    order = canonical_paths(paths)
    node_of = {(): 0}
    for k, t in enumerate(order):
        node_of[t] = k + 1
    absent = [t for t in order if t[:-1] not in node_of]
    if absent:
        raise MissingParentError(f"missing parent for {absent[0]}")
    parent = np.array([-1] + [node_of[t[:-1]] for t in order], dtype=np.int64)
    depth = np.array([0] + [len(t) for t in order], dtype=np.int64)
    rows = ancestor_rows(parent)
    return parent, depth, rows, node_of


def check_topology(parent):
    """Raise :class:`TopologyError` unless parent is a parent-before-child tree.

    Node 0 is the only root (``parent[0] == -1``) and every other node i has
    ``0 <= parent[i] < i`` (a parent-before-child flattening, "Tree
    Verification", *Tree Attention*).
    """
    parent = np.asarray(parent)
    if parent.size == 0 or parent[0] != -1:
        raise TopologyError("node 0 must be the root (parent -1)")
    for i in range(1, parent.size):
        if not 0 <= parent[i] < i:
            raise TopologyError(f"node {i} has parent {parent[i]}")


def ancestor_rows(parent):
    """Per node, the set {node itself} U {its ancestors} as a Python int bit row.

    Found by following parent pointers up to the root (mask page, "The
    mask.": each node attends to itself and its ancestors).
    """
    parent = np.asarray(parent)
    check_topology(parent)
    rows = []
    for i in range(parent.size):
        bits, j = 0, i
        while j != -1:
            bits |= 1 << j
            j = int(parent[j])
        rows.append(bits)
    return rows


def depth_of(parent):
    """Number of parent hops from each node to the root (root depth 0)."""
    parent = np.asarray(parent)
    check_topology(parent)
    out = np.zeros(parent.size, dtype=np.int64)
    for i in range(1, parent.size):
        out[i] = out[parent[i]] + 1
    return out


def dense_mask(rows, n):
    """Bit rows -> boolean matrix ``m[i, j]`` = node i may attend to node j."""
    return np.array([[bool((rows[i] >> j) & 1) for j in range(n)] for i in range(n)])


def positions(depth, prefix_len):
    """Position ids of the tree nodes: prefix length + depth (siblings equal)."""
    return int(prefix_len) + np.asarray(depth, dtype=np.int64)


def path_to_root(parent, i):
    """Node ids on the root-to-node path of node i, root first."""
    chain = []
    j = int(i)
    while j != -1:
        chain.append(j)
        j = int(parent[j])
    return chain[::-1]


def tree_mask_batch(parent, seq_lens, n_nodes=None):
    """Batched structure for per-request parent arrays.

    ``parent`` is int [B, N]; returns (rows uint64 [B, N], depth int [B, N],
    pos int [B, N], ok bool [B]).  A request whose parent row fails
    :func:`check_topology` gets ``ok = False`` and zero rows / depth / pos.

    Ragged trees in a bucket of N ("Build the tree attention mask ...",
    "What interviewers probe next": CUDA graph capture keeps a fixed tree
    shape per batch bucket): with ``n_nodes`` request b is the tree of its
    first n_b = clamp(n_nodes[b], 1, N) nodes and the others are absent, with
    row 0, depth 0 and position -1 (no position: nothing rotates or attends
    to them).
    """
    parent = np.asarray(parent)
    B, N = parent.shape
    rows = np.zeros((B, N), dtype=np.uint64)
    depth = np.zeros((B, N), dtype=np.int64)
    pos = np.zeros((B, N), dtype=np.int64)
    ok = np.ones(B, dtype=bool)
    for b in range(B):
        n = N if n_nodes is None else min(max(int(n_nodes[b]), 1), N)
        pos[b, n:] = -1
        try:
            r = ancestor_rows(parent[b, :n])
        except TopologyError:
            ok[b] = False
            continue
        rows[b, :n] = np.array(r, dtype=np.uint64)
        depth[b, :n] = depth_of(parent[b, :n])
        pos[b, :n] = positions(depth[b, :n], seq_lens[b])
    return rows, depth, pos, ok
