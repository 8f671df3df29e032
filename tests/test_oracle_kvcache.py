"""Pins of the path-commit oracle (oracle/kvcache.py).

The commit is checked against attention, not against a restatement of
itself: after the accepted path is copied into the paged cache, ordinary
decode attention of the last path node's query over the committed cache
(prefix + path, in cache order) must equal that node's tree-attention output
from the one-pass verification ("Tree Verification", *Tree Attention*: a
node's output equals a separate pass over its root-to-node path)."""

import numpy as np
import pytest

from oracle import attention as OA
from oracle import kvcache as OK
from oracle import tree as OT

PAGE_PATHS = [(0,), (1,), (0, 0), (0, 1), (1, 0), (0, 0, 0), (0, 0, 1), (0, 1, 0), (0, 0, 0, 0)]


def _inputs(rng, B, N, Hq, Hkv, D, bs, lens, reserve):
    need = (np.asarray(lens) + reserve + bs - 1) // bs
    max_blocks = int(need.max())
    nblk = int(need.sum()) + 3
    perm = rng.permutation(nblk)
    table = np.zeros((B, max_blocks), dtype=np.int32)
    off = 0
    for b in range(B):
        table[b, :need[b]] = perm[off:off + need[b]]
        off += int(need[b])
    kc = rng.standard_normal((nblk, Hkv, bs, D))
    vc = rng.standard_normal((nblk, Hkv, bs, D))
    q = rng.standard_normal((B, N, Hq, D))
    kt = rng.standard_normal((B, N, Hkv, D))
    vt = rng.standard_normal((B, N, Hkv, D))
    return q, kc, vc, table, kt, vt


def _decode(q_row, kc, vc, table_row, length, G, D, pos):
    """Ordinary attention of one node's query (rotated at pos) over cache rows 0..length-1."""
    keys = OA.gather_prefix(kc, table_row, length)
    vals = OA.gather_prefix(vc, table_row, length)
    out = np.empty_like(q_row)
    qr = OA.rope(q_row, pos)
    for h in range(q_row.shape[0]):
        s = keys[:, h // G] @ qr[h] / np.sqrt(D)
        e = np.exp(s - s.max())
        out[h] = (e[:, None] * vals[:, h // G]).sum(0) / e.sum()
    return out


@pytest.mark.parametrize("bs", [4, 16])
def test_commit_then_decode_equals_tree_attention(bs):
    rng = np.random.default_rng(300 + bs)
    parent, depth, rows, _ = OT.build_tree(PAGE_PATHS)
    N, Hq, Hkv, D = parent.size, 4, 2, 16
    lens = np.array([5, 15, 16, 0])
    B = lens.size
    q, kc, vc, table, kt, vt = _inputs(rng, B, N, Hq, Hkv, D, bs, lens, reserve=N)
    out, _ = OA.tree_attention(q, kc, vc, table, lens, kt, vt, parent)
    # the device stores tree keys rotated at L + depth: commit those
    kt_rot = np.stack([np.stack([OA.rope(kt[b, i], lens[b] + depth[i]) for i in range(N)]) for b in range(B)])
    # root-to-node paths of the tree (parent = [-1, 0, 0, 1, 1, 2, 3, 3, 4, 6])
    paths = [[0, 1, 3, 6, 9], [0], [0, 2, 5], [0, 1, 4, 8]]
    cols = max(len(x) for x in paths)
    path = np.full((B, cols), -1, dtype=np.int64)
    n_out = np.array([len(x) for x in paths])
    for b, x in enumerate(paths):
        path[b, :len(x)] = x
    kc2, vc2, lens2 = OK.commit_path(kc, vc, table, lens, kt_rot, vt, path, n_out)
    np.testing.assert_array_equal(lens2, lens + n_out)
    for b in range(B):
        u = paths[b][-1]
        got = _decode(q[b, u], kc2, vc2, table[b], lens2[b], Hq // Hkv, D, lens[b] + depth[u])
        np.testing.assert_allclose(got, out[b, u], rtol=0, atol=1e-12)
        # untouched: the prefix rows and every slot beyond the committed ones
        np.testing.assert_array_equal(OA.gather_prefix(kc2, table[b], lens[b]),
                                      OA.gather_prefix(kc, table[b], lens[b]))


def test_commit_leaves_other_slots_and_rejects_overflow():
    rng = np.random.default_rng(310)
    parent, depth, rows, _ = OT.build_tree(PAGE_PATHS)
    N = parent.size
    lens = np.array([3, 7])
    q, kc, vc, table, kt, vt = _inputs(rng, 2, N, 2, 1, 8, 4, lens, reserve=2)
    path = np.array([[0, 2], [0, 1]])
    n_out = np.array([2, 2])
    kc2, vc2, _ = OK.commit_path(kc, vc, table, lens, kt, vt, path, n_out)
    changed = np.argwhere(np.any(kc2 != kc, axis=-1))
    expect = set()
    for b in range(2):
        for j in range(2):
            t = lens[b] + j
            expect.add((int(table[b, t // 4]), 0, int(t % 4)))
    assert {tuple(int(x) for x in c) for c in changed} == expect
    # request 1 from position 8 with five path nodes reaches 12, table column
    # 12 // 4 = 3, past the table's 3 columns
    too_long = np.array([[0, 1, -1, -1, -1], [0, 1, 3, 6, 9]])
    lens_far = np.array([3, 8])
    with pytest.raises(ValueError):
        OK.commit_path(kc, vc, table, lens_far, kt, vt, too_long, np.array([2, 5]))


def test_stop_at_bad_equals_the_commit_of_the_path_before_it():
    """With stop_at_bad, a path whose step j cannot be committed (bad node,
    or a position past the block table) commits exactly what the same path
    cut to its first j steps commits."""
    rng = np.random.default_rng(311)
    parent, depth, rows, _ = OT.build_tree(PAGE_PATHS)
    N = parent.size
    lens = np.array([3, 7, 5])
    q, kc, vc, table, kt, vt = _inputs(rng, 3, N, 2, 1, 8, 4, lens, reserve=2)
    path = np.array([[0, 2, N + 4, 5], [0, 1, 3, -1], [0, 1, 3, 6]])
    n_out = np.array([4, 4, 4])
    lens_far = np.array([3, 7, 10])  # request 2: positions 10..13 reach table column 3, past its width
    got = OK.commit_path(kc, vc, table, lens_far, kt, vt, path, n_out, stop_at_bad=True)
    cut = []
    for b in range(3):
        j = 0
        while j < n_out[b]:
            t = lens_far[b] + j
            if not (0 <= path[b, j] < N) or t // 4 >= table.shape[1]:
                break
            j += 1
        cut.append(j)
    assert cut == [2, 3, 2]
    ref = OK.commit_path(kc, vc, table, lens_far, kt, vt, path, np.array(cut))
    for a, r in zip(got, ref):
        np.testing.assert_array_equal(a, r)
