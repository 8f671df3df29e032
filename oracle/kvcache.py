"""Oracle: commit of the accepted path's tree K/V to the paged cache (test
infrastructure).

Definition followed
-------------------
"Build the tree attention mask that verifies a draft tree in one pass",
*What it costs.*: a serving system writes the tree's K/V to scratch and,
after verification, copies the accepted path into the cache.  "Tree
Verification" (stable-lab), *The Cost Side*: the accepted nodes' K/V rows
become the next step's prefix.

The accepted path of request b is ``path[b, 0 .. n_out[b] - 1]`` as the
acceptance step reports it: node ``path[b, 0]`` is the root (the last
accepted token of the previous step), and node ``path[b, j]`` sits at depth
j, i.e. at position ``L_b + j``.  Committing copies tree row
``path[b, j]`` (every KV head) into cache position ``L_b + j`` -- block
``block_table[b, (L_b + j) // block_size]``, slot
``(L_b + j) % block_size`` -- and the prefix length becomes
``L_b + n_out[b]``.  The tree keys are committed as given (the device path
stores them rotated at ``L_b + depth``, which is their cache position).
The token emitted after the last path node has no K/V yet: it is the next
step's root.

The pages define no failure; the library's reading (``stop_at_bad=True``):
a path step that cannot be committed -- a node outside the tree, a
position without a block in the table (or a table entry outside the
cache) -- ends the committed prefix there, so the prefix length never counts
a slot that was not written.
"""

from __future__ import annotations

import numpy as np


def commit_path(k_cache, v_cache, block_table, seq_lens, k_tree, v_tree, path, n_out, stop_at_bad=False):
    """Returns (k_cache', v_cache', seq_lens') with the accepted rows copied in.

    k_cache, v_cache [num_blocks, Hkv, block_size, D]; block_table
    [B, max_blocks]; seq_lens [B]; k_tree, v_tree [B, N, Hkv, D]; path
    [B, cols] node indices; n_out [B].  Raises if a position does not fit the
    block table, unless ``stop_at_bad``: then the first step that cannot be
    committed ends the request's commit (module docstring).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    lens = np.array(seq_lens, dtype=np.int64, copy=True)
    bs = kc.shape[2]
    for b in range(lens.size):
        L = int(seq_lens[b])
        done = int(n_out[b])
        for j in range(int(n_out[b])):
            node = int(path[b, j])
            t = L + j
            fits = t // bs < block_table.shape[1] and 0 <= int(block_table[b, t // bs]) < kc.shape[0]
            if stop_at_bad and not (0 <= node < k_tree.shape[1] and fits):
                done = j
                break
            if t // bs >= block_table.shape[1]:
                raise ValueError(f"request {b}: position {t} beyond its block table")
            blk = int(block_table[b, t // bs])
            kc[blk, :, t % bs, :] = k_tree[b, node]
            vc[blk, :, t % bs, :] = v_tree[b, node]
        lens[b] = L + done
    return kc, vc, lens
