"""Plain CPU oracle for one-pass draft-tree verification.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code with the CUDA library (no kernels, headers, helpers or
tables) and imports nothing from the ``speculative_decoding_tree_attn_gb300``
package; both sides receive the same seeded inputs from the workload
generator and nothing else.

Everything is written as the plain definition the pages give, in float64
(numpy), with no blocking, fusion or reordering beyond the definition:

* ``tree``        -- rank paths -> parent / depth / ancestor rows / positions.
* ``attention``   -- depth-indexed RoPE and, per node, ordinary causal
                     attention over the node's own root-to-node path.
* ``accept``      -- greedy tree walk, the chain verifier of the sampling
                     page, the tree walk with sibling residual updates, and
                     the fixed-point inverse-CDF sampler they share.
* ``kvcache``     -- commit of the accepted path's tree K/V into the paged
                     cache.

Every function is pinned by ``tests/test_oracle_*.py`` (``-m "not gpu"``)
against facts the pages print or mathematics fixes; no function here is
"parity unpinned".
"""

from . import accept, attention, kvcache, tree  # noqa: F401
