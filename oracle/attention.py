"""Oracle: depth-indexed RoPE and tree attention (test infrastructure).

Definition followed
-------------------
"Tree Verification" (stable-lab), *Tree Attention*: under the tree mask one
forward pass gives, at every node v, exactly the distribution a separate
pass over the context followed by v's root-to-node path would give, and
position ids follow depth.  "Encode branch histories in masks and
positions" (study.greatitself.com) asks that each node's output be compared
with an independent ordinary run on its exact path.  So the oracle does not
use a mask or a depth array at all: for every node it walks ``parent`` up to
the root, lays out

    keys   = prefix K (positions 0..L-1, already rotated in the cache)
             + RoPE(K_tree[a_k], L + k) for the path a_0 = root .. a_d = node
    values = prefix V + V_tree[a_0 .. a_d]
    query  = RoPE(Q[node], L + d)

and takes ordinary softmax attention of the query over those keys -- the
last row of a causal pass over the path -- in float64.  Each query head h
reads KV head ``h // (Hq / Hkv)`` (grouped-query attention).

Readings where the pages are silent: RoPE is the rotate-half form (pairs k
and k + D/2) with angle ``pos * base**(-2k/D)``, base 10000 by default; the
softmax scale defaults to ``1/sqrt(D)``; the root's K/V is tree row 0 (it is
the last accepted token, not yet in the cache); the paged cache is laid out
``[num_blocks, Hkv, block_size, D]`` and position t of request b lives in
block ``block_table[b, t // block_size]``, slot ``t % block_size``.

Ragged trees ("Build the tree attention mask ...", "What interviewers probe
next": a fixed tree shape per batch bucket): with ``n_nodes`` request b holds
nodes 0 .. n_b - 1 and a node i >= n_b is absent.  An absent node has no
position and no tree keys: its query is taken as given (not rotated) and
attends to the prefix alone; with an empty prefix it has no keys at all and
its row is zero with log-normaliser -inf.
"""

from __future__ import annotations

import numpy as np

from .tree import depth_of, path_to_root


def rope_angles(pos, head_dim, base=10000.0):
    """Rotation angles ``pos * base**(-2k/D)`` for k < D/2, float64."""
    k = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = np.power(float(base), -2.0 * k / head_dim)
    return np.multiply.outer(np.asarray(pos, dtype=np.float64), inv_freq)


def rope(x, pos, base=10000.0):
    """Rotate-half RoPE of ``x[..., D]`` at positions ``pos`` (broadcast over
    ``x.shape[:-1]``): (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin)."""
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    ang = rope_angles(pos, x.shape[-1], base)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def gather_prefix_heads(cache, block_row, prefix_len):
    """Prefix rows 0..L-1 of one request from a paged cache, per KV head ->
    [Hkv, L, D] f64: position t is slot t % block_size of block
    block_row[t // block_size] (whole blocks are gathered, then cut at L)."""
    nb, Hkv, block_size, D = cache.shape
    L = int(prefix_len)
    used = -(-L // block_size)
    blocks = np.asarray(block_row)[:used]
    x = np.asarray(cache[blocks], dtype=np.float64)                      # [used, Hkv, bs, D]
    return np.ascontiguousarray(x.transpose(1, 0, 2, 3).reshape(Hkv, used * block_size, D)[:, :L])


def gather_prefix(cache, block_row, prefix_len):
    """Prefix rows 0..L-1 of one request from a paged cache -> [L, Hkv, D] f64."""
    return gather_prefix_heads(cache, block_row, prefix_len).transpose(1, 0, 2)


def _softmax_attend(qh, key_parts, val_parts, scale):
    """Ordinary attention of query rows qh [G, D] over the key set made of
    ``key_parts`` (a list of [T_k, D] arrays laid end to end, values
    likewise): one score row over all keys, one softmax, and the weighted sum
    of the values taken part by part (the same sum, reassociated, so that the
    long prefix is never copied next to each node's path).  An empty key set
    gives zero rows and log-normaliser -inf."""
    if sum(k.shape[0] for k in key_parts) == 0:
        return np.zeros((qh.shape[0], val_parts[0].shape[-1])), np.full(qh.shape[0], -np.inf)
    s = np.concatenate([qh @ k.T for k in key_parts], axis=1) * scale
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=1, keepdims=True)
    o = np.zeros((qh.shape[0], val_parts[0].shape[-1]))
    start = 0
    for v in val_parts:
        o += e[:, start:start + v.shape[0]] @ v
        start += v.shape[0]
    return o / z, (m + np.log(z))[:, 0]


def tree_attention(q, k_cache, v_cache, block_table, seq_lens, k_tree, v_tree,
                   parent, *, rope_base=10000.0, scale=None, nodes=None,
                   mutant=None, n_nodes=None, rotate=True):
    """Per-node path attention (see module docstring).

    Shapes: q [B, N, Hq, D]; k_tree, v_tree [B, N, Hkv, D] (q and k_tree NOT
    yet rotated); caches [num_blocks, Hkv, block_size, D]; block_table
    [B, max_blocks]; seq_lens [B]; parent [N] (one tree for all requests) or
    [B, N].  ``nodes`` optionally lists the (b, i) pairs to compute (others
    stay NaN).  ``n_nodes`` [B] (optional): ragged trees, nodes >= n_nodes[b]
    absent (module docstring).  Returns (out [B, N, Hq, D] f64, lse [B, N, Hq] f64, natural
    log of the softmax normaliser).

    ``rotate=False`` takes ``q`` and ``k_tree`` as already rotated (each node
    at its own position L + depth): the same per-path attention with the
    RoPE step left out.  It lets a test give the attention kernel alone the
    rotated rows, so that its output is compared without the rounding of a
    separate rotation in the input precision.

    ``mutant`` exists only for the negative-control tests and models the two
    mistakes the mask page lists: ``"causal_flat"`` lets node i see every
    node 0..i of the flattened order (siblings included) and
    ``"sequential_positions"`` rotates tree node j at L + j instead of
    L + depth.
    """
    q = np.asarray(q)
    B, N, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    parent = np.asarray(parent)
    out = np.full((B, N, Hq, D), np.nan)
    lse = np.full((B, N, Hq), np.nan)
    want = {}
    if nodes is None:
        for b in range(B):
            want[b] = list(range(N))
    else:
        for b, i in nodes:
            want.setdefault(int(b), []).append(int(i))
    for b, node_list in want.items():
        par = parent[b] if parent.ndim == 2 else parent
        L = int(seq_lens[b])
        # prefix keys and values of each KV head, [L, D] contiguous
        pk = gather_prefix_heads(k_cache, block_table[b], L)
        pv = gather_prefix_heads(v_cache, block_table[b], L)
        n_b = N if n_nodes is None else min(max(int(n_nodes[b]), 1), N)
        dep = depth_of(par[:n_b])
        for i in node_list:
            if i >= n_b:  # absent: the prefix alone, query as given
                qi = np.asarray(q[b, i], dtype=np.float64)
                for kvh in range(Hkv):
                    o, l = _softmax_attend(qi[kvh * G:(kvh + 1) * G], [pk[kvh]], [pv[kvh]], scale)
                    out[b, i, kvh * G:(kvh + 1) * G] = o
                    lse[b, i, kvh * G:(kvh + 1) * G] = l
                continue
            if mutant == "causal_flat":
                chain = list(range(i + 1))
                key_pos = L + dep[chain]
                q_pos = L + dep[i]
            elif mutant == "sequential_positions":
                chain = path_to_root(par, i)
                key_pos = L + np.asarray(chain)
                q_pos = L + i
            elif mutant is None:
                chain = path_to_root(par, i)
                key_pos = L + np.arange(len(chain))
                q_pos = L + len(chain) - 1
            else:
                raise ValueError(mutant)
            kt = np.asarray(k_tree[b, chain], dtype=np.float64)
            qi = np.asarray(q[b, i], dtype=np.float64)
            if rotate:
                kt = rope(kt, np.asarray(key_pos)[:, None], rope_base)
                qi = rope(qi, q_pos, rope_base)
            vt = np.asarray(v_tree[b, chain], dtype=np.float64)
            for kvh in range(Hkv):
                # keys: the prefix, then the root-to-node path
                o, l = _softmax_attend(qi[kvh * G:(kvh + 1) * G], [pk[kvh], kt[:, kvh]], [pv[kvh], vt[:, kvh]], scale)
                out[b, i, kvh * G:(kvh + 1) * G] = o
                lse[b, i, kvh * G:(kvh + 1) * G] = l
    return out, lse
