"""Oracle: tree acceptance, greedy and stochastic (test infrastructure).

Sources
-------
* Greedy: "Build the tree attention mask that verifies a draft tree in one
  pass", *The mask.* (walk from the root while some child's draft token equals
  the target's choice after the current node; every visited node emits the
  target's choice -- accepted token, correction or bonus) and "Encode branch
  histories in masks and positions" (a node's logits predict its children: the
  prediction offset).
* Chain sampling: "Implement the lossless speculative sampling verifier for a
  batch with ragged draft lengths", *A strong answer* (accept draft x when
  u * q(x) < p(x), stop at the first rejection, replacement from the
  normalised residual max(0, p - q), bonus from p at the next position, out
  padded with -1, n_out = accepted + 1, ragged num_draft, empty batch legal)
  and *Details that matter in review* 1-4 (no division; cumulative product for
  the first rejection; position j is the bonus position of a row with j
  drafts; p = q falls back to p).
* Tree sampling: the same page, *What interviewers probe next* ("Now the
  drafter proposes a tree": after a sampled child is rejected the target at
  that node becomes the normalised residual and the next sibling is tested
  against it) and "Tree Verification", *Accepting on a Tree* (top-down walk,
  first child that passes becomes the path, all rejected -> replacement from
  that node's distribution, a leaf earns the bonus).

Readings (the pages leave these open; the same choices are documented for
the CUDA side):

* Random numbers are inputs: ``u_accept[b, c]`` is the uniform used when child
  c is tested (one per test), ``u_final[b]`` the uniform of the one
  replacement-or-bonus draw.  In the chain layout the page's ``u[b, j]`` is
  ``u_accept[b, j + 1]``.
* Children are tried in ascending node index (= ascending rank); the draft
  distribution at a node is unchanged between siblings (siblings are i.i.d.
  draws from it), only the target moves to the residual.
* Floating-point cumulative sums are order dependent, so the sampled index is
  taken on a canonical fixed-point image of the distribution: a probability r
  becomes the integer rint(r * 2**40); integer prefix sums are exact in any
  order.  The row sampler of the page (count of prefix sums below u * total,
  clamped to V - 1) is then applied exactly.
* Level 0 at a node is the raw target row p; the first acceptance test is the
  page's ``u * q(x) < p(x)`` evaluated exactly in float64 (a product of two
  float32 numbers is exact).  After a rejection the residual is held as
  integer weights w with total W: level 1 is w = max(0, P - Q) with
  P = rint(2**40 p), Q = rint(2**40 q); level m + 1 is
  w' = max(0, w - floor((W * Q + 2**39) / 2**40)) (the residual of w / W
  against q, rescaled by W).  A sibling at level m >= 1 is accepted iff
  fl64(fl64(u * q(x)) * W) < w(x).  If an update leaves total mass 0, the
  previous level is kept (the page's p = q guard).
"""

from __future__ import annotations

import math

import numpy as np

FIX_BITS = 40
FIX_ONE = 1 << FIX_BITS


# ----------------------------------------------------------------------------
# fixed-point distribution images and the inverse-CDF row sampler
# ----------------------------------------------------------------------------

def fixed_image(r):
    """float32 probabilities -> int64 weights rint(r * 2**40) (half to even)."""
    r64 = np.asarray(r, dtype=np.float32).astype(np.float64)
    return np.rint(r64 * float(FIX_ONE)).astype(np.int64)


def sample_index(weights, u):
    """Inverse-CDF draw from integer weights [..., V] with float32 uniforms [...].

    The sampling page's row sampler: the index is the number of prefix sums
    that lie below u times the total, clamped to V - 1.  Prefix sums are exact
    integers; the threshold u * W is one float64 product (W < 2**53), and an
    integer S lies below the real threshold T exactly when S < ceil(T).
    """
    w = np.asarray(weights, dtype=np.int64)
    total = w.sum(axis=-1)
    if np.any(total >= (1 << 53)):
        raise ValueError("fixed-point mass out of range")
    t = np.asarray(u, dtype=np.float32).astype(np.float64) * total.astype(np.float64)
    thr = np.ceil(t).astype(np.int64)
    below = np.count_nonzero(np.cumsum(w, axis=-1) < thr[..., None], axis=-1)
    idx = np.minimum(below, w.shape[-1] - 1)
    return int(idx) if idx.ndim == 0 else idx


def residual_update(w, scale, q_fixed):
    """One rejection: weights w (mass ``scale``) minus the draft, clamped at 0.

    Exact integer arithmetic: w' = max(0, w - floor((scale * Q + 2**39) / 2**40)).
    """
    sub = (np.asarray(q_fixed, dtype=object) * int(scale) + (1 << (FIX_BITS - 1))) >> FIX_BITS
    diff = np.asarray(w, dtype=object) - sub
    return np.maximum(diff, 0).astype(np.int64)


# ----------------------------------------------------------------------------
# greedy
# ----------------------------------------------------------------------------

def argmax_rows(logits):
    """Target choice per row: largest logit, ties to the lowest index."""
    return np.argmax(np.asarray(logits, dtype=np.float32), axis=-1)


def _children(par, node, n_valid):
    return [c for c in range(node + 1, n_valid) if int(par[c]) == node]


def tree_accept_greedy(target_argmax, tokens, parent, n_nodes=None):
    """Greedy tree walk, per request.

    target_argmax [B, N]: the target's choice after node i (predicts i's
    children); tokens [B, N]: draft token at node i (tokens[:, 0] unused);
    parent [N] or [B, N]; n_nodes [B] (nodes >= n_nodes[b] do not exist).
    Returns out [B, N] (-1 padded), n_out [B], path [B, N] (accepted node ids,
    root first, -1 padded).
    """
    target_argmax = np.asarray(target_argmax)
    tokens = np.asarray(tokens)
    parent = np.asarray(parent)
    B, N = tokens.shape
    n_nodes = np.full(B, N) if n_nodes is None else np.asarray(n_nodes)
    out = np.full((B, N), -1, dtype=np.int64)
    path = np.full((B, N), -1, dtype=np.int64)
    n_out = np.zeros(B, dtype=np.int64)
    for b in range(B):
        par = parent[b] if parent.ndim == 2 else parent
        node, k = 0, 0
        path[b, 0] = 0
        while True:
            choice = int(target_argmax[b, node])
            out[b, k] = choice
            k += 1
            nxt = next((c for c in _children(par, node, int(n_nodes[b]))
                        if int(tokens[b, c]) == choice), None)
            if nxt is None:
                break
            node = nxt
            path[b, k] = node
        n_out[b] = k
    return out, n_out, path


# ----------------------------------------------------------------------------
# stochastic: the chain verifier of the sampling page
# ----------------------------------------------------------------------------

def verify_chain(draft, q, p, num_draft, u, u_final, mutant=None):
    """Chain verifier with explicit uniforms, vectorised over the batch.

    draft [B, K] tokens drawn from q [B, K, V]; p [B, K + 1, V]; num_draft [B];
    u [B, K] float32 (one per accept test); u_final [B] float32.  Returns out
    [B, K + 1] (-1 padded) and n_out [B] = accepted + 1.

    ``mutant`` is for the negative-control tests only: ``"resample_p"`` draws
    the replacement from p instead of the residual, ``"reused_uniform"`` uses
    u[:, 0] for every position, ``"no_bonus"`` emits nothing after a fully
    accepted row.
    """
    draft = np.asarray(draft)
    B, K = draft.shape
    V = np.asarray(p).shape[-1]
    out = np.full((B, K + 1), -1, dtype=np.int64)
    if B == 0:
        return out, np.zeros(0, dtype=np.int64)
    q = np.asarray(q, dtype=np.float32)
    p = np.asarray(p, dtype=np.float32)
    num_draft = np.asarray(num_draft)
    u = np.asarray(u, dtype=np.float32)
    if mutant == "reused_uniform":
        u = np.repeat(u[:, :1], K, axis=1)
    u_final = np.asarray(u_final, dtype=np.float32)
    rows = np.arange(B)
    if K:
        idx = draft[..., None]
        p_tok = np.take_along_axis(p[:, :K], idx, axis=-1)[..., 0].astype(np.float64)
        q_tok = np.take_along_axis(q, idx, axis=-1)[..., 0].astype(np.float64)
        passed = (u.astype(np.float64) * q_tok < p_tok) & (np.arange(K)[None] < num_draft[:, None])
        n_acc = np.cumprod(passed, axis=1).sum(axis=1)
    else:
        n_acc = np.zeros(B, dtype=np.int64)
    rejected = n_acc < num_draft
    P = fixed_image(p[rows, n_acc])
    dist = P
    if K and mutant != "resample_p":
        Q = fixed_image(q[rows, np.minimum(n_acc, K - 1)])
        resid = np.maximum(P - Q, 0)
        use = rejected & (resid.sum(axis=1) > 0)
        dist = np.where(use[:, None], resid, P)
    out_tokens = sample_index(dist, u_final)
    keep = np.arange(K)[None] < n_acc[:, None]
    out[:, :K] = np.where(keep, draft, -1)
    n_out = n_acc + 1
    if mutant == "no_bonus":
        full = ~rejected
        out[rows[~full], n_acc[~full]] = out_tokens[~full]
        n_out = np.where(full, n_acc, n_acc + 1)
    else:
        out[rows, n_acc] = out_tokens
    return out, n_out


# ----------------------------------------------------------------------------
# stochastic: the tree walk with sibling residual updates
# ----------------------------------------------------------------------------

def tree_accept_sample(p, q, tokens, parent, n_nodes, u_accept, u_final, mutant=None):
    """Stochastic tree walk, per request (see module docstring).

    p [B, N, V] target distribution after node i (predicts i's children);
    q [B, N, V] the draft distribution node i's children were drawn from;
    tokens [B, N]; parent [N] or [B, N]; n_nodes [B]; u_accept [B, N] and
    u_final [B] float32.  Returns out [B, N] (-1 padded), n_out [B],
    path [B, N] (accepted node ids, root first, -1 padded).

    ``mutant="siblings_vs_p"`` exists only for a negative-control test: later
    siblings are tested against the raw row p instead of the residual (the
    double counting "Tree Verification", *Accepting on a Tree*, warns about).
    """
    p = np.asarray(p, dtype=np.float32)
    q = np.asarray(q, dtype=np.float32)
    tokens = np.asarray(tokens)
    parent = np.asarray(parent)
    u_accept = np.asarray(u_accept, dtype=np.float32)
    u_final = np.asarray(u_final, dtype=np.float32)
    B, N, V = p.shape
    out = np.full((B, N), -1, dtype=np.int64)
    path = np.full((B, N), -1, dtype=np.int64)
    n_out = np.zeros(B, dtype=np.int64)
    for b in range(B):
        par = parent[b] if parent.ndim == 2 else parent
        node, k = 0, 0
        path[b, 0] = 0
        while True:
            pr, qr = p[b, node], q[b, node]
            w, scale = None, FIX_ONE          # None: level 0, the raw row p
            taken = None
            for c in _children(par, node, int(n_nodes[b])):
                x = int(tokens[b, c])
                if not 0 <= x < V:
                    raise ValueError(f"draft token {x} outside the vocabulary")
                uq = np.float64(u_accept[b, c]) * np.float64(qr[x])
                if w is None or mutant == "siblings_vs_p":
                    ok = uq < np.float64(pr[x])
                else:
                    ok = uq * np.float64(scale) < np.float64(w[x])
                if ok:
                    taken = c
                    break
                nxt = residual_update(fixed_image(pr) if w is None else w, scale, fixed_image(qr))
                mass = int(nxt.sum())
                if mass > 0:
                    w, scale = nxt, mass
            if taken is not None:
                out[b, k] = int(tokens[b, taken])
                k += 1
                node = taken
                path[b, k] = node
                continue
            dist = fixed_image(pr) if w is None else w
            out[b, k] = sample_index(dist, u_final[b])
            k += 1
            break
        n_out[b] = k
    return out, n_out, path
