"""End-to-end losslessness harness for stochastic verifiers (test helper).

Runs the protocol of the sampling page's losslessness test: a target and a
drafter that are Markov chains over a small vocabulary with a start state
generate sequences by repeated draft-and-verify rounds; the joint
distribution of the first ``n_tokens`` tokens is then compared with the exact
product of the target's transition probabilities by a chi-square statistic.

The verifier under test is a callable with the tree interface
``verify(p, q, tokens, parent, n_nodes, u_accept, u_final) -> (out, n_out)``
(numpy in, numpy out), so the same harness drives the oracle and the GPU.
Drafting (sampling node tokens from the drafter's rows) is input synthesis
and lives here, not in any verifier.
"""

import itertools

import numpy as np


def draft_round(parent, state0, qt, rng):
    """Sample a draft tree: node c's token ~ qt[state(parent(c))].

    Returns tokens [B, N] and state [B, N] (state of the root is state0, the
    state of any other node is its own token)."""
    B, N = state0.size, len(parent)
    tokens = np.zeros((B, N), dtype=np.int32)
    state = np.zeros((B, N), dtype=np.int64)
    state[:, 0] = state0
    V = qt.shape[1]
    for c in range(1, N):
        rows = qt[state[:, parent[c]]].astype(np.float64)
        cum = np.cumsum(rows, axis=1)
        u = rng.random(B) * cum[:, -1]
        tok = np.minimum((u[:, None] >= cum).sum(axis=1), V - 1)
        tokens[:, c] = tok
        state[:, c] = tok
    return tokens, state


def processed(table, temperature=1.0, top_p=1.0):
    """A sampler's processing of probability rows: temperature (p^(1/T),
    renormalised -- softmax(logits / T) of the same logits), then top-p (keep
    the most probable tokens, highest first and ties by lower index, up to
    and including the one where the kept mass first reaches top_p; the rest
    set to zero and the kept mass renormalised).  Returns float32 rows."""
    t = np.asarray(table, dtype=np.float64) ** (1.0 / temperature)
    t /= t.sum(axis=-1, keepdims=True)
    order = np.argsort(-t, axis=-1, kind="stable")
    sorted_t = np.take_along_axis(t, order, axis=-1)
    before = np.cumsum(sorted_t, axis=-1) - sorted_t    # mass ahead of each token
    keep_sorted = before < top_p
    keep = np.zeros_like(keep_sorted)
    np.put_along_axis(keep, order, keep_sorted, axis=-1)
    t = np.where(keep, t, 0.0)
    t /= t.sum(axis=-1, keepdims=True)
    return t.astype(np.float32)


def generate(verify, pt, qt, parent, n_seq, n_tokens, seed, batch=None, pt_verify=None, qt_verify=None):
    """Sequences of ``n_tokens`` tokens from repeated draft/verify rounds.

    The drafter samples from ``qt``; the verifier is handed ``pt_verify`` and
    ``qt_verify`` (default: ``pt`` and ``qt``), so a test can give it rows
    that differ from the ones actually sampled."""
    pt_v = pt if pt_verify is None else pt_verify
    qt_v = qt if qt_verify is None else qt_verify
    V = pt.shape[1]
    start = V
    parent = np.asarray(parent)
    N = parent.size
    rng = np.random.default_rng(seed)
    seqs = np.full((n_seq, n_tokens), -1, dtype=np.int64)
    filled = np.zeros(n_seq, dtype=np.int64)
    last = np.full(n_seq, start, dtype=np.int64)
    while True:
        active = np.nonzero(filled < n_tokens)[0]
        if active.size == 0:
            break
        tokens, state = draft_round(parent, last[active], qt, rng)
        p = pt_v[state].astype(np.float32)
        q = qt_v[state].astype(np.float32)
        n_nodes = np.full(active.size, N, dtype=np.int32)
        u_accept = rng.random((active.size, N), dtype=np.float32)
        u_final = rng.random(active.size, dtype=np.float32)
        out, n_out = verify(p, q, tokens, parent, n_nodes, u_accept, u_final)
        out = np.asarray(out)
        n_out = np.asarray(n_out)
        for j in range(N):
            take = (n_out > j) & (filled[active] < n_tokens)
            idx = active[take]
            seqs[idx, filled[idx]] = out[take, j]
            filled[idx] += 1
            last[idx] = out[take, j]
    return seqs


def chi_square(seqs, pt):
    """Chi-square of the joint token distribution against the target chain."""
    V = pt.shape[1]
    n_tokens = seqs.shape[1]
    counts = np.zeros((V,) * n_tokens)
    np.add.at(counts, tuple(seqs.T), 1)
    expect = np.zeros_like(counts)
    for cell in itertools.product(range(V), repeat=n_tokens):
        pr, prev = 1.0, V
        for t in cell:
            pr *= float(pt[prev, t])
            prev = t
        expect[cell] = pr
    expect *= seqs.shape[0]
    return float(((counts - expect) ** 2 / expect).sum())


def chi_square_support(seqs, pt):
    """Chi-square over the cells the target can produce, for targets with
    zero entries: returns (statistic, degrees of freedom, sequences that fell
    in a zero-probability cell)."""
    V = pt.shape[1]
    n_tokens = seqs.shape[1]
    counts = np.zeros((V,) * n_tokens)
    np.add.at(counts, tuple(seqs.T), 1)
    expect = np.zeros_like(counts)
    for cell in itertools.product(range(V), repeat=n_tokens):
        pr, prev = 1.0, V
        for t in cell:
            pr *= float(pt[prev, t])
            prev = t
        expect[cell] = pr
    expect *= seqs.shape[0]
    live = expect > 0
    stat = float(((counts[live] - expect[live]) ** 2 / expect[live]).sum())
    return stat, int(live.sum()) - 1, int(counts[~live].sum())


def chain_adapter(verify_chain, **kw):
    """Wrap a page-layout chain verifier (draft, q, p, num_draft, u, u_final)
    into the tree interface for chain-shaped trees."""
    def verify(p, q, tokens, parent, n_nodes, u_accept, u_final):
        K = p.shape[1] - 1
        out, n_out = verify_chain(tokens[:, 1:], q[:, :K], p, n_nodes - 1,
                                  u_accept[:, 1:], u_final, **kw)
        return out, n_out
    return verify
