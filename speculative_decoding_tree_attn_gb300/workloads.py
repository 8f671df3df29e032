"""Seeded synthetic workloads for draft-tree verification.

This module only draws inputs: rank-path trees, ragged prefix lengths, paged
block tables, Q/K/V, logits, probability rows, draft tokens and uniforms.  It
holds none of the verification arithmetic (no tree construction, RoPE,
attention or acceptance) and imports neither the CUDA binding nor the oracle,
so it can feed both sides identical inputs.

Tree shapes follow a best-first rule over per-rank acceptance probabilities:
a node is worth the product of its ranks' probabilities and the N - 1 most
valuable paths (ties broken by length, then lexicographically, using exact
rationals) form a static tree, as the mask page describes ("a typical static
tree spends more nodes under high-ranked parents"; "What it buys.").
"""

from __future__ import annotations

import heapq
import math
from dataclasses import dataclass, field
from fractions import Fraction

import numpy as np
import torch

# ---------------------------------------------------------------------------
# tree shapes (rank paths only; node numbering is the method's job)
# ---------------------------------------------------------------------------


def best_first_paths(rank_probs, n_nodes, max_depth):
    """The n_nodes - 1 highest-value rank paths of depth <= max_depth."""
    r = [Fraction(x).limit_denominator(10**6) for x in rank_probs]
    heap = [(-r[k], 1, (k,)) for k in range(len(r))]
    heapq.heapify(heap)
    chosen = []
    while len(chosen) < n_nodes - 1 and heap:
        neg, length, path = heapq.heappop(heap)
        chosen.append(path)
        if length < max_depth:
            for k in range(len(r)):
                heapq.heappush(heap, (neg * r[k], length + 1, path + (k,)))
    return chosen


def path_value(path, rank_probs):
    """Product of the per-rank probabilities along a rank path (exact)."""
    v = Fraction(1)
    for k in path:
        v *= Fraction(rank_probs[k]).limit_denominator(10**6)
    return v


def random_rank_paths(n_nodes, max_depth, rng):
    """Random tree: each new node hangs under a random node of depth < max_depth
    and takes that parent's next free rank."""
    paths = [()]
    n_kids = {(): 0}
    while len(paths) < n_nodes:
        open_nodes = [p for p in paths if len(p) < max_depth]
        par = open_nodes[int(rng.integers(len(open_nodes)))]
        child = par + (n_kids[par],)
        n_kids[par] += 1
        n_kids[child] = 0
        paths.append(child)
    return paths[1:]


# The mask page's 10-node example tree (root + 9): two candidates at depth 1,
# three at depths 2 and 3, one at depth 4, built from rank probabilities
# (0.7, 0.15) -- the example's per-depth sums 0.7 + 0.15, 0.49 + 0.105 + 0.105,
# 0.343 + 0.0735 + 0.0735 and 0.2401 fix its shape.
PAGE_TREE_RANK_PROBS = (0.7, 0.15)
PAGE_TREE_PATHS = best_first_paths(PAGE_TREE_RANK_PROBS, 10, 4)


# ---------------------------------------------------------------------------
# workload configurations
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: str                 # "f32" | "bf16"
    prefix: tuple              # ("fixed", L) | ("uniform", lo, hi)
    block_size: int
    rank_probs: tuple
    n_nodes: int
    max_depth: int
    seed: int
    accept: str = "none"       # "none" | "greedy" | "sample"
    vocab: int = 0
    sample_max_draft: int = 4
    dynamic: bool = False      # one tree per request (dynamic_rank_paths)
    sample_tree: bool = False  # "sample" on the attention tree (sample_tree_inputs), else on chains
    ragged: bool = False       # per-request node counts in the bucket of n_nodes (node_counts)
    notes: str = field(default="", compare=False)

    def paths(self):
        return best_first_paths(self.rank_probs, self.n_nodes, self.max_depth)


def node_counts(w: Workload, B=None):
    """Nodes per request: n_nodes for all, or for a ragged workload a seeded
    draw from U{ceil(N/4) .. N} (each request keeps the first n_b nodes of its
    tree, a tree itself since parents precede children)."""
    B = w.B if B is None else B
    N = w.n_nodes
    if not w.ragged:
        return np.full(B, N, dtype=np.int32)
    rng = np.random.default_rng(w.seed * 1000 + 43)
    return rng.integers(max(1, (N + 3) // 4), N + 1, size=B).astype(np.int32)


def dynamic_rank_paths(w: Workload, B=None):
    """One tree per request with the workload's node budget, as dynamic trees
    (EAGLE-2 / DDTree-style budgeted best-first selection) build them: each
    request's per-rank confidences are drawn around the workload's rank
    probabilities (Dirichlet, concentration 20, sorted so rank 0 stays the
    most likely) and its tree is the best-first selection under them."""
    B = w.B if B is None else B
    rng = np.random.default_rng(w.seed * 1000 + 29)
    base = np.asarray(w.rank_probs, dtype=np.float64)
    total = float(base.sum())
    out = []
    for _ in range(B):
        conf = np.sort(rng.dirichlet(base / total * 20.0) * total)[::-1]
        out.append(best_first_paths(tuple(float(x) for x in conf), w.n_nodes, w.max_depth))
    return out


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_b1_f32", 1, 1, 1, 64, "f32", ("fixed", 32), 16,
                 PAGE_TREE_RANK_PROBS, 10, 4, 1, accept="greedy", vocab=1000,
                 notes="the mask page's 10-node tree; plus seeded random depth<=4 trees in tests"),
        Workload("gqa_b8_l512_2048_n26", 8, 32, 8, 128, "bf16", ("uniform", 512, 2048), 16,
                 (0.70, 0.15, 0.08, 0.04), 26, 5, 2, accept="greedy", vocab=32000,
                 notes="Llama-like GQA; greedy accept over a 32000 vocabulary"),
        Workload("b64_l1k_8k_n64_greedy", 64, 32, 8, 128, "bf16", ("uniform", 1024, 8192), 16,
                 (0.45, 0.2, 0.12, 0.08, 0.06, 0.04, 0.03, 0.02), 64, 6, 3,
                 accept="greedy", vocab=32000),
        Workload("long_b16_l32k_n33", 16, 64, 8, 128, "bf16", ("fixed", 32768), 64,
                 (0.75, 0.12, 0.06, 0.03), 33, 8, 4, accept="none"),
        Workload("b256_l2k_4k_n10_sample", 256, 32, 8, 128, "bf16", ("uniform", 2048, 4096), 16,
                 PAGE_TREE_RANK_PROBS, 10, 4, 5, accept="sample", vocab=128000,
                 sample_max_draft=4),
        Workload("b64_l1k_8k_n64_dynamic", 64, 32, 8, 128, "bf16", ("uniform", 1024, 8192), 16,
                 (0.45, 0.2, 0.12, 0.08, 0.06, 0.04, 0.03, 0.02), 64, 6, 6,
                 accept="greedy", vocab=32000, dynamic=True,
                 notes="the 64-request workload with one best-first tree per request"),
        Workload("b64_l1k_8k_n64_ragged", 64, 32, 8, 128, "bf16", ("uniform", 1024, 8192), 16,
                 (0.45, 0.2, 0.12, 0.08, 0.06, 0.04, 0.03, 0.02), 64, 6, 8,
                 accept="greedy", vocab=32000, dynamic=True, ragged=True,
                 notes="one best-first tree per request, n_b ~ U{16..64} nodes in the bucket of 64"),
        Workload("b64_l1k_8k_n64_sample", 64, 32, 8, 128, "bf16", ("uniform", 1024, 8192), 16,
                 (0.45, 0.2, 0.12, 0.08, 0.06, 0.04, 0.03, 0.02), 64, 6, 7,
                 accept="sample", vocab=32000, sample_tree=True,
                 notes="the 64-request workload verified stochastically on its tree (i.i.d. siblings)"),
    ]
}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def prefix_lengths(w: Workload, seed_offset=0):
    rng = np.random.default_rng(w.seed * 1000 + 11 + seed_offset)
    if w.prefix[0] == "fixed":
        return np.full(w.B, w.prefix[1], dtype=np.int32)
    lo, hi = w.prefix[1], w.prefix[2]
    return rng.integers(lo, hi + 1, size=w.B).astype(np.int32)


def block_table_for(seq_lens, block_size, seed, spare_blocks=0):
    """Non-contiguous paging: request b owns ceil(L_b / block_size) physical
    blocks drawn from a seeded random permutation.  Unused table entries are 0."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    need = (seq_lens + block_size - 1) // block_size
    max_blocks = max(1, int(need.max()) if need.size else 1)
    total = int(need.sum()) + int(spare_blocks)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(max(total, 1)).astype(np.int32)
    table = np.zeros((seq_lens.size, max_blocks), dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += int(n)
    return table, max(total, 1)


def attention_inputs(w: Workload, device="cpu", seq_lens=None, n_nodes=None, tree_scale=1.0, reserve=0):
    """Q, paged K/V cache, block table, prefix lengths and tree K/V ~ N(0, 1).

    Returns a dict of tensors on ``device``: q [B, N, Hq, D], k_cache/v_cache
    [num_blocks, Hkv, block_size, D], block_table [B, max_blocks] int32,
    seq_lens [B] int32, k_tree/v_tree [B, N, Hkv, D]; values in ``w.dtype``.
    ``tree_scale`` multiplies the tree keys (mask-sensitivity cases);
    ``reserve`` places blocks for that many positions past each prefix (room
    to commit an accepted path).
    """
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    N = w.n_nodes if n_nodes is None else int(n_nodes)
    lens = prefix_lengths(w) if seq_lens is None else np.asarray(seq_lens, dtype=np.int32)
    table, num_blocks = block_table_for(lens + int(reserve), w.block_size, w.seed * 1000 + 13)
    g = _gen(w.seed * 1000 + 17, device)

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dt)

    B = lens.size
    out = {
        "q": randn(B, N, w.Hq, w.D),
        "k_cache": randn(num_blocks, w.Hkv, w.block_size, w.D),
        "v_cache": randn(num_blocks, w.Hkv, w.block_size, w.D),
        "k_tree": randn(B, N, w.Hkv, w.D),
        "v_tree": randn(B, N, w.Hkv, w.D),
        "block_table": torch.from_numpy(table).to(device),
        "seq_lens": torch.from_numpy(lens).to(device),
    }
    if tree_scale != 1.0:
        out["k_tree"] = (out["k_tree"].float() * tree_scale).to(dt)
    return out


def sibling_rank(parent):
    """Rank of each node among its siblings (ascending node index)."""
    parent = np.asarray(parent)
    seen = {}
    rank = np.zeros(parent.size, dtype=np.int64)
    for i in range(1, parent.size):
        p = int(parent[i])
        rank[i] = seen.get(p, 0)
        seen[p] = rank[i] + 1
    return rank


def greedy_inputs(w: Workload, parent, device="cpu", rank_probs=None, B=None):
    """Draft tokens and target logits ~ N(0, 2) with a planted argmax.

    At each node the target's choice is the draft token of its rank-k child
    with probability rank_probs[k] (when that child exists), otherwise a token
    that no child carries.  Sibling draft tokens are distinct.  ``parent`` is
    the [N] parent array of the static tree, or [B, N] for one tree per
    request.
    """
    rank_probs = w.rank_probs if rank_probs is None else rank_probs
    B = w.B if B is None else B
    V = w.vocab
    parent = np.asarray(parent)
    N = parent.shape[-1]
    rng = np.random.default_rng(w.seed * 1000 + 19)
    shared = parent.ndim == 1
    if shared:
        rank = sibling_rank(parent)
        kids = [[c for c in range(N) if parent[c] == n] for n in range(N)]
    tokens = np.zeros((B, N), dtype=np.int32)
    choice = np.zeros((B, N), dtype=np.int64)
    cum = np.cumsum(np.asarray(rank_probs, dtype=np.float64))
    for b in range(B):
        if not shared:  # one tree per request: parent [B, N]
            rank = sibling_rank(parent[b])
            kids = [[c for c in range(N) if parent[b, c] == n] for n in range(N)]
        for n in range(N):
            ks = kids[n]
            toks = rng.integers(0, V, size=len(ks) + 1)
            while np.unique(toks).size != toks.size:
                toks = rng.integers(0, V, size=len(ks) + 1)
            for c, t in zip(ks, toks[:-1]):
                tokens[b, c] = t
            r = int(np.searchsorted(cum, rng.random(), side="right"))
            hit = [c for c in ks if rank[c] == r]
            choice[b, n] = tokens[b, hit[0]] if hit else toks[-1]
    g = _gen(w.seed * 1000 + 23, device)
    logits = torch.randn(B, N, V, generator=g, device=device, dtype=torch.float32) * math.sqrt(2.0)
    ch = torch.from_numpy(choice).to(device)
    top = logits.max(dim=-1).values + 1.0
    logits.scatter_(-1, ch[..., None], top[..., None])
    return {"tokens": torch.from_numpy(tokens).to(device), "logits": logits}


def sample_chain_inputs(w: Workload, device="cpu", B=None, V=None, max_draft=None,
                        noise_std=0.5, logit_std=math.sqrt(2.0)):
    """Chain verifier inputs: p = softmax(logits), q = softmax(logits + noise).

    Rows: p, q [B, K + 1, V] float32 (row j = the distributions after node j of
    the chain; draft j + 1 is drawn from q row j), tokens [B, K + 1] (tokens[:, 0]
    unused), n_nodes [B] = num_draft + 1 with num_draft ~ U{0..K}, parent
    [K + 1] of the chain, u_accept [B, K + 1] and u_final [B] float32 U[0, 1).
    """
    B = w.B if B is None else B
    V = w.vocab if V is None else V
    K = w.sample_max_draft if max_draft is None else max_draft
    g = _gen(w.seed * 1000 + 29, device)
    logits = torch.randn(B, K + 1, V, generator=g, device=device) * logit_std
    noise = torch.randn(B, K + 1, V, generator=g, device=device) * noise_std
    p = torch.softmax(logits, dim=-1)
    q = torch.softmax(logits + noise, dim=-1)
    drafts = torch.multinomial(q[:, :K].reshape(B * K, V), 1, generator=g).reshape(B, K) if K else \
        torch.zeros(B, 0, dtype=torch.int64, device=device)
    tokens = torch.zeros(B, K + 1, dtype=torch.int32, device=device)
    tokens[:, 1:] = drafts.to(torch.int32)
    rng = np.random.default_rng(w.seed * 1000 + 31)
    num_draft = rng.integers(0, K + 1, size=B).astype(np.int32)
    u_accept = rng.random((B, K + 1), dtype=np.float32)
    u_final = rng.random(B, dtype=np.float32)
    parent = np.arange(-1, K, dtype=np.int32)
    return {
        "p": p.float().contiguous(), "q": q.float().contiguous(), "tokens": tokens,
        "n_nodes": torch.from_numpy(num_draft + 1).to(device),
        "parent": torch.from_numpy(parent).to(device),
        "u_accept": torch.from_numpy(u_accept).to(device),
        "u_final": torch.from_numpy(u_final).to(device),
    }


def sample_tree_inputs(w: Workload, parent, device="cpu", B=None, V=None, noise_std=0.5,
                       logit_std=math.sqrt(2.0)):
    """Tree verifier inputs with i.i.d. siblings: p = softmax(logits),
    q = softmax(logits + noise) per node, and every child's token drawn on
    its own from its parent's q row (siblings may repeat, as when a drafter
    samples several candidates with replacement).

    parent int [N] (shared) or [B, N].  Returns p, q [B, N, V] float32, tokens
    [B, N] int32 (column 0 unused), n_nodes [B] = N, parent as given (int32),
    u_accept [B, N] and u_final [B] float32 U[0, 1).
    """
    B = w.B if B is None else B
    V = w.vocab if V is None else V
    par = np.asarray(parent, dtype=np.int64)
    N = par.shape[-1]
    g = _gen(w.seed * 1000 + 37, device)
    logits = torch.randn(B, N, V, generator=g, device=device) * logit_std
    p = torch.softmax(logits, dim=-1)
    logits += torch.randn(B, N, V, generator=g, device=device) * noise_std
    q = torch.softmax(logits, dim=-1)
    del logits
    tokens = torch.zeros(B, N, dtype=torch.int32, device=device)
    if N > 1:
        pb = np.broadcast_to(par, (B, N))[:, 1:]
        rows = q[torch.arange(B, device=device)[:, None], torch.from_numpy(np.ascontiguousarray(pb)).to(device)]
        draws = torch.multinomial(rows.reshape(B * (N - 1), V), 1, generator=g).reshape(B, N - 1)
        tokens[:, 1:] = draws.to(torch.int32)
    rng = np.random.default_rng(w.seed * 1000 + 41)
    u_accept = rng.random((B, N), dtype=np.float32)
    u_final = rng.random(B, dtype=np.float32)
    return {
        "p": p.contiguous(), "q": q.contiguous(), "tokens": tokens,
        "n_nodes": torch.full((B,), N, dtype=torch.int32, device=device),
        "parent": torch.from_numpy(np.ascontiguousarray(par.astype(np.int32))).to(device),
        "u_accept": torch.from_numpy(u_accept).to(device),
        "u_final": torch.from_numpy(u_final).to(device),
    }


def markov_tables(vocab, seed):
    """Random target and drafter Markov chains over ``vocab`` tokens plus a
    start state (row ``vocab``): rows are Dirichlet(1) draws, float32."""
    rng = np.random.default_rng(seed)
    pt = rng.dirichlet(np.ones(vocab), size=vocab + 1).astype(np.float32)
    qt = rng.dirichlet(np.ones(vocab), size=vocab + 1).astype(np.float32)
    return pt, qt
