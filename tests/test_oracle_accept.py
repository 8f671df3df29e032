"""Pins for the oracle's acceptance (CPU only).

Greedy: the mask page's two example walks, the page's expected tokens per
step (Monte Carlo over its rank model), and exact equality with plain greedy
decoding of a deterministic target.  Stochastic: the sampling page's 2.533
acceptance check and its 2.19 no-bonus figure, the chi-square losslessness
test with its negative controls, the page's small checks (p = q, zero drafts,
empty batch, one-hot target), an exact-rational brute force of the fixed-point
row sampler, and agreement of the tree walk with the chain verifier.  The
sampling page's processed-distribution note: with temperature / top-p
applied to p (and q as the drafter sampled it) the walk is lossless with
respect to the processed target, and handing it unprocessed rows shows up as
bias.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import accept as A
from oracle import tree as T
from speculative_decoding_tree_attn_gb300 import workloads as W

from markov_harness import chain_adapter, chi_square, chi_square_support, generate, processed


def page_tree():
    parent, depth, rows, node_of = T.build_tree(W.PAGE_TREE_PATHS)
    return parent, node_of


# ---------------------------------------------------------------- greedy

def test_greedy_second_rank_branch():
    parent, node_of = page_tree()
    N = parent.size
    tokens = np.arange(100, 100 + N)[None]
    am = np.full((1, N), 7)
    am[0, 0] = tokens[0, node_of[(1,)]]          # target picks the rank-1 candidate
    am[0, node_of[(1,)]] = tokens[0, node_of[(1, 0)]]
    out, n_out, path = A.tree_accept_greedy(am, tokens, parent)
    assert n_out[0] == 3
    assert out[0, :3].tolist() == [tokens[0, 2], tokens[0, 5], 7]
    assert path[0, :3].tolist() == [0, 2, 5] and out[0, 3] == -1


def test_greedy_deepest_leaf(mask_facts):
    parent, node_of = page_tree()
    N = parent.size
    tokens = np.arange(100, 100 + N)[None]
    am = np.full((1, N), 3)
    for path in [(), (0,), (0, 0), (0, 0, 0)]:
        am[0, node_of[path]] = tokens[0, node_of[path + (0,)]]
    out, n_out, path = A.tree_accept_greedy(am, tokens, parent)
    assert n_out[0] == int(mask_facts["deepest_leaf_tokens"][0][0])
    assert path[0, :5].tolist() == [0, 1, 3, 6, 9]
    assert out[0, :5].tolist() == [101, 103, 106, 109, 3]


def test_greedy_ragged_nodes_and_duplicates():
    # duplicate sibling tokens: the lower node index is followed
    parent = np.array([-1, 0, 0, 1, 2])
    tokens = np.array([[0, 5, 5, 8, 9]])
    am = np.array([[5, 8, 9, 1, 1]])
    out, n_out, path = A.tree_accept_greedy(am, tokens, parent)
    assert path[0, :2].tolist() == [0, 1] and out[0, :3].tolist() == [5, 8, 1]
    # nodes >= n_nodes do not exist
    out, n_out, path = A.tree_accept_greedy(am, tokens, parent, n_nodes=[3])
    assert out[0, :3].tolist() == [5, 8, -1] and n_out[0] == 2


def _mc_greedy(parent, r, n_walks, seed):
    N = parent.size
    rank = W.sibling_rank(parent)
    rng = np.random.default_rng(seed)
    tokens = np.zeros((n_walks, N), dtype=np.int64)
    tokens[:, 1:] = 10 + rank[1:]
    cum = np.cumsum(r)
    draw = np.searchsorted(cum, rng.random((n_walks, N)), side="right")
    am = np.where(draw < len(r), 10 + draw, 1)
    out, n_out, path = A.tree_accept_greedy(am, tokens, parent)
    return n_out


@pytest.mark.parametrize("shape", ["tree", "chain"])
def test_greedy_expected_tokens(mask_facts, shape):
    r = [float(x) for x in mask_facts["rank_probs"][0]]
    if shape == "tree":
        parent, _ = page_tree()
        exact = 1 + sum(float(W.path_value(p, r)) for p in W.PAGE_TREE_PATHS)
        page = float(mask_facts["tree_expected_tokens"][0][0])
    else:
        parent = np.arange(-1, 4)
        exact = sum(r[0] ** k for k in range(5))
        page = float(mask_facts["chain_expected_tokens"][0][0])
    assert round(exact, 2) == page
    n_out = _mc_greedy(parent, r, 200_000, 11)
    se = n_out.std() / math.sqrt(n_out.size)
    assert abs(n_out.mean() - exact) < 4 * se


def test_greedy_equals_plain_greedy_decoding():
    """Speculative greedy rounds reproduce plain greedy decoding exactly."""
    rng = np.random.default_rng(12)
    V = 50
    f = rng.integers(0, V, size=V + 1)                      # target's argmax after token t
    guess1 = np.where(rng.random(V + 1) < 0.7, f, rng.integers(0, V, size=V + 1))
    guess2 = np.where(rng.random(V + 1) < 0.6, f, rng.integers(0, V, size=V + 1))
    n_tok = 60
    plain, t = [], V
    for _ in range(n_tok):
        t = int(f[t])
        plain.append(t)
    for paths in [[(0,), (0, 0), (0, 0, 0), (0, 0, 0, 0)], W.PAGE_TREE_PATHS]:
        parent, depth, rows, node_of = T.build_tree(paths)
        by_node = {v: k for k, v in node_of.items()}
        N = parent.size
        seq, last = [], V
        while len(seq) < n_tok:
            state = np.zeros(N, dtype=np.int64)
            tokens = np.zeros(N, dtype=np.int64)
            state[0] = last
            for c in range(1, N):
                g = guess1 if by_node[c][-1] == 0 else guess2
                tokens[c] = g[state[parent[c]]]
                state[c] = tokens[c]
            am = f[state]                                   # node i's row predicts its children
            out, n_out, _ = A.tree_accept_greedy(am[None], tokens[None], parent)
            seq.extend(out[0, :n_out[0]].tolist())
            last = seq[-1]
        assert seq[:n_tok] == plain


def test_argmax_ties_lowest_index():
    x = np.array([[1.0, 3.0, 3.0, -2.0], [0.0, 0.0, 0.0, 0.0]], dtype=np.float32)
    assert A.argmax_rows(x).tolist() == [1, 0]


# ---------------------------------------------------------------- fixed-point sampler

def test_sample_index_exact_rational():
    rng = np.random.default_rng(13)
    for _ in range(400):
        V = int(rng.integers(1, 9))
        w = rng.integers(0, 50, size=V)
        w[rng.integers(V)] += 1
        u = np.float32(rng.random())
        total = int(w.sum())
        thr = Fraction(float(u)) * total
        prefix = np.cumsum(w)
        want = min(sum(1 for s in prefix if s < thr), V - 1)
        assert A.sample_index(w, u) == want


def test_sample_index_distribution():
    w = A.fixed_image(np.array([0.1, 0.0, 0.6, 0.3], dtype=np.float32))
    u = np.random.default_rng(14).random(200_000, dtype=np.float32)
    idx = A.sample_index(np.broadcast_to(w, (u.size, 4)), u)
    freq = np.bincount(idx, minlength=4) / u.size
    np.testing.assert_allclose(freq, [0.1, 0.0, 0.6, 0.3], atol=0.004)


def test_fixed_image_and_residual():
    assert A.fixed_image(np.float32(1.0)) == 1 << 40
    assert A.fixed_image(np.float32(0.5)) == 1 << 39
    P = A.fixed_image(np.array([0.5, 0.25, 0.25], dtype=np.float32))
    Q = A.fixed_image(np.array([0.25, 0.5, 0.25], dtype=np.float32))
    np.testing.assert_array_equal(A.residual_update(P, A.FIX_ONE, Q), np.maximum(P - Q, 0))
    w = np.array([3, 0, 5])
    # residual of w / 8 against q = (0.25, 0.5, 0.25): 8 * q = (2, 4, 2)
    np.testing.assert_array_equal(A.residual_update(w, 8, Q), [1, 0, 3])


# ---------------------------------------------------------------- chain verifier

def test_alpha_expected_tokens(verifier_facts):
    f = verifier_facts
    p = np.array([float(x) for x in f["target_p"][0]], dtype=np.float32)
    V = int(f["drafter_q_uniform"][0][0])
    q = np.full(V, 1.0 / V, dtype=np.float32)
    alpha = float(np.minimum(p, q).sum())
    assert round(alpha, 2) == float(f["alpha"][0][0])
    K = int(f["num_draft"][0][0])
    exact = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert round(exact, 3) == float(f["expected_tokens"][0][0])
    B = int(f["measured_rows"][0][0])
    rng = np.random.default_rng(15)
    draft = rng.choice(V, size=(B, K), p=q.astype(np.float64))
    u = rng.random((B, K), dtype=np.float32)
    uf = rng.random(B, dtype=np.float32)
    P = np.broadcast_to(p, (B, K + 1, V))
    Q = np.broadcast_to(q, (B, K, V))
    out, n_out = A.verify_chain(draft, Q, P, np.full(B, K), u, uf)
    se = n_out.std() / math.sqrt(B)
    assert abs(n_out.mean() - exact) < 4 * se
    assert abs(n_out.mean() - float(f["measured_tokens"][0][0])) < 0.01
    # negative control: forgetting the bonus gives the page's 2.19
    out, n_nb = A.verify_chain(draft, Q, P, np.full(B, K), u, uf, mutant="no_bonus")
    assert round(exact - alpha ** K, 2) == float(f["no_bonus_tokens"][0][0])
    assert abs(n_nb.mean() - float(f["no_bonus_tokens"][0][0])) < 4 * se + 0.005


def _markov_facts(f):
    V = int(f["chi2_vocab"][0][0])
    n_seq = int(f["chi2_sequences"][0][0])
    n_tok = int(f["chi2_tokens"][0][0])
    K = int(f["chi2_drafts_per_round"][0][0])
    assert V ** n_tok == int(f["chi2_cells"][0][0])
    return V, n_seq, n_tok, K, float(f["chi2_threshold"][0][0])


def test_chain_lossless_chi_square(verifier_facts):
    V, n_seq, n_tok, K, thr = _markov_facts(verifier_facts)
    pt, qt = W.markov_tables(V, 16)
    parent = np.arange(-1, K)
    seqs = generate(chain_adapter(A.verify_chain), pt, qt, parent, n_seq, n_tok, 17)
    assert chi_square(seqs, pt) < thr


@pytest.mark.parametrize("mutant", ["resample_p", "reused_uniform"])
def test_chain_negative_controls_fail(verifier_facts, mutant):
    V, n_seq, n_tok, K, thr = _markov_facts(verifier_facts)
    pt, qt = W.markov_tables(V, 16)
    parent = np.arange(-1, K)
    seqs = generate(chain_adapter(A.verify_chain, mutant=mutant), pt, qt, parent, n_seq, n_tok, 17)
    assert chi_square(seqs, pt) > thr


def test_chi_square_threshold_value(verifier_facts):
    scipy_stats = pytest.importorskip("scipy.stats")
    df = int(verifier_facts["chi2_df"][0][0])
    assert abs(scipy_stats.chi2.ppf(0.999, df) - float(verifier_facts["chi2_threshold"][0][0])) < 0.1


def test_p_equals_q_accepts_everything():
    rng = np.random.default_rng(18)
    B, K, V = 500, 4, 7
    p = rng.dirichlet(np.ones(V), size=(B, K + 1)).astype(np.float32)
    nd = rng.integers(0, K + 1, size=B)
    draft = rng.integers(0, V, size=(B, K))
    out, n_out = A.verify_chain(draft, p[:, :K], p, nd, rng.random((B, K), dtype=np.float32),
                                rng.random(B, dtype=np.float32))
    np.testing.assert_array_equal(n_out, nd + 1)


def test_zero_drafts_draw_from_target():
    rng = np.random.default_rng(19)
    B, K = 100_000, 3
    p = np.array([0.2, 0.5, 0.05, 0.25], dtype=np.float32)
    P = np.broadcast_to(p, (B, K + 1, 4))
    out, n_out = A.verify_chain(rng.integers(0, 4, size=(B, K)), P[:, :K], P, np.zeros(B, dtype=np.int64),
                                rng.random((B, K), dtype=np.float32), rng.random(B, dtype=np.float32))
    assert (n_out == 1).all() and (out[:, 1:] == -1).all()
    freq = np.bincount(out[:, 0], minlength=4) / B
    np.testing.assert_allclose(freq, p, atol=0.006)


def test_empty_batch():
    out, n_out = A.verify_chain(np.zeros((0, 3), dtype=np.int64), np.zeros((0, 3, 5)), np.zeros((0, 4, 5)),
                                np.zeros(0), np.zeros((0, 3)), np.zeros(0))
    assert out.shape == (0, 4) and n_out.shape == (0,)


def test_one_hot_target_run_length():
    rng = np.random.default_rng(20)
    B, K, V = 300, 5, 6
    amax = rng.integers(0, V, size=(B, K + 1))
    p = np.zeros((B, K + 1, V), dtype=np.float32)
    np.put_along_axis(p, amax[..., None], 1.0, axis=-1)
    q = rng.dirichlet(np.ones(V), size=(B, K)).astype(np.float32)
    q = np.maximum(q, 1e-3).astype(np.float32)
    draft = np.where(rng.random((B, K)) < 0.7, amax[:, :K], rng.integers(0, V, size=(B, K)))
    out, n_out = A.verify_chain(draft, q, p, np.full(B, K), rng.random((B, K), dtype=np.float32),
                                rng.random(B, dtype=np.float32))
    match = draft == amax[:, :K]
    run = np.cumprod(match, axis=1).sum(axis=1)
    np.testing.assert_array_equal(n_out, run + 1)
    np.testing.assert_array_equal(out[np.arange(B), run], amax[np.arange(B), run])


# ---------------------------------------------------------------- tree walk

def test_tree_walk_equals_chain_verifier():
    rng = np.random.default_rng(21)
    for V in [5, 64]:
        B, K = 400, 4
        p = rng.dirichlet(np.ones(V) * 0.5, size=(B, K + 1)).astype(np.float32)
        q = rng.dirichlet(np.ones(V) * 0.5, size=(B, K + 1)).astype(np.float32)
        q[:50] = p[:50]
        tokens = rng.integers(0, V, size=(B, K + 1))
        n_nodes = rng.integers(1, K + 2, size=B)
        ua = rng.random((B, K + 1), dtype=np.float32)
        uf = rng.random(B, dtype=np.float32)
        out_t, n_t, path = A.tree_accept_sample(p, q, tokens, np.arange(-1, K), n_nodes, ua, uf)
        out_c, n_c = A.verify_chain(tokens[:, 1:], q[:, :K], p, n_nodes - 1, ua[:, 1:], uf)
        np.testing.assert_array_equal(n_t, n_c)
        np.testing.assert_array_equal(out_t[:, :K + 1], out_c)
        for b in range(B):
            assert path[b, :n_t[b]].tolist() == list(range(n_t[b]))


TREES = {
    "two_iid_siblings": [(0,), (1,), (0, 0), (1, 0)],
    "three_iid_siblings": [(0,), (1,), (2,), (0, 0), (2, 0)],
}


@pytest.mark.parametrize("name", sorted(TREES))
def test_tree_lossless_chi_square(verifier_facts, name):
    V, _, n_tok, _, thr = _markov_facts(verifier_facts)
    parent, *_ = T.build_tree(TREES[name])
    pt, qt = W.markov_tables(V, 22)

    def verify(p, q, tokens, par, n_nodes, ua, uf):
        out, n_out, _ = A.tree_accept_sample(p, q, tokens, par, n_nodes, ua, uf)
        return out, n_out
    seqs = generate(verify, pt, qt, parent, 40_000, n_tok, 23)
    assert chi_square(seqs, pt) < thr


def test_tree_siblings_against_raw_target_fail(verifier_facts):
    V, _, n_tok, _, thr = _markov_facts(verifier_facts)
    parent, *_ = T.build_tree(TREES["three_iid_siblings"])
    pt, qt = W.markov_tables(V, 22)

    def verify(p, q, tokens, par, n_nodes, ua, uf):
        out, n_out, _ = A.tree_accept_sample(p, q, tokens, par, n_nodes, ua, uf, mutant="siblings_vs_p")
        return out, n_out
    seqs = generate(verify, pt, qt, parent, 40_000, n_tok, 23)
    assert chi_square(seqs, pt) > thr


# ---------------------------------------------------------------- processed distributions

def test_processing_helper():
    """The harness's sampler processing: identity at T = 1, top_p = 1; the
    softmax(logits / T) form; a hand-worked top-p cut."""
    rng = np.random.default_rng(24)
    t = rng.dirichlet(np.ones(6), size=5)
    np.testing.assert_allclose(processed(t), t, rtol=1e-6)
    logits = rng.standard_normal((3, 8))
    e = np.exp(logits / 0.6)
    np.testing.assert_allclose(processed(np.exp(logits) / np.exp(logits).sum(-1, keepdims=True), 0.6),
                               e / e.sum(-1, keepdims=True), rtol=1e-5)
    np.testing.assert_allclose(processed(np.array([[0.15, 0.5, 0.05, 0.3]]), 1.0, 0.8), [[0, 0.625, 0, 0.375]],
                               rtol=1e-6)
    np.testing.assert_allclose(processed(np.array([[0.15, 0.5, 0.05, 0.3]]), 1.0, 0.81),
                               [[0.15 / 0.95, 0.5 / 0.95, 0, 0.3 / 0.95]], rtol=1e-6)


def _processed_tables(V):
    pt, qt = W.markov_tables(V, 22)
    # the target samples at T = 0.8 with top-p 0.9; the drafter at its own T = 1.3, top-p 0.95
    return pt, qt, processed(pt, 0.8, 0.9), processed(qt, 1.3, 0.95)


def _tree_verify(p, q, tokens, par, n_nodes, ua, uf):
    out, n_out, _ = A.tree_accept_sample(p, q, tokens, par, n_nodes, ua, uf)
    return out, n_out


def test_processed_target_lossless(verifier_facts):
    scipy_stats = pytest.importorskip("scipy.stats")
    V, _, n_tok, _, _ = _markov_facts(verifier_facts)
    parent, *_ = T.build_tree(TREES["three_iid_siblings"])
    pt, qt, pp, qp = _processed_tables(V)
    seqs = generate(_tree_verify, pp, qp, parent, 40_000, n_tok, 23)
    stat, df, outside = chi_square_support(seqs, pp)
    assert outside == 0 and df < V ** n_tok - 1       # top-p removed some cells
    assert stat < scipy_stats.chi2.ppf(0.999, df)


@pytest.mark.parametrize("wrong", ["raw_p", "raw_q"])
def test_mismatched_processing_is_bias(verifier_facts, wrong):
    scipy_stats = pytest.importorskip("scipy.stats")
    V, _, n_tok, _, _ = _markov_facts(verifier_facts)
    parent, *_ = T.build_tree(TREES["three_iid_siblings"])
    pt, qt, pp, qp = _processed_tables(V)
    kw = {"pt_verify": pt} if wrong == "raw_p" else {"qt_verify": qt}
    seqs = generate(_tree_verify, pp, qp, parent, 40_000, n_tok, 23, **kw)
    stat, df, outside = chi_square_support(seqs, pp)
    assert stat > scipy_stats.chi2.ppf(0.999, df) or outside > 0
