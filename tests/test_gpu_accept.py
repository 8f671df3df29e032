"""GPU parity of tree acceptance against the oracle: bit-exact tokens, n_out
and paths for greedy (from logits or from target choices) and for the
stochastic walk given the same uniforms; plus the sampling page's
losslessness chi-square run end to end through the GPU kernel."""

import numpy as np
import pytest
import torch

from markov_harness import chi_square, chi_square_support, generate, processed
from oracle import accept as OA
from oracle import tree as OT
from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _cmp(gpu, ref_out, ref_n, ref_path, out_cols=None):
    out, n_out, path = (t.cpu().numpy() for t in gpu)
    np.testing.assert_array_equal(n_out, ref_n)
    k = ref_out.shape[1] if out_cols is None else out_cols
    np.testing.assert_array_equal(out[:, :k], ref_out[:, :k])
    np.testing.assert_array_equal(path[:, :k], ref_path[:, :k])


@pytest.mark.parametrize("name", ["tiny_b1_f32", "gqa_b8_l512_2048_n26", "b64_l1k_8k_n64_greedy"])
def test_greedy_from_logits_bit_exact(name):
    w = W.WORKLOADS[name]
    parent, *_ = OT.build_tree(w.paths())
    g = W.greedy_inputs(w, parent, device="cuda")
    par = torch.from_numpy(parent.astype(np.int32)).cuda()
    res = capi.tv_tree_accept_greedy(g["tokens"], par, logits=g["logits"])
    am = OA.argmax_rows(g["logits"].cpu().numpy())
    ref = OA.tree_accept_greedy(am, g["tokens"].cpu().numpy(), parent)
    _cmp(res, *ref)
    assert res[1].float().mean().item() > 1.0


def test_greedy_ties_and_target_choices():
    V, N = 1000, 10
    parent, *_ = OT.build_tree(W.PAGE_TREE_PATHS)
    rng = np.random.default_rng(110)
    B = 300
    tokens = rng.integers(0, 5, size=(B, N)).astype(np.int32)
    logits = rng.integers(0, 4, size=(B, N, V)).astype(np.float32)      # many ties
    par = torch.from_numpy(parent.astype(np.int32)).cuda()
    res = capi.tv_tree_accept_greedy(torch.from_numpy(tokens).cuda(), par, logits=torch.from_numpy(logits).cuda())
    am = OA.argmax_rows(logits)
    _cmp(res, *OA.tree_accept_greedy(am, tokens, parent))
    am2 = rng.integers(0, 5, size=(B, N)).astype(np.int32)
    n_nodes = rng.integers(1, N + 1, size=B).astype(np.int32)
    res = capi.tv_tree_accept_greedy(torch.from_numpy(tokens).cuda(), par, target_argmax=torch.from_numpy(am2).cuda(),
                                     n_nodes=torch.from_numpy(n_nodes).cuda())
    _cmp(res, *OA.tree_accept_greedy(am2, tokens, parent, n_nodes))


def test_greedy_odd_vocab_and_per_request_parents():
    rng = np.random.default_rng(111)
    B, N, V = 40, 20, 997
    parents = np.stack([OT.build_tree(W.random_rank_paths(N, 5, rng))[0] for _ in range(B)]).astype(np.int32)
    tokens = rng.integers(0, 3, size=(B, N)).astype(np.int32)
    logits = rng.standard_normal((B, N, V)).astype(np.float32)
    logits[..., :3] += 2.5
    res = capi.tv_tree_accept_greedy(torch.from_numpy(tokens).cuda(), torch.from_numpy(parents).cuda(),
                                     logits=torch.from_numpy(logits).cuda())
    _cmp(res, *OA.tree_accept_greedy(OA.argmax_rows(logits), tokens, parents))


def test_greedy_overflow_flag():
    parent = np.arange(-1, 7).astype(np.int32)
    tokens = np.full((1, 8), 5, dtype=np.int32)
    am = np.full((1, 8), 5, dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, n_out, path = capi.tv_tree_accept_greedy(torch.from_numpy(tokens).cuda(), torch.from_numpy(parent).cuda(),
                                                  target_argmax=torch.from_numpy(am).cuda(), out_cols=3,
                                                  status=status)
    assert status.item() == capi.TV_DEV_OUT_OVERFLOW and n_out.item() == 3


KERNELS = {"auto": 0, "cluster": 1, "single_cta": 2, "stream": 3, "grid": 4, "auto_ws": 0}


def _kw(kernel, B, N, V):
    """flags of one kernel choice, with a workspace for the grid sampler and
    for TV_SAMPLE_AUTO allowed to pick it ("auto_ws")."""
    kw = {"flags": KERNELS[kernel]}
    if kernel in ("grid", "auto_ws"):
        kw["workspace"] = capi.alloc_workspace(capi.tv_accept_sample_workspace_size(B, N, V))
    return kw


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_sample_full_workload_bit_exact(kernel):
    """B=256 chains over a 128000-token vocabulary, ragged num_draft ~ U{0..4}."""
    w = W.WORKLOADS["b256_l2k_4k_n10_sample"]
    s = W.sample_chain_inputs(w, device="cuda")
    kw = _kw(kernel, *s["p"].shape)
    res = capi.tv_tree_accept_sample(s["p"], s["q"], s["tokens"], s["parent"], s["u_accept"], s["u_final"],
                                     n_nodes=s["n_nodes"], **kw)
    c = {k: v.cpu().numpy() for k, v in s.items()}
    ref = OA.tree_accept_sample(c["p"], c["q"], c["tokens"], c["parent"], c["n_nodes"], c["u_accept"], c["u_final"])
    _cmp(res, *ref)
    K = c["p"].shape[1] - 1
    out_c, n_c = OA.verify_chain(c["tokens"][:, 1:], c["q"][:, :K], c["p"], c["n_nodes"] - 1, c["u_accept"][:, 1:],
                                 c["u_final"])
    np.testing.assert_array_equal(res[1].cpu().numpy(), n_c)
    # the chain call reads the page's arrays in place: the same bits
    out2, n2 = capi.tv_chain_accept_sample(s["p"], s["q"][:, :K].contiguous(), s["tokens"][:, 1:].contiguous(),
                                           s["u_accept"][:, 1:].contiguous(), s["u_final"],
                                           num_draft=(s["n_nodes"] - 1).contiguous(), **kw)
    np.testing.assert_array_equal(n2.cpu().numpy(), n_c)
    np.testing.assert_array_equal(out2.cpu().numpy(), out_c)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_sample_tree_full_workload_bit_exact(kernel):
    """B=64 requests verified stochastically on the 64-node tree over a
    32000-token vocabulary, siblings drawn i.i.d. from their parent's q."""
    w = W.WORKLOADS["b64_l1k_8k_n64_sample"]
    parent, *_ = OT.build_tree(w.paths())
    s = W.sample_tree_inputs(w, parent, device="cuda")
    res = capi.tv_tree_accept_sample(s["p"], s["q"], s["tokens"], s["parent"], s["u_accept"], s["u_final"],
                                     n_nodes=s["n_nodes"], **_kw(kernel, *s["p"].shape))
    c = {k: v.cpu().numpy() for k, v in s.items()}
    ref = OA.tree_accept_sample(c["p"], c["q"], c["tokens"], c["parent"], c["n_nodes"], c["u_accept"], c["u_final"])
    _cmp(res, *ref)
    # walks leave the root's level and end both by rejection and at leaves
    n = res[1].cpu().numpy()
    assert n.mean() > 2.0 and n.min() >= 1


@pytest.mark.parametrize("V,B,kernel",
                         [(V, 200, k) for V in (4, 33, 1000, 4096) for k in ("cluster", "single_cta", "stream", "grid")]
                         + [(V, 12, k) for V in (160000, 160001) for k in ("auto", "single_cta", "grid")])
def test_sample_trees_with_sibling_levels(V, B, kernel):
    """Trees with up to 5 siblings per node: several residual levels per node,
    on every kernel.  Vocabularies above 136,512 have no on-chip-state
    cluster kernel (aligned rows and odd V both)."""
    rng = np.random.default_rng(120 + V)
    N = 16
    paths = [(0,), (1,), (2,), (3,), (4,), (0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (4, 0), (0, 0, 0), (0, 0, 1),
             (0, 1, 0), (1, 0, 0)]
    parent, *_ = OT.build_tree(paths)
    p = rng.dirichlet(np.ones(V) * 0.3, size=(B, N)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.3, size=(B, N)).astype(np.float32)
    q[:20] = p[:20]
    tokens = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        for c in range(1, N):
            row = q[b, parent[c]].astype(np.float64)
            tokens[b, c] = rng.choice(V, p=row / row.sum())
    n_nodes = rng.integers(1, N + 1, size=B).astype(np.int32)
    ua = rng.random((B, N), dtype=np.float32)
    uf = rng.random(B, dtype=np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    res = capi.tv_tree_accept_sample(t(p), t(q), t(tokens), t(parent.astype(np.int32)), t(ua), t(uf),
                                     n_nodes=t(n_nodes), **_kw(kernel, B, N, V))
    _cmp(res, *OA.tree_accept_sample(p, q, tokens, parent, n_nodes, ua, uf))
    if V > 136512:
        with pytest.raises(capi.TVError, match="UNSUPPORTED"):
            capi.tv_tree_accept_sample(t(p), t(q), t(tokens), t(parent.astype(np.int32)), t(ua), t(uf),
                                       flags=capi.TV_SAMPLE_CLUSTER)


@pytest.mark.parametrize("V,kernel", [(4096, "cluster"), (4096, "single_cta"), (4096, "stream"), (4096, "grid"),
                                      (160000, "auto"), (160000, "single_cta"), (160000, "grid")])
def test_sample_kept_level_after_empty_residual(V, kernel):
    """A rejection whose residual pass leaves no mass keeps the level (the
    p = q guard) and the final draw still uses that level's weights: q is
    one-hot at token t and p puts 1.5 on t (rows may sum to 2), the children
    carry tokens with q = 0, so the second and third rejections find an
    empty residual."""
    t = V * 3 // 4 + 1
    B, N = 2, 4
    parent = np.array([-1, 0, 0, 0], dtype=np.int32)
    p = np.zeros((B, N, V), dtype=np.float32)
    q = np.zeros((B, N, V), dtype=np.float32)
    p[:, :, t] = 1.5
    q[:, :, t] = 1.0
    tokens = np.array([[0, 7, 7, 9]] * B, dtype=np.int32)
    ua = np.full((B, N), 0.5, dtype=np.float32)
    uf = np.array([0.3, 0.9], dtype=np.float32)
    n_nodes = np.full(B, N, dtype=np.int32)
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    res = capi.tv_tree_accept_sample(tt(p), tt(q), tt(tokens), tt(parent), tt(ua), tt(uf), n_nodes=tt(n_nodes),
                                     **_kw(kernel, B, N, V))
    ref = OA.tree_accept_sample(p, q, tokens, parent, n_nodes, ua, uf)
    _cmp(res, *ref)
    assert (ref[1] == 1).all() and (ref[0][:, 0] == t).all()


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_sample_chain_empty_residual_draws_from_p(kernel):
    """A chain whose only child is rejected with an empty residual: p = q
    rows and a draft token both give probability 0 (u q(x) < p(x) fails at
    0 < 0), so max(0, P - Q) sums to 0, the level is kept and the
    replacement is drawn from p itself; the other requests accept every
    draft (u < 1 with p(x) = q(x) > 0) and draw the bonus."""
    rng = np.random.default_rng(150)
    B, N, V = 40, 4, 3000
    parent = np.arange(-1, N - 1, dtype=np.int32)
    p = rng.dirichlet(np.ones(V) * 0.5, size=(B, N)).astype(np.float32)
    p[:, :, 17] = 0.0
    q = p.copy()
    tokens = rng.integers(18, V, size=(B, N)).astype(np.int32)
    tokens[: B // 2, 2] = 17  # the second draft is rejected with nothing left
    ua = rng.random((B, N), dtype=np.float32)
    uf = rng.random(B, dtype=np.float32)
    n_nodes = np.full(B, N, dtype=np.int32)
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    res = capi.tv_tree_accept_sample(tt(p), tt(q), tt(tokens), tt(parent), tt(ua), tt(uf), n_nodes=tt(n_nodes),
                                     **_kw(kernel, B, N, V))
    ref = OA.tree_accept_sample(p, q, tokens, parent, n_nodes, ua, uf)
    _cmp(res, *ref)
    assert (ref[1][: B // 2] == 2).all() and (ref[1][B // 2:] == N).all()


def test_sample_truncated_walk_same_on_every_kernel():
    """out_cols shorter than the accepted chain: every kernel flags
    TV_DEV_OUT_OVERFLOW and returns the same first out_cols tokens as the
    oracle's walk, without the final draw."""
    rng = np.random.default_rng(151)
    B, N, V, cols = 30, 6, 2000, 3
    parent = np.arange(-1, N - 1, dtype=np.int32)
    p = rng.dirichlet(np.ones(V), size=(B, N)).astype(np.float32)
    rows = p.astype(np.float64)
    rows /= rows.sum(axis=2, keepdims=True)
    tokens = np.stack([[rng.choice(V, p=rows[b, max(c - 1, 0)]) for c in range(N)] for b in range(B)]).astype(np.int32)
    ua = rng.random((B, N), dtype=np.float32)
    uf = rng.random(B, dtype=np.float32)
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ref = OA.tree_accept_sample(p, p, tokens, parent, np.full(B, N, np.int32), ua, uf)
    assert (ref[1] == N).all()  # q = p: every draft is accepted
    for kernel in sorted(KERNELS):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, n_out, path = capi.tv_tree_accept_sample(tt(p), tt(p), tt(tokens), tt(parent), tt(ua), tt(uf),
                                                      out_cols=cols, status=status, **_kw(kernel, B, N, V))
        assert status.item() == capi.TV_DEV_OUT_OVERFLOW, kernel
        assert (n_out.cpu().numpy() == cols).all(), kernel
        np.testing.assert_array_equal(out.cpu().numpy(), ref[0][:, :cols])
        np.testing.assert_array_equal(path.cpu().numpy(), ref[2][:, :cols])


def test_grid_sampler_arguments():
    """The grid sampler needs a large enough, 16-byte aligned workspace and
    V <= 2^20; TV_SAMPLE_AUTO without one keeps to the single-launch
    kernels."""
    B, N, V = 3, 2, 500
    p = torch.full((B, N, V), 1.0 / V, device="cuda")
    tokens = torch.zeros(B, N, dtype=torch.int32, device="cuda")
    parent = torch.tensor([-1, 0], dtype=torch.int32, device="cuda")
    ua, uf = torch.zeros(B, N, device="cuda"), torch.full((B,), 0.5, device="cuda")
    need = capi.tv_accept_sample_workspace_size(B, N, V)
    assert need == 16 * B + 16 * B * 1
    call = lambda **kw: capi.tv_tree_accept_sample(p, p, tokens, parent, ua, uf, **kw)
    with pytest.raises(capi.TVError, match="INVALID_ARG"):
        call(flags=capi.TV_SAMPLE_GRID)
    with pytest.raises(capi.TVError, match="INVALID_ARG"):
        call(flags=capi.TV_SAMPLE_GRID, workspace=capi.alloc_workspace(need)[: need - 16])
    with pytest.raises(capi.TVError, match="INVALID_ARG"):
        call(flags=capi.TV_SAMPLE_GRID, workspace=capi.alloc_workspace(need + 64)[8: need + 8])
    with pytest.raises(capi.TVError, match="INVALID_ARG"):
        call(flags=5, workspace=capi.alloc_workspace(need))
    big = torch.full((1, 1, (1 << 20) + 1), 0.5 ** 20, device="cuda")
    z = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.TVError, match="UNSUPPORTED"):
        capi.tv_tree_accept_sample(big, big, z, parent[:1], torch.zeros(1, 1, device="cuda"), uf[:1],
                                   flags=capi.TV_SAMPLE_GRID,
                                   workspace=capi.alloc_workspace(capi.tv_accept_sample_workspace_size(1, 1, big.shape[2])))
    ref = call(flags=capi.TV_SAMPLE_SINGLE_CTA)
    for kw in ({}, {"flags": capi.TV_SAMPLE_GRID, "workspace": capi.alloc_workspace(need)}):
        for a, b in zip(call(**kw), ref):
            assert torch.equal(a, b)


def test_sample_bad_token_flag():
    p = torch.full((1, 2, 8), 0.125, device="cuda")
    tokens = torch.tensor([[0, 9]], dtype=torch.int32, device="cuda")
    parent = torch.tensor([-1, 0], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, n_out, path = capi.tv_tree_accept_sample(p, p, tokens, parent, torch.zeros(1, 2, device="cuda"),
                                                  torch.full((1,), 0.5, device="cuda"), status=status)
    assert status.item() == capi.TV_DEV_BAD_TOKEN and n_out.item() == 1


def _gpu_verify(p, q, tokens, parent, n_nodes, ua, uf, kernel="auto"):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out, n_out, _ = capi.tv_tree_accept_sample(t(p), t(q), t(tokens.astype(np.int32)), t(parent.astype(np.int32)),
                                               t(ua), t(uf), n_nodes=t(n_nodes.astype(np.int32)),
                                               **_kw(kernel, *p.shape))
    return out.cpu().numpy(), n_out.cpu().numpy()


def test_gpu_chain_lossless_chi_square(verifier_facts):
    f = verifier_facts
    V, n_seq = int(f["chi2_vocab"][0][0]), int(f["chi2_sequences"][0][0])
    n_tok, K, thr = int(f["chi2_tokens"][0][0]), int(f["chi2_drafts_per_round"][0][0]), float(f["chi2_threshold"][0][0])
    pt, qt = W.markov_tables(V, 16)
    seqs = generate(_gpu_verify, pt, qt, np.arange(-1, K), n_seq, n_tok, 130)
    assert chi_square(seqs, pt) < thr


@pytest.mark.parametrize("kernel", ["cluster", "single_cta", "stream", "grid"])
def test_gpu_tree_lossless_chi_square(verifier_facts, kernel):
    f = verifier_facts
    V, n_tok, thr = int(f["chi2_vocab"][0][0]), int(f["chi2_tokens"][0][0]), float(f["chi2_threshold"][0][0])
    parent, *_ = OT.build_tree([(0,), (1,), (2,), (0, 0), (2, 0)])
    pt, qt = W.markov_tables(V, 22)
    verify = lambda *a: _gpu_verify(*a, kernel=kernel)
    seqs = generate(verify, pt, qt, parent, 200_000, n_tok, 131)
    assert chi_square(seqs, pt) < thr


def test_gpu_sample_processed_target_lossless(verifier_facts):
    """Temperature / top-p processed target and drafter rows: the GPU walk's
    output follows the processed target."""
    scipy_stats = pytest.importorskip("scipy.stats")
    f = verifier_facts
    V, n_tok = int(f["chi2_vocab"][0][0]), int(f["chi2_tokens"][0][0])
    parent, *_ = OT.build_tree([(0,), (1,), (2,), (0, 0), (2, 0)])
    pt, qt = W.markov_tables(V, 22)
    pp, qp = processed(pt, 0.8, 0.9), processed(qt, 1.3, 0.95)
    seqs = generate(_gpu_verify, pp, qp, parent, 100_000, n_tok, 132)
    stat, df, outside = chi_square_support(seqs, pp)
    assert outside == 0 and stat < scipy_stats.chi2.ppf(0.999, df)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_sample_edge_shapes(kernel):
    """A one-token vocabulary (every draw is token 0), a root-only tree (the
    bonus draw only) and a large batch (2048 requests), on every kernel."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    rng = np.random.default_rng(140)
    cases = []
    B, N = 5, 4
    cases.append((np.ones((B, N, 1), np.float32), np.ones((B, N, 1), np.float32), np.zeros((B, N), np.int32),
                  np.arange(-1, N - 1, dtype=np.int32)))
    B, N, V = 7, 1, 300
    p = rng.dirichlet(np.ones(V), size=(B, N)).astype(np.float32)
    cases.append((p, p.copy(), np.zeros((B, N), np.int32), np.array([-1], np.int32)))
    B, N, V = 2048, 4, 1000
    p = rng.dirichlet(np.ones(V) * 0.5, size=(B, N)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=(B, N)).astype(np.float32)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    cases.append((p, q, tok, np.array([-1, 0, 0, 1], np.int32)))
    for p, q, tok, par in cases:
        B, N, V = p.shape
        n_nodes = rng.integers(1, N + 1, size=B).astype(np.int32)
        ua = rng.random((B, N), dtype=np.float32)
        uf = rng.random(B, dtype=np.float32)
        res = capi.tv_tree_accept_sample(t(p), t(q), t(tok), t(par), t(ua), t(uf), n_nodes=t(n_nodes),
                                         **_kw(kernel, B, N, V))
        _cmp(res, *OA.tree_accept_sample(p, q, tok, par, n_nodes, ua, uf))
        if V == 1:
            assert (res[0].cpu().numpy()[:, 0] == 0).all()


def test_greedy_edge_shapes():
    """Root-only trees, a one-token vocabulary and a large batch."""
    rng = np.random.default_rng(141)
    for B, N, V in ((9, 1, 500), (6, 5, 1), (4096, 3, 64)):
        parent = np.arange(-1, N - 1, dtype=np.int32)
        tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
        logits = rng.standard_normal((B, N, V)).astype(np.float32)
        par = torch.from_numpy(parent).cuda()
        res = capi.tv_tree_accept_greedy(torch.from_numpy(tokens).cuda(), par, logits=torch.from_numpy(logits).cuda())
        _cmp(res, *OA.tree_accept_greedy(OA.argmax_rows(logits), tokens, parent))


def test_page_interfaces():
    """The pages' own call shapes: the chain verifier verify(draft, q, p,
    num_draft, u, u_final) and accept_greedy(parent, tokens, target_argmax),
    against the oracle."""
    rng = np.random.default_rng(142)
    B, K, V = 300, 5, 700
    p = rng.dirichlet(np.ones(V) * 0.4, size=(B, K + 1)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.4, size=(B, K)).astype(np.float32)
    q[:30] = p[:30, :K]
    draft = np.stack([[rng.choice(V, p=q[b, j] / q[b, j].sum()) for j in range(K)] for b in range(B)]).astype(np.int32)
    nd = rng.integers(0, K + 1, size=B).astype(np.int32)
    u = rng.random((B, K), dtype=np.float32)
    uf = rng.random(B, dtype=np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out, n_out = capi.verify_chain(t(draft), t(q), t(p), t(nd), t(u), t(uf))
    r_out, r_n = OA.verify_chain(draft, q, p, nd, u, uf)
    np.testing.assert_array_equal(n_out.cpu().numpy(), r_n)
    np.testing.assert_array_equal(out.cpu().numpy(), r_out)
    parent, *_ = OT.build_tree(W.PAGE_TREE_PATHS)
    tokens = rng.integers(0, 4, size=(B, parent.size)).astype(np.int32)
    am = rng.integers(0, 4, size=(B, parent.size)).astype(np.int32)
    res = capi.accept_greedy(t(parent.astype(np.int32)), t(tokens), t(am))
    _cmp(res, *OA.tree_accept_greedy(am, tokens, parent))


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_chain_call_allocates_nothing(kernel):
    """verify_chain with its outputs passed in allocates no device memory
    (neither through PyTorch nor behind it) and matches the oracle bit for
    bit, with num_draft given or not and for K = 0 (bonus draw only)."""
    rng = np.random.default_rng(143)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    for B, K, V, give_nd in ((64, 7, 5000, True), (64, 7, 5000, False), (9, 0, 333, True)):
        p = rng.dirichlet(np.ones(V) * 0.3, size=(B, K + 1)).astype(np.float32)
        q = rng.dirichlet(np.ones(V) * 0.3, size=(B, K)).astype(np.float32)
        q[:B // 4] = p[:B // 4, :K]
        draft = np.stack([[rng.choice(V, p=q[b, j] / q[b, j].sum()) for j in range(K)] for b in range(B)]
                         ).astype(np.int32).reshape(B, K)
        nd = rng.integers(0, K + 1, size=B).astype(np.int32) if give_nd else np.full(B, K, np.int32)
        u = rng.random((B, K), dtype=np.float32)
        uf = rng.random(B, dtype=np.float32)
        args = [t(draft), t(q), t(p), t(nd) if give_nd else None, t(u), t(uf)]
        out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
        n_out = torch.empty(B, dtype=torch.int32, device="cuda")
        kw = _kw(kernel, B, K + 1, V)
        capi.verify_chain(*args, out=out, n_out=n_out, **kw)  # first call: one-time set-up
        r = None  # drop the previous case's outputs before counting
        torch.cuda.synchronize()
        alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        for _ in range(3):
            r = capi.verify_chain(*args, out=out, n_out=n_out, **kw)
        torch.cuda.synchronize()
        assert r[0] is out and r[1] is n_out
        assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.mem_get_info()[0] == free0
        r_out, r_n = OA.verify_chain(draft, q, p, nd, u, uf)
        np.testing.assert_array_equal(n_out.cpu().numpy(), r_n)
        np.testing.assert_array_equal(out.cpu().numpy(), r_out)
