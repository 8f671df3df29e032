"""Pins for the oracle's RoPE and tree attention (CPU only).

The oracle computes each node separately over its own root-to-node path.  It
is pinned here against other formulations:

* RoPE equals multiplication of (x1 + i x2) by exp(i angle) (complex numbers),
  keeps norms and makes dot products depend only on the position difference;
* an empty tree (root only) is textbook decode attention over L + 1 keys and a
  chain tree is ordinary causal attention (torch's scaled_dot_product_attention
  in float64);
* a general tree equals ONE masked pass over [prefix | all nodes] with the
  ancestor mask and depth positions (the "Tree Verification" correctness
  condition), computed with torch's masked scaled_dot_product_attention;
* with ``rotate=False`` (queries and tree keys given already rotated) a
  general tree is the same one masked pass with no rotation at all, and
  rotating the inputs first at L + depth reproduces the default;
* permuting the physical blocks of the paged cache changes nothing;
* the two mistakes the mask page lists (causal mask over flattened nodes,
  sequential positions) move outputs by far more than the bf16 tolerance, so
  a parity test against this oracle can fail.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle import tree as T
from speculative_decoding_tree_attn_gb300 import workloads as W


def test_rope_is_complex_rotation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 64))
    pos = np.array([0, 1, 7, 1000, 32775])
    got = A.rope(x, pos)
    ang = A.rope_angles(pos, 64)
    z = (x[:, :32] + 1j * x[:, 32:]) * np.exp(1j * ang)
    np.testing.assert_allclose(got, np.concatenate([z.real, z.imag], -1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(A.rope(x, 0), x, atol=0)
    np.testing.assert_allclose(np.linalg.norm(got, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    # the frequency of pair k is base ** (-2k / D)
    np.testing.assert_allclose(A.rope_angles(1, 64)[[0, 1, 31]],
                               [1.0, 10000 ** (-2 / 64), 10000 ** (-62 / 64)], rtol=1e-15)


def test_rope_relative_positions():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((2, 128))
    for m, n, s in [(3, 1, 5), (100, 40, 1000), (32768, 12, 7)]:
        a = A.rope(q, m) @ A.rope(k, n)
        b = A.rope(q, m + s) @ A.rope(k, n + s)
        assert abs(a - b) < 1e-9


def _sdpa(qm, km, vm, mask=None, causal=False):
    """torch SDPA in float64 on [H, T, D] tensors."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).double()
    o = F.scaled_dot_product_attention(t(qm)[None], t(km)[None], t(vm)[None],
                                       attn_mask=None if mask is None else torch.from_numpy(mask)[None],
                                       is_causal=causal)
    return o[0].numpy()


def _case(B, N, Hq, Hkv, D, lens, bs, seed, paths=None):
    w = W.Workload("t", B, Hq, Hkv, D, "f32", ("fixed", 0), bs, (0.7, 0.15), N, 8, seed)
    inp = W.attention_inputs(w, seq_lens=lens)
    return {k: v.numpy() for k, v in inp.items()}


def test_empty_tree_is_decode_attention():
    inp = _case(2, 1, 4, 2, 32, [19, 0], 8, 3)
    parent = np.array([-1])
    out, lse = A.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                inp["seq_lens"], inp["k_tree"], inp["v_tree"], parent)
    for b in range(2):
        L = int(inp["seq_lens"][b])
        pk = A.gather_prefix(inp["k_cache"], inp["block_table"][b], L)
        pv = A.gather_prefix(inp["v_cache"], inp["block_table"][b], L)
        keys = np.concatenate([pk, A.rope(inp["k_tree"][b, :1], L)], 0)   # [L+1, Hkv, D]
        vals = np.concatenate([pv, inp["v_tree"][b, :1]], 0)
        qr = A.rope(inp["q"][b, 0], L)                                     # [Hq, D]
        kh = np.repeat(keys.transpose(1, 0, 2), 2, axis=0)
        vh = np.repeat(vals.transpose(1, 0, 2), 2, axis=0)
        ref = _sdpa(qr[:, None, :], kh, vh)[:, 0]
        np.testing.assert_allclose(out[b, 0], ref, rtol=0, atol=1e-12)


def test_chain_tree_is_causal_attention():
    N = 6
    inp = _case(1, N, 2, 1, 16, [11], 4, 4)
    parent = np.arange(-1, N - 1)
    out, _ = A.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                              inp["seq_lens"], inp["k_tree"], inp["v_tree"], parent)
    L = 11
    pk = A.gather_prefix(inp["k_cache"], inp["block_table"][0], L)
    pv = A.gather_prefix(inp["v_cache"], inp["block_table"][0], L)
    pos = L + np.arange(N)
    keys = np.concatenate([pk, A.rope(inp["k_tree"][0], pos[:, None])], 0)[:, 0]   # [L+N, D]
    vals = np.concatenate([pv, inp["v_tree"][0]], 0)[:, 0]
    qs = A.rope(inp["q"][0], pos[:, None]).transpose(1, 0, 2)                        # [Hq, N, D]
    # causal rows L..L+N-1 of a causal pass: queries at the end of the sequence
    mask = np.tril(np.ones((L + N, L + N), dtype=bool))[L:]
    ref = _sdpa(qs, np.repeat(keys[None], 2, 0), np.repeat(vals[None], 2, 0), mask=mask)
    np.testing.assert_allclose(out[0].transpose(1, 0, 2), ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [5, 6, 7])
def test_tree_equals_one_masked_pass(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(2, 40))
    paths = W.random_rank_paths(N, 6, rng)
    parent, depth, rows, _ = T.build_tree(paths)
    Hq, Hkv, D = 6, 2, 32
    lens = [int(x) for x in rng.integers(0, 50, size=2)]
    inp = _case(2, N, Hq, Hkv, D, lens, 8, seed)
    out, lse = A.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                inp["seq_lens"], inp["k_tree"], inp["v_tree"], parent)
    tm = T.dense_mask(rows, N)
    for b in range(2):
        L = lens[b]
        pos = T.positions(depth, L)
        pk = A.gather_prefix(inp["k_cache"], inp["block_table"][b], L)
        pv = A.gather_prefix(inp["v_cache"], inp["block_table"][b], L)
        keys = np.concatenate([pk, A.rope(inp["k_tree"][b], pos[:, None])], 0)   # [L+N, Hkv, D]
        vals = np.concatenate([pv, inp["v_tree"][b]], 0)
        qs = A.rope(inp["q"][b], pos[:, None]).transpose(1, 0, 2)                 # [Hq, N, D]
        full = np.concatenate([np.ones((N, L), dtype=bool), tm], 1)              # [N, L+N]
        G = Hq // Hkv
        kh = np.repeat(keys.transpose(1, 0, 2), G, 0)
        vh = np.repeat(vals.transpose(1, 0, 2), G, 0)
        ref = _sdpa(qs, kh, vh, mask=full)
        np.testing.assert_allclose(out[b].transpose(1, 0, 2), ref, rtol=0, atol=1e-11)
        s = np.einsum("hnd,htd->hnt", qs, kh) / np.sqrt(D)
        s = np.where(full[None], s, -np.inf)
        ref_lse = torch.logsumexp(torch.from_numpy(s), dim=-1).numpy()
        np.testing.assert_allclose(lse[b].transpose(1, 0), ref_lse, rtol=0, atol=1e-11)


@pytest.mark.parametrize("seed", [15, 16])
def test_prerotated_inputs_are_one_masked_pass_without_rope(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(2, 40))
    paths = W.random_rank_paths(N, 6, rng)
    parent, depth, rows, _ = T.build_tree(paths)
    Hq, Hkv, D = 6, 2, 32
    lens = [int(x) for x in rng.integers(0, 50, size=2)]
    inp = _case(2, N, Hq, Hkv, D, lens, 8, seed)
    out, lse = A.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                inp["seq_lens"], inp["k_tree"], inp["v_tree"], parent, rotate=False)
    tm = T.dense_mask(rows, N)
    G = Hq // Hkv
    for b in range(2):
        L = lens[b]
        pk = A.gather_prefix(inp["k_cache"], inp["block_table"][b], L)
        pv = A.gather_prefix(inp["v_cache"], inp["block_table"][b], L)
        keys = np.concatenate([pk, np.asarray(inp["k_tree"][b], dtype=np.float64)], 0)
        vals = np.concatenate([pv, np.asarray(inp["v_tree"][b], dtype=np.float64)], 0)
        qs = np.asarray(inp["q"][b], dtype=np.float64).transpose(1, 0, 2)
        full = np.concatenate([np.ones((N, L), dtype=bool), tm], 1)
        kh = np.repeat(keys.transpose(1, 0, 2), G, 0)
        vh = np.repeat(vals.transpose(1, 0, 2), G, 0)
        np.testing.assert_allclose(out[b].transpose(1, 0, 2), _sdpa(qs, kh, vh, mask=full), rtol=0, atol=1e-11)
        s = np.einsum("hnd,htd->hnt", qs, kh) / np.sqrt(D)
        ref_lse = torch.logsumexp(torch.from_numpy(np.where(full[None], s, -np.inf)), dim=-1).numpy()
        np.testing.assert_allclose(lse[b].transpose(1, 0), ref_lse, rtol=0, atol=1e-11)
    # rotating q and the tree keys at L + depth first gives the default mode
    pos = np.stack([T.positions(depth, L) for L in lens])                         # [B, N]
    q_rot = A.rope(inp["q"], pos[:, :, None])
    kt_rot = A.rope(inp["k_tree"], pos[:, :, None])
    out2, lse2 = A.tree_attention(q_rot, inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                                  kt_rot, inp["v_tree"], parent, rotate=False)
    out1, lse1 = A.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                                  inp["k_tree"], inp["v_tree"], parent)
    np.testing.assert_allclose(out2, out1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse1, rtol=0, atol=1e-12)


def test_gather_prefix_position_by_position():
    """Prefix position t is slot t % block_size of block block_table[t // block_size]."""
    rng = np.random.default_rng(21)
    nb, Hkv, bs, D = 9, 3, 4, 5
    cache = rng.standard_normal((nb, Hkv, bs, D))
    row = rng.permutation(nb)
    for L in (0, 1, 3, 4, 5, 17, 36):
        got = A.gather_prefix(cache, row, L)
        assert got.shape == (L, Hkv, D)
        for t in range(L):
            assert np.array_equal(got[t], cache[row[t // bs], :, t % bs, :])
        heads = A.gather_prefix_heads(cache, row, L)
        assert np.array_equal(heads, got.transpose(1, 0, 2))


def test_block_permutation_invariance():
    rng = np.random.default_rng(8)
    parent, depth, rows, _ = T.build_tree(W.PAGE_TREE_PATHS)
    inp = _case(2, 10, 4, 2, 32, [40, 23], 8, 8)
    a, _ = A.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                            inp["seq_lens"], inp["k_tree"], inp["v_tree"], parent)
    perm = rng.permutation(inp["k_cache"].shape[0])
    inv = np.argsort(perm)
    b, _ = A.tree_attention(inp["q"], inp["k_cache"][perm], inp["v_cache"][perm], inv[inp["block_table"]],
                            inp["seq_lens"], inp["k_tree"], inp["v_tree"], parent)
    np.testing.assert_allclose(a, b, rtol=0, atol=0)


@pytest.mark.parametrize("mutant", ["causal_flat", "sequential_positions"])
@pytest.mark.parametrize("L", [0, 1, 16, 65])
def test_negative_controls_fail_bf16_tolerance(mutant, L):
    parent, depth, rows, _ = T.build_tree(W.PAGE_TREE_PATHS)
    inp = _case(1, 10, 4, 1, 64, [L], 16, 9)
    good, _ = A.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                               inp["seq_lens"], inp["k_tree"], inp["v_tree"], parent)
    bad, _ = A.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                              inp["seq_lens"], inp["k_tree"], inp["v_tree"], parent, mutant=mutant)
    assert np.abs(good - bad).max() > 10 * 2e-2


def test_ragged_absent_nodes_and_empty_key_set():
    """Absent nodes of a ragged tree: the prefix alone, with the query as
    given; with an empty prefix no key at all -- a zero row and lse -inf.
    Valid rows equal the truncated tree's rows."""
    rng = np.random.default_rng(78)
    N, Hq, Hkv, D, bs = 6, 4, 2, 8, 4
    parent = np.array([-1, 0, 0, 1, 1, 3])
    for L in (0, 7):
        nb = max((L + bs - 1) // bs, 1)
        kc = rng.standard_normal((nb, Hkv, bs, D))
        vc = rng.standard_normal((nb, Hkv, bs, D))
        q = rng.standard_normal((1, N, Hq, D))
        kt = rng.standard_normal((1, N, Hkv, D))
        vt = rng.standard_normal((1, N, Hkv, D))
        table = np.arange(nb)[None]
        out, lse = A.tree_attention(q, kc, vc, table, np.array([L]), kt, vt, parent, n_nodes=[4])
        full, flse = A.tree_attention(q[:, :4], kc, vc, table, np.array([L]), kt[:, :4], vt[:, :4], parent[:4])
        np.testing.assert_array_equal(out[0, :4], full[0])
        np.testing.assert_array_equal(lse[0, :4], flse[0])
        if L == 0:
            assert (out[0, 4:] == 0).all() and np.isneginf(lse[0, 4:]).all()
        else:
            # prefix-only softmax of the unrotated query, written out directly
            keys = kc[0, :, :L] if nb == 1 else np.concatenate([kc[j] for j in range(nb)], axis=1)[:, :L]
            vals = vc[0, :, :L] if nb == 1 else np.concatenate([vc[j] for j in range(nb)], axis=1)[:, :L]
            for i in (4, 5):
                for h in range(Hq):
                    s = keys[h // 2] @ q[0, i, h] / np.sqrt(D)
                    e = np.exp(s - s.max())
                    np.testing.assert_allclose(out[0, i, h], e @ vals[h // 2] / e.sum(), rtol=1e-12, atol=1e-12)
