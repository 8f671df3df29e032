"""Ragged trees in one bucket: every request holds its own tree of n_b <= N
nodes (n_nodes [B]); nodes >= n_b are absent.  Checked against the oracle on
the whole path -- tv_tree_mask (absent rows 0, position -1, their parent
entries never read), tv_rope_apply (absent rows untouched), both attention
kernels (an absent node attends to the prefix alone, an empty key set gives
a zero row with lse -inf) and greedy acceptance -- and one CUDA graph
captured for the bucket replays any ragged batch."""

import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import BF16_TOL, to_np
from oracle import accept as OA
from oracle import attention as OAt
from oracle import tree as OT
from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LENS = [0, 0, 5, 64, 300, 17, 0, 128, 1, 250]
COUNTS = [1, 26, 5, 13, 26, 2, 9, 20, 26, 7]


def _case():
    base = W.WORKLOADS["gqa_b8_l512_2048_n26"]
    w = dataclasses.replace(base, name="ragged_small", B=len(LENS), dynamic=True, seed=41)
    paths = W.dynamic_rank_paths(w)
    clean = np.stack([OT.build_tree(p)[0] for p in paths]).astype(np.int32)
    n_nodes = np.array(COUNTS, dtype=np.int32)
    par = clean.copy()
    for b, n in enumerate(n_nodes):
        par[b, n:] = 999  # absent nodes: never read
    inp = W.attention_inputs(w, device="cuda", seq_lens=np.array(LENS, dtype=np.int32))
    return w, clean, par, n_nodes, inp


@pytest.mark.parametrize("flags", [0, 1])
def test_ragged_trees_all_rows(flags):
    w, clean, par, n_nodes, inp = _case()
    B, N = par.shape
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nn_d = torch.from_numpy(n_nodes).cuda()
    mask, depth, pos = capi.tv_tree_mask(torch.from_numpy(par).cuda(), inp["seq_lens"], status=status, n_nodes=nn_d)
    ref_mask, ref_depth, ref_pos, ok = OT.tree_mask_batch(par, np.array(LENS), n_nodes)
    assert ok.all()
    np.testing.assert_array_equal(mask.cpu().numpy().view(np.uint64), ref_mask)
    np.testing.assert_array_equal(depth.cpu().numpy(), ref_depth)
    np.testing.assert_array_equal(pos.cpu().numpy(), ref_pos)
    table = capi.tv_rope_table(int(pos.max().item()) + 1, w.D, device="cuda")
    q, kt = inp["q"].clone(), inp["k_tree"].clone()
    capi.tv_rope_apply(q, kt, pos, table, status=status)
    for b, n in enumerate(n_nodes):  # absent rows untouched
        assert torch.equal(q[b, n:], inp["q"][b, n:]) and torch.equal(kt[b, n:], inp["k_tree"][b, n:])
    lse = torch.empty(B, N, w.Hq, dtype=torch.float32, device="cuda")
    out = capi.tv_tree_attn_verify(q, inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], kt,
                                   inp["v_tree"], mask, lse=lse, flags=flags, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    bs = inp["k_cache"].shape[2]
    got, got_lse = to_np(out), lse.cpu().numpy()
    for b in range(B):
        L = LENS[b]
        nb = max((L + bs - 1) // bs, 1)
        blocks = inp["block_table"][b, :nb].long()
        o, l = OAt.tree_attention(to_np(inp["q"][b:b + 1]), to_np(inp["k_cache"][blocks]),
                                  to_np(inp["v_cache"][blocks]), np.arange(nb)[None], np.array([L]),
                                  to_np(inp["k_tree"][b:b + 1]), to_np(inp["v_tree"][b:b + 1]), clean[b],
                                  n_nodes=n_nodes[b:b + 1])
        assert np.abs(got[b] - o[0]).max() <= BF16_TOL, b
        fin = np.isfinite(l[0])
        # lse carries the bf16 rounding of the rotated query and keys
        assert np.abs(got_lse[b][fin] - l[0][fin]).max() <= 5e-2
        assert np.array_equal(np.isneginf(got_lse[b]), np.isneginf(l[0]))
        if L == 0:
            assert (got[b, n_nodes[b]:] == 0).all()  # no key at all
    # greedy walk over the valid nodes only
    g = W.greedy_inputs(w, clean, device="cuda")
    res = capi.tv_tree_accept_greedy(g["tokens"], torch.from_numpy(par).cuda(), logits=g["logits"], n_nodes=nn_d)
    am = OA.argmax_rows(g["logits"].cpu().numpy())
    r_out, r_n, r_path = OA.tree_accept_greedy(am, g["tokens"].cpu().numpy(), clean, n_nodes)
    np.testing.assert_array_equal(res[1].cpu().numpy(), r_n)
    np.testing.assert_array_equal(res[0].cpu().numpy(), r_out)
    np.testing.assert_array_equal(res[2].cpu().numpy(), r_path)


def test_ragged_valid_rows_equal_truncated_trees():
    """A request's valid rows do not depend on the bucket: running it alone
    with N = n_b gives the same rows up to the rounding of a different split
    of its prefix over CTAs."""
    w, clean, par, n_nodes, inp = _case()
    B, N = par.shape
    nn_d = torch.from_numpy(n_nodes).cuda()
    mask, _, pos = capi.tv_tree_mask(torch.from_numpy(par).cuda(), inp["seq_lens"], n_nodes=nn_d)
    table = capi.tv_rope_table(int(pos.max().item()) + 1, w.D, device="cuda")
    q, kt = inp["q"].clone(), inp["k_tree"].clone()
    capi.tv_rope_apply(q, kt, pos, table)
    out = capi.tv_tree_attn_verify(q, inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], kt,
                                   inp["v_tree"], mask, flags=capi.TV_ATTN_SIMT)
    for b in [1, 3, 9]:
        n = int(n_nodes[b])
        sl = slice(b, b + 1)
        m1, _, p1 = capi.tv_tree_mask(torch.from_numpy(clean[b, :n].copy()).cuda(), inp["seq_lens"][sl])
        q1 = inp["q"][sl, :n].contiguous()
        k1 = inp["k_tree"][sl, :n].contiguous()
        capi.tv_rope_apply(q1, k1, p1, table)
        o1 = capi.tv_tree_attn_verify(q1, inp["k_cache"], inp["v_cache"], inp["block_table"][sl].contiguous(),
                                      inp["seq_lens"][sl].contiguous(), k1, inp["v_tree"][sl, :n].contiguous(), m1,
                                      flags=capi.TV_ATTN_SIMT)
        assert (out[b, :n].float() - o1[0].float()).abs().max().item() <= 1e-2, b


def _step(st):
    c, i = capi, st["inp"]
    c.tv_tree_mask(st["parent"], i["seq_lens"], mask=st["mask"], depth=st["depth"], pos=st["pos"],
                   n_nodes=st["n_nodes"])
    st["q"].copy_(i["q"])
    st["kt"].copy_(i["k_tree"])
    c.tv_rope_apply(st["q"], st["kt"], st["pos"], st["table"])
    c.tv_tree_attn_verify(st["q"], i["k_cache"], i["v_cache"], i["block_table"], i["seq_lens"], st["kt"],
                          i["v_tree"], st["mask"], out=st["out"], workspace=st["ws"])
    g = st["greedy"]
    c.tv_tree_accept_greedy(g["tokens"], st["parent"], logits=g["logits"], n_nodes=st["n_nodes"], out=st["acc"],
                            n_out=st["n"], path=st["path"])


def test_ragged_graph_one_bucket():
    """One graph captured for the bucket N; the trees and n_nodes in its
    buffers change between replays and each replay equals direct calls."""
    w, clean, par, n_nodes, inp = _case()
    B, N = par.shape
    dev = "cuda"
    st = {"inp": inp, "parent": torch.from_numpy(par).to(dev), "n_nodes": torch.from_numpy(n_nodes).to(dev),
          "mask": torch.empty(B, N, dtype=torch.int64, device=dev),
          "depth": torch.empty(B, N, dtype=torch.int32, device=dev),
          "pos": torch.empty(B, N, dtype=torch.int32, device=dev),
          "table": capi.tv_rope_table(max(LENS) + N + 1, w.D, device=dev),
          "q": torch.empty_like(inp["q"]), "kt": torch.empty_like(inp["k_tree"]), "out": torch.empty_like(inp["q"]),
          "ws": capi.alloc_workspace(capi.tv_tree_attn_workspace_size(B, N, w.Hq, w.Hkv, w.D, inp["q"].dtype,
                                                                      w.block_size)),
          "greedy": W.greedy_inputs(w, clean, device=dev),
          "acc": torch.empty(B, N, dtype=torch.int32, device=dev),
          "n": torch.empty(B, dtype=torch.int32, device=dev),
          "path": torch.empty(B, N, dtype=torch.int32, device=dev)}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(st)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(st)
    rng = np.random.default_rng(42)
    for trial in range(3):
        if trial:
            other = np.stack([OT.build_tree(W.random_rank_paths(N, 5, rng))[0] for _ in range(B)]).astype(np.int32)
            st["parent"].copy_(torch.from_numpy(other))
            st["n_nodes"].copy_(torch.from_numpy(rng.integers(1, N + 1, size=B).astype(np.int32)))
        graph.replay()
        torch.cuda.synchronize()
        replay = [st[k].clone() for k in ("mask", "out", "acc", "n", "path")]
        _step(st)
        torch.cuda.synchronize()
        direct = [st[k] for k in ("mask", "out", "acc", "n", "path")]
        for a, d in zip(replay, direct):
            assert torch.equal(a, d)
