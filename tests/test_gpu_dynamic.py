"""Dynamic trees: one best-first tree per request (parent [B, N]) through the
whole path -- tv_tree_mask with a per-request parent stride, depth-indexed
RoPE, tree attention with per-request ancestor rows and greedy acceptance
with per-request parents -- against the oracle run on each request's own
tree."""

import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import BF16_TOL, max_err, to_np
from oracle import accept as OA
from oracle import attention as OAt
from oracle import tree as OT
from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(w, pairs_per_b=None):
    paths = W.dynamic_rank_paths(w)
    gpu_par = np.stack([capi.tv_tree_build(p)[0] for p in paths]).astype(np.int32)
    ora_par = np.stack([OT.build_tree(p)[0] for p in paths])
    inp = W.attention_inputs(w, device="cuda")
    par_d = torch.from_numpy(gpu_par).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask, depth, pos = capi.tv_tree_mask(par_d, inp["seq_lens"], status=status)
    table = capi.tv_rope_table(int(pos.max().item()) + 1, w.D, device="cuda")
    q, kt = inp["q"].clone(), inp["k_tree"].clone()
    capi.tv_rope_apply(q, kt, pos, table, status=status)
    out = capi.tv_tree_attn_verify(q, inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], kt,
                                   inp["v_tree"], mask, status=status)
    g = W.greedy_inputs(w, ora_par, device="cuda")
    res = capi.tv_tree_accept_greedy(g["tokens"], par_d, logits=g["logits"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # oracle on each request's own tree
    ref_mask, ref_depth, ref_pos, _ = OT.tree_mask_batch(ora_par, inp["seq_lens"].cpu().numpy())
    np.testing.assert_array_equal(mask.cpu().numpy().view(np.uint64), ref_mask)
    np.testing.assert_array_equal(pos.cpu().numpy(), ref_pos)
    B, N = gpu_par.shape
    rng = np.random.default_rng(w.seed)
    if pairs_per_b is None:
        pairs = [(b, i) for b in range(B) for i in range(N)]
    else:
        bs = sorted(set(rng.integers(0, B, size=pairs_per_b[0]).tolist()))
        pairs = [(b, int(i)) for b in bs for i in sorted({0, N - 1, *rng.integers(0, N, size=pairs_per_b[1])})]
    ref = {}
    for b in sorted({b for b, _ in pairs}):
        nodes = [i for bb, i in pairs if bb == b]
        bsz = inp["k_cache"].shape[2]
        L = int(inp["seq_lens"][b])
        nb = max((L + bsz - 1) // bsz, 1)
        blocks = inp["block_table"][b, :nb].long()
        o, _ = OAt.tree_attention(to_np(inp["q"][b:b + 1]), to_np(inp["k_cache"][blocks]), to_np(inp["v_cache"][blocks]),
                                  np.arange(nb)[None], np.array([L]), to_np(inp["k_tree"][b:b + 1]),
                                  to_np(inp["v_tree"][b:b + 1]), ora_par[b], nodes=[(0, i) for i in nodes])
        for i in nodes:
            ref[(b, i)] = (o[0, i], None)
    assert max_err(out, ref, pairs) <= BF16_TOL
    am = OA.argmax_rows(g["logits"].cpu().numpy())
    r_out, r_n, r_path = OA.tree_accept_greedy(am, g["tokens"].cpu().numpy(), ora_par)
    np.testing.assert_array_equal(res[1].cpu().numpy(), r_n)
    for b in range(B):
        k = int(r_n[b])
        np.testing.assert_array_equal(res[0][b, :k].cpu().numpy(), r_out[b, :k])
        np.testing.assert_array_equal(res[2][b, :k].cpu().numpy(), r_path[b, :k])
    return paths


def test_dynamic_trees_small_all_rows():
    base = W.WORKLOADS["gqa_b8_l512_2048_n26"]
    w = dataclasses.replace(base, name="dyn_small", B=6, prefix=("uniform", 30, 300), dynamic=True, seed=31)
    paths = _run(w)
    assert len({tuple(p) for p in paths}) > 1  # the requests really have different trees


def test_dynamic_trees_b64_sampled_rows():
    _run(W.WORKLOADS["b64_l1k_8k_n64_dynamic"], pairs_per_b=(3, 4))
