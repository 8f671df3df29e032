"""GPU parity of tv_kv_commit (the accepted path's tree K/V copied into the
paged cache) against the oracle, bit for bit, plus the property that the
commit serves the next step: attention of the last accepted node as a
one-node tree over the committed cache equals its output in the tree pass."""

import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import BF16_TOL, F32_TOL, gpu_pipeline, to_np
from oracle import accept as OA
from oracle import kvcache as OK
from oracle import tree as OT
from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _oracle_commit(inp, path, n_out):
    kc, vc, lens = OK.commit_path(to_np(inp["k_cache"]), to_np(inp["v_cache"]), inp["block_table"].cpu().numpy(),
                                  inp["seq_lens"].cpu().numpy(), to_np(inp["k_tree"]), to_np(inp["v_tree"]),
                                  path, n_out)
    return kc, vc, lens


def _gpu_commit(inp, path, n_out, status=None):
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    lens = capi.tv_kv_commit(kc, vc, inp["block_table"], inp["seq_lens"], inp["k_tree"], inp["v_tree"],
                             torch.from_numpy(path.astype(np.int32)).cuda(),
                             torch.from_numpy(n_out.astype(np.int32)).cuda(), status=status)
    torch.cuda.synchronize()
    return kc, vc, lens


@pytest.mark.parametrize("name", ["gqa_b8_l512_2048_n26", "b64_l1k_8k_n64_greedy", "long_b16_l32k_n33"])
def test_commit_greedy_paths_bit_exact(name):
    w = W.WORKLOADS[name]
    parent, depth, *_ = OT.build_tree(w.paths())
    inp = W.attention_inputs(w, device="cuda", reserve=int(depth.max()) + 1)
    g = W.greedy_inputs(w if w.vocab else dataclasses.replace(w, vocab=1000), parent, device="cuda")
    out, n_out, path = OA.tree_accept_greedy(OA.argmax_rows(g["logits"].cpu().numpy()), g["tokens"].cpu().numpy(),
                                             parent)
    kc, vc, lens = _gpu_commit(inp, path, n_out)
    okc, ovc, olens = _oracle_commit(inp, path, n_out)
    np.testing.assert_array_equal(lens.cpu().numpy(), olens)
    assert torch.equal(kc.float().cpu(), torch.from_numpy(okc).float())
    assert torch.equal(vc.float().cpu(), torch.from_numpy(ovc).float())


@pytest.mark.parametrize("dtype,bs,Hkv,D", [("f32", 16, 1, 64), ("bf16", 64, 8, 128), ("bf16", 16, 2, 256)])
def test_commit_block_edges_and_shapes(dtype, bs, Hkv, D):
    rng = np.random.default_rng(400 + bs + D)
    N = 12
    paths = W.random_rank_paths(N, 5, rng)
    parent, depth, *_ = OT.build_tree(paths)
    w = W.Workload("case", 4, 2 * Hkv, Hkv, D, dtype, ("fixed", 0), bs, (0.7, 0.15), N, 5, 410 + bs)
    lens = [bs - 1, bs, 0, 3 * bs - 2]
    inp = W.attention_inputs(w, device="cuda", seq_lens=lens, reserve=int(depth.max()) + 1)
    leaves = [i for i in range(N) if i not in set(parent[1:].tolist())]
    B = len(lens)
    cols = int(depth.max()) + 2
    path = np.full((B, cols), -1, dtype=np.int64)
    n_out = np.zeros(B, dtype=np.int64)
    for b in range(B):
        chain = OT.path_to_root(parent, leaves[b % len(leaves)])
        path[b, :len(chain)] = chain
        n_out[b] = len(chain) if b != 2 else 1
    kc, vc, new_lens = _gpu_commit(inp, path, n_out)
    okc, ovc, olens = _oracle_commit(inp, path, n_out)
    np.testing.assert_array_equal(new_lens.cpu().numpy(), olens)
    assert torch.equal(kc.float().cpu(), torch.from_numpy(okc).float())
    assert torch.equal(vc.float().cpu(), torch.from_numpy(ovc).float())


def test_commit_stops_at_the_first_step_it_cannot_commit():
    """A bad node or a position without a block ends the commit there: the
    steps before it are copied, nothing after, and the new prefix length
    counts only the copied steps (bit for bit against the oracle's
    stop_at_bad reading)."""
    w = W.Workload("case", 3, 2, 1, 64, "f32", ("fixed", 0), 16, (0.7, 0.15), 6, 3, 420)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[14, 3, 5], reserve=2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # request 0: 5 rows from 14 reach position 16, past its 1-block table
    # width (step 2); request 1: node 9 >= N at step 1, then a valid node;
    # request 2: a negative node at step 2
    path = np.array([[0, 1, 2, 3, 4], [0, 9, 1, -1, -1], [0, 1, -3, 2, -1]])
    n_out = np.array([5, 3, 4])
    kc, vc, lens = _gpu_commit(inp, path, n_out, status=status)
    assert int(status.item()) == capi.TV_DEV_OUT_OVERFLOW | capi.TV_DEV_BAD_TOPOLOGY
    okc, ovc, olens = OK.commit_path(to_np(inp["k_cache"]), to_np(inp["v_cache"]), inp["block_table"].cpu().numpy(),
                                     inp["seq_lens"].cpu().numpy(), to_np(inp["k_tree"]), to_np(inp["v_tree"]),
                                     path, n_out, stop_at_bad=True)
    np.testing.assert_array_equal(olens, [16, 4, 7])
    np.testing.assert_array_equal(lens.cpu().numpy(), olens)
    assert torch.equal(kc.float().cpu(), torch.from_numpy(okc).float())
    assert torch.equal(vc.float().cpu(), torch.from_numpy(ovc).float())


@pytest.mark.parametrize("name", ["gqa_b8_l512_2048_n26", "tiny_b1_f32"])
def test_committed_cache_serves_the_next_step(name):
    """The last accepted node's tree-pass output equals a one-node tree (that
    node as the root) attending over the cache with the rest of the path
    committed -- both computed on the GPU."""
    w = W.WORKLOADS[name]
    paths = w.paths()
    parent, depth, *_ = OT.build_tree(paths)
    inp = W.attention_inputs(w, device="cuda", reserve=int(depth.max()) + 1)
    g = W.greedy_inputs(w, parent, device="cuda")
    out_tree, _ = gpu_pipeline(inp, paths)          # rotates copies of q / k_tree inside
    _, n_out, path = capi.tv_tree_accept_greedy(g["tokens"], torch.from_numpy(parent.astype(np.int32)).cuda(),
                                                logits=g["logits"])
    # rotate the tree keys as the pipeline did, then commit all path nodes but the last
    pos = inp["seq_lens"][:, None] + torch.from_numpy(depth.astype(np.int32)).cuda()[None, :]
    table = capi.tv_rope_table(int(pos.max().item()) + 2, w.D, device="cuda")
    q_rot, kt_rot = inp["q"].clone(), inp["k_tree"].clone()
    capi.tv_rope_apply(q_rot, kt_rot, pos.to(torch.int32).contiguous(), table)
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    head = (n_out - 1).clamp(min=0).to(torch.int32)
    lens2 = capi.tv_kv_commit(kc, vc, inp["block_table"], inp["seq_lens"], kt_rot, inp["v_tree"], path, head)
    B = w.B
    last = path[torch.arange(B), (n_out - 1).long()].long()
    rows = torch.arange(B, device="cuda")
    q1 = q_rot[rows, last][:, None].contiguous()
    kt1 = kt_rot[rows, last][:, None].contiguous()
    vt1 = inp["v_tree"][rows, last][:, None].contiguous()
    mask1 = torch.ones(B, 1, dtype=torch.int64, device="cuda")
    out1 = capi.tv_tree_attn_verify(q1, kc, vc, inp["block_table"], lens2, kt1, vt1, mask1)
    torch.cuda.synchronize()
    ref = out_tree[rows, last].float()
    tol = F32_TOL if w.dtype == "f32" else BF16_TOL
    assert (out1[:, 0].float() - ref).abs().max().item() <= tol
