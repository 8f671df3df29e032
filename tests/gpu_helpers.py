"""Helpers for the GPU parity tests: run the library's pipeline on seeded
inputs and cut out per-request inputs for the oracle (which only ever sees
generator outputs, never anything the CUDA path computed)."""

import numpy as np
import torch

from oracle import attention as OA
from oracle import tree as OT
from speculative_decoding_tree_attn_gb300 import capi

BF16_TOL = 2e-2
F32_TOL = 1e-4


def to_np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def gpu_pipeline(inp, paths, flags=0, num_ctas=0, rope_base=10000.0, want_lse=False):
    """tree_build -> tree_mask -> rope_apply -> tree_attn_verify on the device."""
    dev = inp["q"].device
    parent, depth, rows, _, n = capi.tv_tree_build(paths)
    assert n == inp["q"].shape[1]
    parent_d = torch.from_numpy(parent).to(dev)
    seq_lens = inp["seq_lens"]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mask, depth_d, pos = capi.tv_tree_mask(parent_d, seq_lens, status=status)
    D = inp["q"].shape[-1]
    max_pos = int(seq_lens.max().item()) + n + 1
    table = capi.tv_rope_table(max_pos, D, rope_base, device=dev)
    q = inp["q"].clone()
    kt = inp["k_tree"].clone()
    capi.tv_rope_apply(q, kt, pos, table, status=status)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev) if want_lse else None
    out = capi.tv_tree_attn_verify(q, inp["k_cache"], inp["v_cache"], inp["block_table"], seq_lens, kt,
                                   inp["v_tree"], mask, lse=lse, flags=flags, num_ctas=num_ctas, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse


def oracle_rows(inp, paths, pairs, rope_base=10000.0):
    """Oracle outputs for the (b, i) pairs: returns {(b, i): (out [Hq, D], lse [Hq])}.

    Only the blocks of the requests involved are copied to the host."""
    parent, depth, rows, _ = OT.build_tree(paths)
    res = {}
    by_b = {}
    for b, i in pairs:
        by_b.setdefault(int(b), []).append(int(i))
    bs = inp["k_cache"].shape[2]
    for b, nodes in by_b.items():
        L = int(inp["seq_lens"][b].item())
        nb = (L + bs - 1) // bs
        blocks = inp["block_table"][b, :max(nb, 1)].long()
        kc = to_np(inp["k_cache"][blocks])
        vc = to_np(inp["v_cache"][blocks])
        table = np.arange(max(nb, 1), dtype=np.int64)[None]
        out, lse = OA.tree_attention(to_np(inp["q"][b:b + 1]), kc, vc, table, np.array([L]),
                                     to_np(inp["k_tree"][b:b + 1]), to_np(inp["v_tree"][b:b + 1]), parent,
                                     rope_base=rope_base, nodes=[(0, i) for i in nodes])
        for i in nodes:
            res[(b, i)] = (out[0, i], lse[0, i])
    return res


def max_err(gpu_out, ref, pairs):
    g = to_np(gpu_out)
    return max(float(np.abs(g[b, i] - ref[(b, i)][0]).max()) for b, i in pairs)
