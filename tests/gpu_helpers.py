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

# Log-sum-exp (natural log) tolerance of the attention kernels when they are
# given the rotated rows in the input precision (no rounding of their own
# inputs): scores are exact bf16 (or float32) products summed in float32
# (relative error <= D * 2^-24 of sum |q_i k_i|, about 7e-4 absolute at the
# largest scores seen here, times the 1/sqrt(D) scale), the weights come from
# a hardware exp2 (relative error about 2^-22) and their sum is float32 over at
# most ~600 tile partial sums (relative error <= 600 * 2^-24 ~ 4e-5); the
# merge of split pieces adds a few float32 roundings.  Their sum stays below
# 1.5e-4, whatever the prefix length used here.
LSE_TOL = {torch.bfloat16: 1.5e-4, torch.float32: 1.5e-4}

# Unit roundoff of the input precision: the rows the RoPE kernel writes are
# the exact rotation rounded to nearest, |err| <= u |value| (plus a float32
# rotation error below 2^-21 of the pair's magnitude).
ROUND_U = {torch.bfloat16: 2.0 ** -8, torch.float32: 2.0 ** -24}


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


def prerotated(inp, paths, rope_base=10000.0):
    """The workload's Q and tree K rotated at L_b + depth by the oracle in
    float64, then rounded to the input precision: inputs for the attention
    kernel alone, compared with the oracle run without RoPE on these same
    rows (rotate=False)."""
    parent, depth, rows, _ = OT.build_tree(paths)
    lens = inp["seq_lens"].cpu().numpy().astype(np.int64)
    pos = lens[:, None] + depth[None, :]
    dt, dev = inp["q"].dtype, inp["q"].device
    q = OA.rope(to_np(inp["q"]), pos[:, :, None], rope_base)
    kt = OA.rope(to_np(inp["k_tree"]), pos[:, :, None], rope_base)
    return dict(inp, q=torch.from_numpy(q).to(dt).to(dev), k_tree=torch.from_numpy(kt).to(dt).to(dev))


def gpu_attention(inp, paths, flags=0, num_ctas=0):
    """tree_build -> tree_mask -> tree_attn_verify (rows already rotated)."""
    dev = inp["q"].device
    parent, depth, rows, _, n = capi.tv_tree_build(paths)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mask, _, _ = capi.tv_tree_mask(torch.from_numpy(parent).to(dev), inp["seq_lens"], status=status)
    lse = torch.empty(inp["q"].shape[:3], dtype=torch.float32, device=dev)
    out = capi.tv_tree_attn_verify(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                                   inp["k_tree"], inp["v_tree"], mask, lse=lse, flags=flags, num_ctas=num_ctas,
                                   status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse


def lse_err(gpu_lse, ref, pairs):
    """Largest |lse difference|; an empty key set must give -inf on both sides."""
    g = to_np(gpu_lse)
    worst = 0.0
    for b, i in pairs:
        r = ref[(b, i)][1]
        fin = np.isfinite(r)
        assert np.array_equal(np.isfinite(g[b, i]), fin), (b, i)
        if fin.any():
            worst = max(worst, float(np.abs(g[b, i][fin] - r[fin]).max()))
    return worst


def lse_pipeline_bound(inp, pairs):
    """Per (b, i): the log-sum-exp error bound [Hq] of the whole path, whose
    RoPE kernel rounds the rotated Q and tree K to the input precision.  A
    score moves by at most scale * (u |q| . |k| for a prefix key, 2u for a
    tree key, whose row is rounded too) <= scale * 2u ||q|| ||k|| (Cauchy-
    Schwarz; rotation keeps norms), and the log-sum-exp by at most the
    largest score move; the kernel's own LSE_TOL comes on top."""
    dt = inp["q"].dtype
    u = ROUND_U[dt] + 2.0 ** -21
    D = inp["q"].shape[-1]
    Hkv = inp["k_tree"].shape[2]
    G = inp["q"].shape[2] // Hkv
    bs = inp["k_cache"].shape[2]
    qn = torch.linalg.vector_norm(inp["q"].double(), dim=-1).cpu().numpy()        # [B, N, Hq]
    kt = torch.linalg.vector_norm(inp["k_tree"].double(), dim=-1).cpu().numpy()  # [B, N, Hkv]
    res = {}
    kmax = {}
    for b, i in pairs:
        if b not in kmax:
            L = int(inp["seq_lens"][b].item())
            km = kt[b].max(axis=0)
            if L > 0:
                nb = (L + bs - 1) // bs
                blk = inp["block_table"][b, :nb].long()
                kn = torch.linalg.vector_norm(inp["k_cache"][blk].double(), dim=-1)     # [nb, Hkv, bs]
                kn = kn.permute(1, 0, 2).reshape(Hkv, nb * bs)[:, :L].max(dim=1).values.cpu().numpy()
                km = np.maximum(km, kn)
            kmax[b] = km
        res[(b, i)] = (2 * u * qn[b, i] * np.repeat(kmax[b], G) / np.sqrt(D) + LSE_TOL[dt])
    return res


def check_lse_within(gpu_lse, ref, pairs, bound):
    g = to_np(gpu_lse)
    for b, i in pairs:
        r = ref[(b, i)][1]
        fin = np.isfinite(r)
        assert np.array_equal(np.isfinite(g[b, i]), fin), (b, i)
        d = np.abs(np.where(fin, g[b, i], 0.0) - np.where(fin, r, 0.0))
        assert (d <= bound[(b, i)]).all(), ((b, i), float(d.max()), float(bound[(b, i)].min()))


def oracle_rows(inp, paths, pairs, rope_base=10000.0, rotate=True):
    """Oracle outputs for the (b, i) pairs: returns {(b, i): (out [Hq, D], lse [Hq])}.

    Only the blocks of the requests involved are copied to the host; with
    rotate=False, Q and the tree keys are taken as already rotated."""
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
                                     rope_base=rope_base, nodes=[(0, i) for i in nodes], rotate=rotate)
        for i in nodes:
            res[(b, i)] = (out[0, i], lse[0, i])
    return res


def max_err(gpu_out, ref, pairs):
    g = to_np(gpu_out)
    return max(float(np.abs(g[b, i] - ref[(b, i)][0]).max()) for b, i in pairs)
