"""RoPE fused into the attention kernels' Q load (tv_tree_attn_verify_rope)
and into the mask kernel (tv_tree_prepare, for the tree keys alone or for Q
and the tree keys): each must give the same bits as the separate path
tv_tree_mask -> tv_rope_apply -> tv_tree_attn_verify (one rotation formula, float32, bf16 rounding), on both
attention kernels, for every GQA width the fused tensor-core path takes, with
ragged trees, empty prefixes and positions past the table; and the fused path
against the oracle at full size."""

import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import BF16_TOL, max_err, oracle_rows
from oracle import tree as OT
from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _case(Hq, Hkv, N, lens, seed, dtype="bf16", bs=16, ragged=None):
    w = W.Workload("fused", len(lens), Hq, Hkv, 128, dtype, ("fixed", 0), bs, (0.6, 0.25, 0.1), N, 8, seed)
    rng = np.random.default_rng(seed)
    par = np.stack([OT.build_tree(W.random_rank_paths(N, 6, rng))[0] for _ in range(len(lens))]).astype(np.int32)
    inp = W.attention_inputs(w, device="cuda", seq_lens=np.array(lens, dtype=np.int32))
    nn = None if ragged is None else torch.tensor(ragged, dtype=torch.int32, device="cuda")
    return w, torch.from_numpy(par).cuda(), inp, nn


def _separate(inp, par, table, nn, flags, lse=False):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask, depth, pos = capi.tv_tree_mask(par, inp["seq_lens"], status=status, n_nodes=nn)
    q, kt = inp["q"].clone(), inp["k_tree"].clone()
    capi.tv_rope_apply(q, kt, pos, table, status=status)
    l = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda") if lse else None
    out = capi.tv_tree_attn_verify(q, inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], kt,
                                   inp["v_tree"], mask, lse=l, flags=flags, status=status)
    return out, l, (mask, depth, pos), kt, status


def _fused(inp, par, table, nn, flags, lse=False):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kt = inp["k_tree"].clone()
    q0 = inp["q"].clone()
    mask, depth, pos = capi.tv_tree_prepare(par, inp["seq_lens"], kt, table, n_nodes=nn, status=status)
    l = torch.empty(q0.shape[:3], dtype=torch.float32, device="cuda") if lse else None
    out = capi.tv_tree_attn_verify_rope(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                        inp["seq_lens"], kt, inp["v_tree"], mask, table, lse=l, flags=flags,
                                        status=status)
    torch.cuda.synchronize()
    assert torch.equal(inp["q"], q0)  # the queries are not modified
    return out, l, (mask, depth, pos), kt, status


CASES = {
    "g4_n26_one_tile": (32, 8, 26, [0, 1, 63, 700, 1500]),
    "g4_n64_two_tiles": (32, 8, 64, [0, 5, 640, 2000]),
    "g8_n33_row_groups": (64, 8, 33, [17, 1000]),
    "g8_n33_tail_rows_bs64": (64, 8, 33, [17, 1000], 64),
    "g16_n20_row_groups": (32, 2, 20, [0, 300, 900]),
    "g2_n40_cuda_core": (8, 4, 40, [3, 500]),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("flags", [capi.TV_ATTN_AUTO, capi.TV_ATTN_SIMT, capi.TV_ATTN_TCGEN05,
                                   capi.TV_ATTN_TCGEN05 | capi.TV_ATTN_CTA_PAIRS])
def test_fused_equals_separate(name, flags):
    Hq, Hkv, N, lens, *bs = CASES[name]
    w, par, inp, _ = _case(Hq, Hkv, N, lens, 300 + N, bs=bs[0] if bs else 16)
    table = capi.tv_rope_table(max(lens) + N + 1, 128, device="cuda")
    if (flags & 3) == capi.TV_ATTN_TCGEN05 and Hq // Hkv not in (4, 8, 16):
        with pytest.raises(capi.TVError, match="UNSUPPORTED"):
            _fused(inp, par, table, None, flags)
        return
    # the automatic choice is the CUDA-core kernel when the fused tensor-core
    # path does not take the width: compare with the same kernel
    sep_flags = capi.TV_ATTN_SIMT if (flags == capi.TV_ATTN_AUTO and Hq // Hkv not in (4, 8, 16)) else flags
    a, la, ma, ka, sa = _separate(inp, par, table, None, sep_flags, lse=True)
    b, lb, mb, kb, sb = _fused(inp, par, table, None, flags, lse=True)
    assert int(sa.item()) == 0 and int(sb.item()) == 0
    for x, y in zip(ma, mb):
        assert torch.equal(x, y)
    assert torch.equal(ka, kb)
    assert torch.equal(a, b)
    assert torch.equal(la, lb)


@pytest.mark.parametrize("flags", [capi.TV_ATTN_TCGEN05, capi.TV_ATTN_SIMT])
def test_fused_ragged_and_short_table(flags):
    """Absent nodes stay unrotated; positions past the table stay unrotated
    and are flagged, on both paths alike."""
    w, par, inp, nn = _case(32, 8, 26, [0, 40, 600, 1], 77, ragged=[5, 26, 13, 1])
    table = capi.tv_rope_table(max([0, 40, 600, 1]) + 27, 128, device="cuda")
    a, _, ma, ka, sa = _separate(inp, par, table, nn, flags)
    b, _, mb, kb, sb = _fused(inp, par, table, nn, flags)
    assert int(sa.item()) == 0 and int(sb.item()) == 0
    assert torch.equal(ka, kb) and torch.equal(a, b)
    short = capi.tv_rope_table(601, 128, device="cuda")  # request 2 (L = 600): depths >= 1 run past it
    a, _, _, ka, sa = _separate(inp, par, short, nn, flags)
    b, _, _, kb, sb = _fused(inp, par, short, nn, flags)
    assert int(sa.item()) == int(sb.item()) == capi.TV_DEV_BAD_POSITION
    assert torch.equal(ka, kb) and torch.equal(a, b)


@pytest.mark.parametrize("name", ["b64_l1k_8k_n64_greedy", "b256_l2k_4k_n10_sample"])
def test_fused_full_size(name):
    """The full workloads: fused equals separate bit for bit, and sampled
    rows against the oracle."""
    w = W.WORKLOADS[name]
    inp = W.attention_inputs(w, device="cuda")
    parent, *_ = capi.tv_tree_build(w.paths())
    par = torch.from_numpy(parent).cuda()
    table = capi.tv_rope_table(int(inp["seq_lens"].max().item()) + w.n_nodes + 1, w.D, device="cuda")
    a, *_ = _separate(inp, par, table, None, 0)
    b, *_ = _fused(inp, par, table, None, 0)
    assert torch.equal(a, b)
    lens = inp["seq_lens"].cpu().numpy()
    bs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 7})
    pairs = [(bb, i) for bb in bs for i in (0, w.n_nodes // 2, w.n_nodes - 1)]
    ref = oracle_rows(inp, w.paths(), pairs)
    assert max_err(b, ref, pairs) <= BF16_TOL


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("ragged", [None, [5, 26, 13, 1]])
def test_prepare_with_q_equals_mask_then_rope(dtype, ragged):
    """tv_tree_prepare rotating Q and the tree keys is tv_tree_mask followed by
    tv_rope_apply, bit for bit, including absent nodes (left untouched)."""
    w, par, inp, nn = _case(32, 8, 26, [0, 3, 700, 1500], 417, dtype=dtype, ragged=ragged)
    table = capi.tv_rope_table(1600, 128, device="cuda")
    a = _separate(inp, par, table, nn, capi.TV_ATTN_AUTO)
    q, kt = inp["q"].clone(), inp["k_tree"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m, d, p = capi.tv_tree_prepare(par, inp["seq_lens"], kt, table, q=q, n_nodes=nn, status=status)
    sq = inp["q"].clone()
    capi.tv_rope_apply(sq, None, a[2][2], table)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(a[4].item()) == 0
    for x, y in zip((m, d, p), a[2]):
        assert torch.equal(x, y)
    assert torch.equal(kt, a[3]) and torch.equal(q, sq)
    # Q alone
    q2 = inp["q"].clone()
    capi.tv_tree_prepare(par, inp["seq_lens"], None, table, q=q2, n_nodes=nn)
    torch.cuda.synchronize()
    assert torch.equal(q2, sq)


def test_prepare_with_q_past_the_table_flags():
    """A position past the table leaves those Q rows as they are and sets
    TV_DEV_BAD_POSITION; rows inside the table are still rotated."""
    w, par, inp, _ = _case(32, 8, 26, [0, 590], 418)
    table = capi.tv_rope_table(593, 128, device="cuda")  # request 1's positions 590.. run past row 592
    q = inp["q"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, _, pos = capi.tv_tree_prepare(par, inp["seq_lens"], None, table, q=q, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & capi.TV_DEV_BAD_POSITION
    bad = (pos >= 593).cpu()
    assert bad.any() and not bad.all()
    assert torch.equal(q.cpu()[bad], inp["q"].cpu()[bad])
    assert not torch.equal(q.cpu()[~bad], inp["q"].cpu()[~bad])
