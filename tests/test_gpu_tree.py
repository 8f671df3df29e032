"""GPU parity: tv_tree_mask and tv_rope_table / tv_rope_apply against the oracle."""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import tree as OT
from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _random_parents(B, N, rng):
    par = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        paths = W.random_rank_paths(N, int(rng.integers(1, 9)), rng)
        par[b] = OT.build_tree(paths)[0]
    return par


@pytest.mark.parametrize("N", [1, 2, 10, 33, 63, 64])
def test_tree_mask_per_request_bit_exact(N):
    rng = np.random.default_rng(40 + N)
    B = 37
    par = _random_parents(B, N, rng)
    lens = rng.integers(0, 40000, size=B).astype(np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask, depth, pos = capi.tv_tree_mask(torch.from_numpy(par).cuda(), torch.from_numpy(lens).cuda(), status=status)
    rows, odepth, opos, ok = OT.tree_mask_batch(par, lens)
    assert ok.all() and status.item() == 0
    np.testing.assert_array_equal(mask.cpu().numpy().view(np.uint64), rows)
    np.testing.assert_array_equal(depth.cpu().numpy(), odepth)
    np.testing.assert_array_equal(pos.cpu().numpy(), opos)


def test_tree_mask_shared_tree_and_page_rows(mask_facts):
    parent, depth, rows, _ = OT.build_tree(W.PAGE_TREE_PATHS)
    lens = np.array([0, 5, 4096], dtype=np.int32)
    mask, d, pos = capi.tv_tree_mask(torch.from_numpy(parent.astype(np.int32)).cuda(), torch.from_numpy(lens).cuda())
    m = mask.cpu().numpy().view(np.uint64)
    for vals in mask_facts["mask_row"]:
        i, cols = int(vals[0]), [int(c) for c in vals[1:]]
        assert all(int(m[b, i]) == sum(1 << c for c in cols) for b in range(3))
    np.testing.assert_array_equal(pos.cpu().numpy(), lens[:, None] + depth[None])


def test_tree_mask_rejects_bad_topology():
    par = np.array([[-1, 0, 1], [-1, 2, 0], [0, 0, 0], [-1, 0, 0]], dtype=np.int32)
    lens = np.array([3, 3, 3, -1], dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask, depth, pos = capi.tv_tree_mask(torch.from_numpy(par).cuda(), torch.from_numpy(lens).cuda(), status=status)
    assert status.item() == capi.TV_DEV_BAD_TOPOLOGY | capi.TV_DEV_BAD_POSITION
    m = mask.cpu().numpy()
    assert m[0].tolist() == [1, 3, 7] and (m[1:] == 0).all()


def test_rope_table_matches_oracle():
    D, max_pos = 128, 33000
    cs = capi.tv_rope_table(max_pos, D).cpu().numpy().astype(np.float64)
    pos = np.array([0, 1, 2, 1000, 32767, 32999])
    ang = OA.rope_angles(pos, D)
    np.testing.assert_allclose(cs[pos, 0], np.cos(ang), rtol=0, atol=1.2e-7)
    np.testing.assert_allclose(cs[pos, 1], np.sin(ang), rtol=0, atol=1.2e-7)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_rope_apply_matches_oracle(dtype):
    """Each rotated element is the exact rotation rounded to the input
    precision: |gpu - oracle| <= u |oracle| (u = 2^-8 for bf16, 2^-24 for
    float32) plus the float32 rotation's own error, at most 2^-21 of the
    pair's magnitude |x1| + |x2| (two products of a float32 table entry,
    itself within 2^-24, and one rounded sum)."""
    g = torch.Generator(device="cuda").manual_seed(41)
    B, N, Hq, Hkv, D = 3, 7, 8, 2, 128
    q = torch.randn(B, N, Hq, D, device="cuda", generator=g).to(dtype)
    kt = torch.randn(B, N, Hkv, D, device="cuda", generator=g).to(dtype)
    pos = torch.randint(0, 40000, (B, N), device="cuda", generator=g, dtype=torch.int32)
    table = capi.tv_rope_table(40001, D)
    q2, k2 = q.clone(), kt.clone()
    capi.tv_rope_apply(q2, k2, pos, table)
    P = pos.cpu().numpy()
    ref_q = OA.rope(q.float().cpu().numpy(), P[..., None])
    ref_k = OA.rope(kt.float().cpu().numpy(), P[..., None])
    u = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -24
    for x, got, ref in ((q, q2, ref_q), (kt, k2, ref_k)):
        x = x.double().cpu().numpy()
        half = x.shape[-1] // 2
        pair = np.abs(x[..., :half]) + np.abs(x[..., half:])
        bound = u * np.abs(ref) + 2.0 ** -21 * np.concatenate([pair, pair], axis=-1)
        err = np.abs(got.double().cpu().numpy() - ref)
        assert (err <= bound).all(), float((err - bound).max())


def test_rope_apply_bad_position_flag():
    q = torch.ones(1, 2, 1, 64, device="cuda")
    pos = torch.tensor([[3, 99]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.tv_rope_apply(q, None, pos, capi.tv_rope_table(10, 64), status=status)
    assert status.item() == capi.TV_DEV_BAD_POSITION
    assert (q[0, 1] == 1).all()
