"""GPU parity of the tree-attention path (tree_build -> tree_mask -> rope_apply
-> tree_attn_verify) against the float64 per-path oracle.

Output tolerances are the ones fixed for this path: max-abs 1e-4 for float32
inputs and 2e-2 for bf16 inputs (float32 accumulation).  Every case is run
twice: the whole path, whose log-sum-exp is held to the bound the input-
precision rounding of the rotated rows allows (gpu_helpers.lse_pipeline_bound),
and the attention kernel alone on rows the oracle rotated, whose log-sum-exp
is held to the kernel's own float32 error (gpu_helpers.LSE_TOL).  Both
kernels are covered: the CUDA-core kernel for every shape, the tcgen05 kernel
for the shapes it accepts.  Small cases compare every output; the full-size
workloads compare every node of several requests (shortest and longest
prefix and split units included) in the launch configuration the bench
times."""

import numpy as np
import pytest
import torch

from gpu_helpers import (BF16_TOL, F32_TOL, LSE_TOL, check_lse_within, gpu_attention, gpu_pipeline, lse_err,
                         lse_pipeline_bound, max_err, oracle_rows, prerotated, to_np)
from oracle import tree as OT
from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu

KERNELS = [capi.TV_ATTN_SIMT, capi.TV_ATTN_TCGEN05]


def tc_available(Hq, Hkv, N, D=128, dtype=torch.bfloat16, bs=16):
    try:
        capi.tv_tree_attn_workspace_size(1, N, Hq, Hkv, D, dtype, bs, 0, capi.TV_ATTN_TCGEN05)
        return True
    except capi.TVError:
        return False


def _workload(B, Hq, Hkv, D, dtype, bs, N, seed):
    return W.Workload("case", B, Hq, Hkv, D, dtype, ("fixed", 0), bs, (0.7, 0.15), N, 8, seed)


def _check_all(inp, paths, tol, flags, num_ctas=0, pairs=None):
    """The whole path and the kernel alone (module docstring) on `pairs`
    (default: every node of every request)."""
    B, N = inp["q"].shape[:2]
    pairs = [(b, i) for b in range(B) for i in range(N)] if pairs is None else pairs
    out, lse = gpu_pipeline(inp, paths, flags=flags, num_ctas=num_ctas, want_lse=True)
    ref = oracle_rows(inp, paths, pairs)
    err = max_err(out, ref, pairs)
    assert err <= tol, err
    check_lse_within(lse, ref, pairs, lse_pipeline_bound(inp, pairs))
    rot = prerotated(inp, paths)
    out_k, lse_k = gpu_attention(rot, paths, flags=flags, num_ctas=num_ctas)
    ref_k = oracle_rows(rot, paths, pairs, rotate=False)
    err_k = max_err(out_k, ref_k, pairs)
    assert err_k <= tol, err_k
    lerr = lse_err(lse_k, ref_k, pairs)
    assert lerr <= LSE_TOL[inp["q"].dtype], lerr
    return out


def test_tiny_page_tree_f32():
    """B=1, one head, D=64, float32, L=32, the mask page's 10-node tree."""
    w = W.WORKLOADS["tiny_b1_f32"]
    inp = W.attention_inputs(w, device="cuda")
    for num_ctas in (0, 1, 2, 5):
        _check_all(inp, W.PAGE_TREE_PATHS, F32_TOL, capi.TV_ATTN_SIMT, num_ctas)


def test_tiny_random_trees_f32():
    rng = np.random.default_rng(50)
    for t in range(6):
        paths = W.random_rank_paths(10, 4, rng)
        w = _workload(1, 1, 1, 64, "f32", 16, 10, 60 + t)
        inp = W.attention_inputs(w, device="cuda", seq_lens=[32])
        _check_all(inp, paths, F32_TOL, capi.TV_ATTN_SIMT)


@pytest.mark.parametrize("L", [0, 1, 15, 16, 17, 63, 64, 65, 127, 128, 129])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefix_edges(L, dtype):
    """Prefix lengths at tile and block edges with a deep tree (mask offsets)."""
    rng = np.random.default_rng(51 + L)
    N = 37
    paths = W.random_rank_paths(N, 8, rng)
    w = _workload(2, 8, 2, 128, dtype, 16, N, 70 + L)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[L, max(L - 1, 0)])
    tol = F32_TOL if dtype == "f32" else BF16_TOL
    for flags in KERNELS:
        if flags == capi.TV_ATTN_TCGEN05 and (dtype == "f32" or not tc_available(8, 2, N)):
            continue
        for num_ctas in (0, 3):
            _check_all(inp, paths, tol, flags, num_ctas)


@pytest.mark.parametrize("N", [1, 2, 3, 8, 16, 31, 32, 33, 47, 63, 64])
def test_node_count_sweep(N):
    """Every node count from a single root to 64 nodes (hard-coded sizes were
    the failure mode of the DDTree post-mortem's mask corruption); 4 heads per
    KV head, so 33 nodes and more (129-256 rows) also run on CTA pairs."""
    rng = np.random.default_rng(80 + N)
    paths = W.random_rank_paths(N, 6, rng)
    for dtype, tol in (("f32", F32_TOL), ("bf16", BF16_TOL)):
        w = _workload(3, 4, 1, 128, dtype, 16, N, 90 + N)
        inp = W.attention_inputs(w, device="cuda", seq_lens=[0, 17, 200])
        for flags in KERNELS + ([capi.TV_ATTN_TCGEN05 | capi.TV_ATTN_CTA_PAIRS] if 4 * N > 128 else []):
            if (flags & 3) == capi.TV_ATTN_TCGEN05 and (dtype == "f32" or not tc_available(4, 1, N)):
                continue
            _check_all(inp, paths, tol, flags)


@pytest.mark.parametrize("G,N", [(8, 33), (16, 20), (4, 64), (2, 64)])
def test_row_groups_and_gqa_widths(G, N):
    """G * N above 256 (two row groups) and several GQA widths, both kernels."""
    rng = np.random.default_rng(120 + G + N)
    paths = W.random_rank_paths(N, 8, rng)
    w = _workload(2, 2 * G, 2, 128, "bf16", 64, N, 121 + G)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[130, 64 * 5 + 7])
    for flags in KERNELS:
        if flags == capi.TV_ATTN_TCGEN05 and not tc_available(2 * G, 2, N, bs=64):
            continue
        for num_ctas in (0, 5):
            _check_all(inp, paths, BF16_TOL, flags, num_ctas)


@pytest.mark.parametrize("flags", KERNELS)
def test_bad_block_table_entries_read_as_zeros(flags):
    """Block-table entries outside [0, num_blocks) (one past the end, one
    negative) are never dereferenced: those positions read as zero keys and
    values, and TV_DEV_BAD_BLOCK is set.  Checked against the oracle run on
    the same table with the bad entries pointing at an all-zero block."""
    paths = W.PAGE_TREE_PATHS
    w = _workload(3, 8, 2, 128, "bf16", 16, 10, 151)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[40, 100, 70])
    nb = inp["k_cache"].shape[0]
    bad = inp["block_table"].clone()
    bad[0, 1] = nb + 3
    bad[1, 0] = -1
    bad[2, 4] = nb
    inp_bad = dict(inp, block_table=bad)
    parent, *_ = capi.tv_tree_build(paths)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask, _, pos = capi.tv_tree_mask(torch.from_numpy(parent).cuda(), inp["seq_lens"], status=status)
    table = capi.tv_rope_table(200, 128, device="cuda")
    q, kt = inp["q"].clone(), inp["k_tree"].clone()
    capi.tv_rope_apply(q, kt, pos, table, status=status)
    out = capi.tv_tree_attn_verify(q, inp["k_cache"], inp["v_cache"], bad, inp["seq_lens"], kt, inp["v_tree"], mask,
                                   flags=flags, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == capi.TV_DEV_BAD_BLOCK
    # the oracle's view: one zero block appended, the bad entries pointing at it
    zero = torch.zeros_like(inp["k_cache"][:1])
    fixed = bad.clone()
    fixed[(fixed < 0) | (fixed >= nb)] = nb
    inp_ref = dict(inp, k_cache=torch.cat([inp["k_cache"], zero]), v_cache=torch.cat([inp["v_cache"], zero]),
                   block_table=fixed)
    pairs = [(b, i) for b in range(3) for i in range(10)]
    ref = oracle_rows(inp_ref, paths, pairs)
    assert max_err(out, ref, pairs) <= BF16_TOL


@pytest.mark.parametrize("bs", [1, 8, 32, 48, 128, 256])
def test_cache_block_sizes(bs):
    """Paged caches with other block sizes: the tcgen05 kernel takes multiples
    of 16 that divide 64 or that 64 divides (one TMA box per block, or a block
    spanning tiles); the others run the CUDA-core kernel (automatic choice)."""
    rng = np.random.default_rng(140 + bs)
    N = 26
    paths = W.random_rank_paths(N, 5, rng)
    w = _workload(3, 8, 2, 128, "bf16", bs, N, 141 + bs)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[bs * 3 + 5, 1, 700])
    tc = tc_available(8, 2, N, bs=bs)
    assert tc == (bs % 16 == 0 and (64 % bs == 0 or bs % 64 == 0))
    for flags in [capi.TV_ATTN_AUTO, capi.TV_ATTN_SIMT] + ([capi.TV_ATTN_TCGEN05] if tc else []):
        for num_ctas in (0, 7):
            _check_all(inp, paths, BF16_TOL, flags, num_ctas)


@pytest.mark.parametrize("D", [64, 256])
def test_other_head_dims_simt(D):
    rng = np.random.default_rng(95 + D)
    paths = W.random_rank_paths(12, 4, rng)
    w = _workload(2, 4, 2, D, "f32", 8, 12, 96)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[45, 3])
    _check_all(inp, paths, F32_TOL, capi.TV_ATTN_SIMT)


def test_mask_sensitive_tree_keys_dominate():
    """Tree keys scaled up so the tree part carries most of the softmax mass."""
    rng = np.random.default_rng(97)
    paths = W.random_rank_paths(26, 5, rng)
    w = _workload(2, 8, 2, 128, "f32", 16, 26, 98)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[64, 300], tree_scale=3.0)
    _check_all(inp, paths, F32_TOL, capi.TV_ATTN_SIMT)
    wb = _workload(2, 8, 2, 128, "bf16", 16, 26, 98)
    inp = W.attention_inputs(wb, device="cuda", seq_lens=[64, 300], tree_scale=2.0)
    for flags in KERNELS:
        if flags == capi.TV_ATTN_TCGEN05 and not tc_available(8, 2, 26):
            continue
        _check_all(inp, paths, BF16_TOL, flags)


@pytest.mark.parametrize("G,N,bs", [(4, 26, 16), (4, 64, 16), (8, 33, 16), (8, 33, 64)])
def test_split_unit_merge_routes(G, N, bs):
    """Units cut into many pieces (long prefixes, wide grids, grids wider than
    the plan so that some slices are empty).  The tensor-core kernel merges a
    split row either in the last piece straight from its accumulator, or from
    every piece's published partial (forced by TV_ATTN_PUBLISH_ALL); both
    routes must match the oracle (outputs, and the log-sum-exp at the
    kernel's own error on pre-rotated rows, where a wrong merge weight would
    show) and each other bit for bit.  The 264-row shape runs with two tail
    warps (block size 16) and with four (64)."""
    if not tc_available(2 * G, 2, N, bs=bs):
        pytest.skip("tensor-core kernel unavailable for this shape")
    rng = np.random.default_rng(140 + G + N)
    paths = W.random_rank_paths(N, 6, rng)
    kinds = [0, capi.TV_ATTN_CTA_PAIRS] if 128 < G * N <= 256 else [0]
    for lens, grids in (([3000, 70, 1500], (2, 7, 40, 152)), ([70, 0, 10], (300,))):
        w = _workload(3, 2 * G, 2, 128, "bf16", bs, N, 141 + N)
        inp = W.attention_inputs(w, device="cuda", seq_lens=lens)
        rot = prerotated(inp, paths)
        pairs = [(b, i) for b in range(3) for i in range(N)]
        ref = oracle_rows(inp, paths, pairs)
        ref_k = oracle_rows(rot, paths, pairs, rotate=False)
        bound = lse_pipeline_bound(inp, pairs)
        for num_ctas, kind in [(c, k) for c in grids for k in kinds]:
            res = []
            for extra in (kind, kind | capi.TV_ATTN_PUBLISH_ALL):
                flags = capi.TV_ATTN_TCGEN05 | extra
                out, lse = gpu_pipeline(inp, paths, flags=flags, num_ctas=num_ctas, want_lse=True)
                assert max_err(out, ref, pairs) <= BF16_TOL, (lens, num_ctas, extra)
                check_lse_within(lse, ref, pairs, bound)
                out_k, lse_k = gpu_attention(rot, paths, flags=flags, num_ctas=num_ctas)
                assert max_err(out_k, ref_k, pairs) <= BF16_TOL, (lens, num_ctas, extra)
                assert lse_err(lse_k, ref_k, pairs) <= LSE_TOL[torch.bfloat16], (lens, num_ctas, extra)
                res.append((out, lse, out_k, lse_k))
            for a, b in zip(res[0], res[1]):
                assert torch.equal(a, b), (lens, num_ctas)


@pytest.mark.parametrize("G,N,grids,kind,bs", [(8, 33, (2, 3, 7), 0, 16), (8, 33, (2, 3, 7), 0, 64),
                                                (4, 64, (2, 5), 0, 16), (4, 26, (3,), 0, 16),
                                                (4, 64, (2, 5), 16, 16)])
def test_repeated_calls_bit_identical(G, N, grids, kind, bs):
    """The same call forty times gives the same bits: every stage of the K/V
    ring is released only after all of its readers are done with it (a tail
    row read through the generic proxy without a proxy fence before the
    release once let the next TMA load overwrite it, here 39 runs in 40)."""
    if not tc_available(2 * G, 2, N, bs=bs):
        pytest.skip("tensor-core kernel unavailable for this shape")
    rng = np.random.default_rng(140 + G + N)
    paths = W.random_rank_paths(N, 6, rng)
    w = _workload(3, 2 * G, 2, 128, "bf16", bs, N, 141 + N)
    inp = prerotated(W.attention_inputs(w, device="cuda", seq_lens=[3000, 70, 1500]), paths)
    for num_ctas in grids:
        first = None
        for _ in range(40):
            out, lse = gpu_attention(inp, paths, flags=capi.TV_ATTN_TCGEN05 | kind, num_ctas=num_ctas)
            if first is None:
                first = (out, lse)
            else:
                assert torch.equal(out, first[0]) and torch.equal(lse, first[1]), num_ctas


def test_deterministic_and_kernel_agreement():
    w = W.WORKLOADS["gqa_b8_l512_2048_n26"]
    inp = W.attention_inputs(w, device="cuda")
    a, _ = gpu_pipeline(inp, w.paths())
    b, _ = gpu_pipeline(inp, w.paths())
    assert torch.equal(a, b)
    s, _ = gpu_pipeline(inp, w.paths(), flags=capi.TV_ATTN_SIMT)
    assert (a.float() - s.float()).abs().max().item() <= 2 * BF16_TOL


def test_workspace_errors():
    w = _workload(1, 2, 1, 64, "f32", 16, 4, 99)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[10])
    parent = torch.tensor([-1, 0, 0, 1], dtype=torch.int32, device="cuda")
    mask, _, _ = capi.tv_tree_mask(parent, inp["seq_lens"])
    with pytest.raises(capi.TVError) as e:
        capi.tv_tree_attn_verify(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                                 inp["k_tree"], inp["v_tree"], mask, workspace=capi.alloc_workspace(256))
    assert e.value.code == -5
    with pytest.raises(capi.TVError) as e:
        capi.tv_tree_attn_verify(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                                 inp["k_tree"], inp["v_tree"], mask, flags=capi.TV_ATTN_TCGEN05)
    assert e.value.code == -4


FULL = ["gqa_b8_l512_2048_n26", "b64_l1k_8k_n64_greedy", "long_b16_l32k_n33", "b256_l2k_4k_n10_sample"]


def _split_requests(lens, w, P):
    """Requests with a unit whose real tiles are cut by a slice boundary of
    the tensor-core plan (P slices of equal tile counts over the units laid
    end to end, each unit's virtual start tiles first), as the kernel derives
    it."""
    rows = (w.Hq // w.Hkv) * w.n_nodes
    cost = 3 if rows <= 128 else 8
    tiles = [(int(L) + 63) // 64 + 1 + cost for L in lens]
    T = sum(t * w.Hkv for t in tiles)
    P = max(1, min(P, (T + 11) // 12))
    bounds = {c * T // P for c in range(1, P)}
    out, start = set(), 0
    for b, t in enumerate(tiles):
        for _ in range(w.Hkv):
            if any(start + cost < x < start + t for x in bounds):
                out.add(b)
            start += t
    return sorted(out)


@pytest.mark.parametrize("name", FULL)
def test_full_size_all_nodes_of_sampled_requests(name):
    """Full workloads in the bench's launch configuration (auto kernel, one
    wave): every node and head of several requests -- the shortest and the
    longest prefix, requests with a unit split across CTAs, random others --
    on the whole path and on the kernel alone (module docstring)."""
    w = W.WORKLOADS[name]
    inp = W.attention_inputs(w, device="cuda")
    paths = w.paths()
    lens = inp["seq_lens"].cpu().numpy()
    rng = np.random.default_rng(100)
    n_req = 5 if w.prefix[0] == "fixed" and w.prefix[1] >= 16384 else 8
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = (w.Hq // w.Hkv) * w.n_nodes
    split = _split_requests(lens, w, sms * (2 if rows <= 128 else 1))
    bs = [int(lens.argmin()), int(lens.argmax())]
    bs += [b for b in split[:2] if b not in bs]
    for b in rng.permutation(w.B).tolist():
        if len(bs) >= n_req:
            break
        if b not in bs:
            bs.append(int(b))
    if w.B > 2:
        assert any(b in split for b in bs), "no request with a split unit sampled"
    pairs = [(b, i) for b in sorted(bs) for i in range(w.n_nodes)]
    _check_all(inp, paths, BF16_TOL, capi.TV_ATTN_AUTO, pairs=pairs)
    if 128 < rows <= 256:  # the same shape on CTA pairs (every node of the same requests)
        _check_all(inp, paths, BF16_TOL, capi.TV_ATTN_AUTO | capi.TV_ATTN_CTA_PAIRS, pairs=pairs)


@pytest.mark.parametrize("G,N,bs,kind", [(4, 26, 16, 0), (4, 64, 16, 0), (8, 33, 16, 0), (8, 33, 64, 0),
                                         (4, 64, 16, 16)])
def test_workspace_zeroed_flag(G, N, bs, kind):
    """Every completed call leaves the workspace's arrival counters at zero
    (the piece that merges a split row resets its counter), so calls with
    TV_ATTN_WORKSPACE_ZEROED on one workspace -- which skip clearing the
    counters -- give the same bits as calls that clear them, call after call,
    on both merge routes and grids that split every unit."""
    if not tc_available(2 * G, 2, N, bs=bs):
        pytest.skip("tensor-core kernel unavailable for this shape")
    rng = np.random.default_rng(160 + G + N + bs)
    paths = W.random_rank_paths(N, 6, rng)
    w = _workload(3, 2 * G, 2, 128, "bf16", bs, N, 161 + N)
    inp = prerotated(W.attention_inputs(w, device="cuda", seq_lens=[3000, 70, 1500]), paths)
    parent, *_ = capi.tv_tree_build(paths)
    mask, _, _ = capi.tv_tree_mask(torch.from_numpy(parent).cuda(), inp["seq_lens"])
    args = (inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], inp["k_tree"],
            inp["v_tree"], mask)
    for num_ctas in (2, 7, 40):
        for extra in (kind, kind | capi.TV_ATTN_PUBLISH_ALL):
            flags = capi.TV_ATTN_TCGEN05 | extra
            ws = capi.alloc_workspace(capi.tv_tree_attn_workspace_size(3, N, 2 * G, 2, 128, torch.bfloat16, bs,
                                                                       num_ctas, flags))
            ref_lse = torch.empty(inp["q"].shape[:3], dtype=torch.float32, device="cuda")
            ref = capi.tv_tree_attn_verify(*args, lse=ref_lse, workspace=ws, num_ctas=num_ctas, flags=flags)
            for _ in range(3):
                out = torch.full_like(inp["q"], float("nan"))
                lse = torch.full_like(ref_lse, float("nan"))
                status = torch.zeros(1, dtype=torch.int32, device="cuda")
                capi.tv_tree_attn_verify(*args, out=out, lse=lse, workspace=ws, num_ctas=num_ctas,
                                         flags=flags | capi.TV_ATTN_WORKSPACE_ZEROED, status=status)
                torch.cuda.synchronize()
                assert int(status.item()) == 0
                assert torch.equal(out, ref) and torch.equal(lse, ref_lse), (num_ctas, extra)


def test_misaligned_output_is_refused():
    """The tensor-core path writes output rows in 32-byte pieces: an output
    pointer off a 32-byte boundary is refused with TV_ERR_INVALID_ARG (and a
    32-byte aligned one that is not 256-byte aligned works)."""
    if not tc_available(8, 2, 10):
        pytest.skip("tensor-core kernel unavailable")
    w = _workload(2, 8, 2, 128, "bf16", 16, 10, 171)
    inp = W.attention_inputs(w, device="cuda", seq_lens=[100, 300])
    parent, *_ = capi.tv_tree_build(W.PAGE_TREE_PATHS)
    mask, _, _ = capi.tv_tree_mask(torch.from_numpy(parent).cuda(), inp["seq_lens"])
    args = (inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], inp["k_tree"],
            inp["v_tree"], mask)
    ref = capi.tv_tree_attn_verify(*args, flags=capi.TV_ATTN_TCGEN05)
    big = torch.empty(ref.numel() + 64, dtype=ref.dtype, device="cuda")
    with pytest.raises(capi.TVError) as e:
        capi.tv_tree_attn_verify(*args, out=big[8:8 + ref.numel()].view(ref.shape), flags=capi.TV_ATTN_TCGEN05)
    assert e.value.code == -1
    out32 = big[16:16 + ref.numel()].view(ref.shape)  # 32 bytes past a 256-byte boundary
    capi.tv_tree_attn_verify(*args, out=out32, flags=capi.TV_ATTN_TCGEN05)
    torch.cuda.synchronize()
    assert torch.equal(out32, ref)
