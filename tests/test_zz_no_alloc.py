"""The allocation-free tree-attention entry point (GPU).

tv_tree_attn_verify_static serves callers that cannot hand the library device
memory when they verify a tree (allocation forbidden after start-up, no
device allocator in their runtime, or cudaMalloc's possible device
synchronisation not allowed).  It keeps its split scratch in a fixed array
inside the library.  These checks call it through the C ABI twice in a row,
with the output and log-sum-exp buffers passed in, and compare each result
with the workspace entry point's within the tolerances of the parity tests
(bf16 on the tensor-core kernel, float32 on the CUDA-core kernel with its
plan and combine); they check that the calls allocate no device memory
(torch's allocator counters do not move and the CUDA free memory does not
shrink) and that a grid whose scratch exceeds the array is refused.  The file
is named so that pytest collects it last.
"""

import pytest
import torch

from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


def _inputs(w):
    inp = W.attention_inputs(w, device="cuda")
    parent, depth, rows, _, n = capi.tv_tree_build(w.paths())
    mask, _, pos = capi.tv_tree_mask(torch.from_numpy(parent).cuda(), inp["seq_lens"])
    table = capi.tv_rope_table(int(inp["seq_lens"].max().item()) + n + 1, w.D)
    capi.tv_rope_apply(inp["q"], inp["k_tree"], pos, table)
    return inp, mask


F32_SPLIT = W.Workload("f32_split", 4, 8, 2, 128, "f32", ("uniform", 300, 3000), 16, (0.7, 0.15), 26, 5, 77)


@pytest.mark.parametrize("name", ["gqa_b8_l512_2048_n26", "b64_l1k_8k_n64_greedy", "f32_split"])
def test_static_matches_workspace_entry_point_twice(name):
    w = F32_SPLIT if name == "f32_split" else W.WORKLOADS[name]
    inp, mask = _inputs(w)
    args = (inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], inp["k_tree"],
            inp["v_tree"], mask)
    # the float32 case runs the CUDA-core kernel on a grid that splits units,
    # so its plan, partials and combine all live in the static array
    extra = {"num_ctas": 23} if name == "f32_split" else {}
    ref_lse = torch.empty(inp["q"].shape[:3], dtype=torch.float32, device="cuda")
    ref = capi.tv_tree_attn_verify(*args, lse=ref_lse, **extra)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(inp["q"])
    lse = torch.empty_like(ref_lse)
    capi.tv_tree_attn_verify_static(*args, out=out, lse=lse, status=status, **extra)  # first call: set-up
    torch.cuda.synchronize()
    tol = TOL[inp["q"].dtype]
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        free_before = torch.cuda.mem_get_info()[0]
        capi.tv_tree_attn_verify_static(*args, out=out, lse=lse, status=status, **extra)
        torch.cuda.synchronize()
        assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == before
        assert torch.cuda.mem_get_info()[0] >= free_before
        assert status.item() == 0
        assert torch.isfinite(out.float()).all()
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= tol, err
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(lse))
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= tol


def test_static_rejects_scratch_beyond_its_maximum():
    inp, mask = _inputs(W.WORKLOADS["b64_l1k_8k_n64_greedy"])
    cap = capi.tv_tree_attn_static_workspace_bytes()
    assert cap == 32 << 20
    with pytest.raises(capi.TVError) as e:
        capi.tv_tree_attn_verify_static(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                        inp["seq_lens"], inp["k_tree"], inp["v_tree"], mask, num_ctas=4096)
    assert e.value.code == -5
    assert "static maximum" in str(e.value)
