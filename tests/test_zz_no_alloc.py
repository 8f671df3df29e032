"""The allocation-free tree-attention entry point (GPU).

tv_tree_attn_verify_static serves callers that cannot hand the library device
memory when they verify a tree (allocation forbidden after start-up, no
device allocator in their runtime, or cudaMalloc's possible device
synchronisation not allowed).  It keeps its split scratch in a fixed array
inside the library.  These checks call it through the C ABI twice in a row
and compare each result with the workspace entry point's, within the bf16
tolerance of the parity tests, and check that a grid whose scratch exceeds
the array is refused.  The file is named so that pytest collects it last.
"""

import numpy as np
import pytest
import torch

from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2


def _inputs(name):
    w = W.WORKLOADS[name]
    inp = W.attention_inputs(w, device="cuda")
    parent, depth, rows, _, n = capi.tv_tree_build(w.paths())
    mask, _, pos = capi.tv_tree_mask(torch.from_numpy(parent).cuda(), inp["seq_lens"])
    table = capi.tv_rope_table(int(inp["seq_lens"].max().item()) + n + 1, w.D)
    capi.tv_rope_apply(inp["q"], inp["k_tree"], pos, table)
    return inp, mask


@pytest.mark.parametrize("name", ["gqa_b8_l512_2048_n26", "b64_l1k_8k_n64_greedy"])
def test_static_matches_workspace_entry_point_twice(name):
    inp, mask = _inputs(name)
    args = (inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"], inp["k_tree"],
            inp["v_tree"], mask)
    ref = capi.tv_tree_attn_verify(*args)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        got = capi.tv_tree_attn_verify_static(*args, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        err = (got.float() - ref.float()).abs().max().item()
        assert err <= BF16_TOL, err
        assert torch.isfinite(got.float()).all()


def test_static_rejects_scratch_beyond_its_maximum():
    inp, mask = _inputs("b64_l1k_8k_n64_greedy")
    cap = capi.tv_tree_attn_static_workspace_bytes()
    assert cap == 32 << 20
    with pytest.raises(capi.TVError) as e:
        capi.tv_tree_attn_verify_static(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                        inp["seq_lens"], inp["k_tree"], inp["v_tree"], mask, num_ctas=4096)
    assert e.value.code == -5
    assert "static maximum" in str(e.value)
