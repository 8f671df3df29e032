"""The C-ABI calls of the path are stream-ordered and allocation-free, so a
whole verification step can be captured as a CUDA graph and replayed: the
replay must give what direct calls give, also after the inputs in the
captured buffers change."""

import pytest
import torch

from speculative_decoding_tree_attn_gb300 import capi
from speculative_decoding_tree_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _step(st):
    c, i = capi, st["inp"]
    c.tv_tree_mask(st["parent"], i["seq_lens"], mask=st["mask"], depth=st["depth"], pos=st["pos"])
    q, kt = st["q"], st["kt"]
    q.copy_(i["q"])
    kt.copy_(i["k_tree"])
    c.tv_rope_apply(q, kt, st["pos"], st["table"])
    c.tv_tree_attn_verify(q, i["k_cache"], i["v_cache"], i["block_table"], i["seq_lens"], kt, i["v_tree"],
                          st["mask"], out=st["out"], workspace=st["ws"])
    g = st["greedy"]
    c.tv_tree_accept_greedy(g["tokens"], st["parent"], logits=g["logits"], out=st["acc"], n_out=st["n"],
                            path=st["path"])


@pytest.mark.parametrize("name", ["gqa_b8_l512_2048_n26", "b64_l1k_8k_n64_greedy"])
def test_graph_replay_matches_direct_calls(name):
    w = W.WORKLOADS[name]
    inp = W.attention_inputs(w, device="cuda")
    parent, _, _, _, n = capi.tv_tree_build(w.paths())
    par = torch.from_numpy(parent).cuda()
    B = w.B
    st = {"inp": inp, "parent": par,
          "mask": torch.empty(B, n, dtype=torch.int64, device="cuda"),
          "depth": torch.empty(B, n, dtype=torch.int32, device="cuda"),
          "pos": torch.empty(B, n, dtype=torch.int32, device="cuda"),
          "table": capi.tv_rope_table(int(inp["seq_lens"].max().item()) + n + 1, w.D, device="cuda"),
          "q": torch.empty_like(inp["q"]), "kt": torch.empty_like(inp["k_tree"]),
          "out": torch.empty_like(inp["q"]),
          "ws": capi.alloc_workspace(capi.tv_tree_attn_workspace_size(B, n, w.Hq, w.Hkv, w.D, inp["q"].dtype,
                                                                      w.block_size)),
          "greedy": W.greedy_inputs(w, parent, device="cuda"),
          "acc": torch.empty(B, n, dtype=torch.int32, device="cuda"),
          "n": torch.empty(B, dtype=torch.int32, device="cuda"),
          "path": torch.empty(B, n, dtype=torch.int32, device="cuda")}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(st)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(st)
    for trial in range(2):
        if trial:
            # new queries and logits in the captured buffers
            inp["q"].copy_(torch.randn_like(inp["q"], dtype=torch.float32).to(inp["q"].dtype))
            st["greedy"]["logits"].copy_(torch.randn_like(st["greedy"]["logits"]))
        graph.replay()
        torch.cuda.synchronize()
        got = {k: st[k].clone() for k in ("out", "acc", "n", "path")}
        _step(st)
        torch.cuda.synchronize()
        assert torch.equal(got["out"], st["out"])
        assert torch.equal(got["n"], st["n"])
        for b in range(B):
            k = int(st["n"][b].item())
            assert torch.equal(got["acc"][b, :k], st["acc"][b, :k])
            assert torch.equal(got["path"][b, :k], st["path"][b, :k])


def test_sampler_captured_on_first_call():
    """The stochastic walk's first call for a shape (its kernel choice queries
    the device's cluster capacity) may itself be inside a CUDA-graph capture;
    the replay equals a direct call."""
    import numpy as np
    rng = np.random.default_rng(160)
    B, N, V = 37, 6, 777  # a vocabulary no other test uses: nothing cached for it yet
    parent = torch.tensor([-1, 0, 0, 1, 1, 2], dtype=torch.int32, device="cuda")
    p = torch.from_numpy(rng.dirichlet(np.ones(V), size=(B, N)).astype(np.float32)).cuda()
    q = torch.from_numpy(rng.dirichlet(np.ones(V), size=(B, N)).astype(np.float32)).cuda()
    tok = torch.from_numpy(rng.integers(0, V, size=(B, N)).astype(np.int32)).cuda()
    ua = torch.from_numpy(rng.random((B, N), dtype=np.float32)).cuda()
    uf = torch.from_numpy(rng.random(B, dtype=np.float32)).cuda()
    out = torch.empty(B, N, dtype=torch.int32, device="cuda")
    n_out = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.empty(B, N, dtype=torch.int32, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        capi.tv_tree_accept_sample(p, q, tok, parent, ua, uf, out=out, n_out=n_out, path=path)
    graph.replay()
    torch.cuda.synchronize()
    ref = capi.tv_tree_accept_sample(p, q, tok, parent, ua, uf)
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(n_out, ref[1]) and torch.equal(path, ref[2])
