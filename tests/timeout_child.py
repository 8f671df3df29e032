"""Child process of test_gpu_timeout.py (run with TREEVERIFY_LIB naming the
development build): for each tensor-core kernel shape, one call whose CTA 0
never receives the loads of one ring tile, then the same call without the
hook on the same stream.  Prints one JSON line per shape."""

import ctypes
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gpu_helpers import BF16_TOL, gpu_attention, max_err, oracle_rows  # noqa: E402
from speculative_decoding_tree_attn_gb300 import capi  # noqa: E402
from speculative_decoding_tree_attn_gb300 import workloads as W  # noqa: E402

# (label, Hq, Hkv, N, block size, prefix lengths): one M tile (G N <= 128),
# two M tiles (<= 256), two M tiles with tail rows (264)
SHAPES = [("one_m_tile", 16, 2, 10, 16, [700, 900]),
          ("two_m_tiles", 16, 2, 26, 16, [700, 900]),
          ("tail_rows", 16, 2, 33, 64, [700, 900])]
SHORT_NS = 200_000  # 0.2 ms wait limit while the hook is set


def main():
    h = capi.lib()
    h.tv_test_set_hooks.restype = ctypes.c_int
    h.tv_test_set_hooks.argtypes = [ctypes.c_ulonglong, ctypes.c_int]
    dev = torch.device("cuda:0")
    for label, Hq, Hkv, N, bs, lens in SHAPES:
        rng = np.random.default_rng(7 + N)
        paths = W.random_rank_paths(N, 8, rng)
        w = W.Workload("timeout", len(lens), Hq, Hkv, 128, "bf16", ("fixed", 0), bs, (0.7, 0.15), N, 8, 11 + N)
        inp = W.attention_inputs(w, device=dev, seq_lens=lens)
        parent, _, _, _, n = capi.tv_tree_build(paths)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        mask, _, _ = capi.tv_tree_mask(torch.from_numpy(parent).to(dev), inp["seq_lens"], status=st)
        # one CTA per unit at most two: CTA 0's slice spans several tiles
        assert h.tv_test_set_hooks(SHORT_NS, 2) == 0
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        out = torch.full_like(inp["q"], float("nan"))
        capi.tv_tree_attn_verify(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"], inp["seq_lens"],
                                 inp["k_tree"], inp["v_tree"], mask, out=out, flags=capi.TV_ATTN_TCGEN05,
                                 num_ctas=2, status=status)
        torch.cuda.synchronize()
        timed_out = int(status.item())
        assert h.tv_test_set_hooks(2_000_000_000, -1) == 0
        out2, _ = gpu_attention(inp, paths, flags=capi.TV_ATTN_TCGEN05, num_ctas=2)
        pairs = [(b, i) for b in range(len(lens)) for i in range(N)]
        err = max_err(out2, oracle_rows(inp, paths, pairs, rotate=False), pairs)
        print(json.dumps({"shape": label, "status": timed_out, "err_after": err, "tol": BF16_TOL}), flush=True)


if __name__ == "__main__":
    main()
