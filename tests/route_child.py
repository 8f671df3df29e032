"""Child process of test_gpu_merge_routes.py (run with TREEVERIFY_LIB naming
the development build): for each tensor-core kernel shape and several CTA
counts (so that units are split between CTAs), the attention output with the
normal merge routes and with the epilogue warps of some TMEM quarters kept
off the direct merge, so that the warps of one M tile merge a split row by
different routes; for the tail-row shape also with the first pair of tail
warps slowed down, so that it still reads its last tile when the other pair
has released the slice's last one.  Prints one JSON line per (shape, CTA
count)."""

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
SHAPES = [("one_m_tile", 16, 2, 10, 16, [3000, 5000, 700, 2000]),
          ("two_m_tiles", 16, 2, 26, 16, [3000, 5000, 700, 2000]),
          ("tail_rows", 16, 2, 33, 64, [3000, 5000, 700, 2000])]
CTAS = [5, 7, 11, 13]
MASKS = [0b0001, 0b0010, 0b0101, 0b1110, 0b1111]
TAIL_DELAYS_NS = [3_000, 20_000]  # sleep of tail pair 0 before each of its tiles


def main():
    h = capi.lib()
    h.tv_test_set_publish_warps.restype = ctypes.c_int
    h.tv_test_set_publish_warps.argtypes = [ctypes.c_int]
    h.tv_test_set_tail_delay.restype = ctypes.c_int
    h.tv_test_set_tail_delay.argtypes = [ctypes.c_ulonglong]
    dev = torch.device("cuda:0")
    for label, Hq, Hkv, N, bs, lens in SHAPES:
        rng = np.random.default_rng(17 + N)
        paths = W.random_rank_paths(N, 8, rng)
        w = W.Workload("routes", len(lens), Hq, Hkv, 128, "bf16", ("fixed", 0), bs, (0.7, 0.15), N, 8, 21 + N)
        inp = W.attention_inputs(w, device=dev, seq_lens=lens)
        pairs = [(b, i) for b in range(len(lens)) for i in range(N)]
        ref = oracle_rows(inp, paths, pairs, rotate=False)
        for ctas in CTAS:
            assert h.tv_test_set_publish_warps(0) == 0
            base, base_lse = gpu_attention(inp, paths, flags=capi.TV_ATTN_TCGEN05, num_ctas=ctas)
            same = True
            for mask in MASKS:
                assert h.tv_test_set_publish_warps(mask) == 0
                out, lse = gpu_attention(inp, paths, flags=capi.TV_ATTN_TCGEN05, num_ctas=ctas)
                same = same and torch.equal(out, base) and torch.equal(lse, base_lse)
            assert h.tv_test_set_publish_warps(0) == 0
            err = max_err(base, ref, pairs)
            print(json.dumps({"shape": label, "ctas": ctas, "bit_identical": bool(same), "err": err,
                              "tol": BF16_TOL}), flush=True)
            if label == "tail_rows":
                same = True
                for d in TAIL_DELAYS_NS:
                    assert h.tv_test_set_tail_delay(d) == 0
                    out, lse = gpu_attention(inp, paths, flags=capi.TV_ATTN_TCGEN05, num_ctas=ctas)
                    same = same and torch.equal(out, base) and torch.equal(lse, base_lse)
                assert h.tv_test_set_tail_delay(0) == 0
                print(json.dumps({"shape": "tail_rows_slow_pair", "ctas": ctas, "bit_identical": bool(same),
                                  "err": max_err(out, ref, pairs), "tol": BF16_TOL}), flush=True)


if __name__ == "__main__":
    main()
