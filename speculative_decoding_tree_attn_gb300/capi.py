"""Thin Python binding of libtreeverify (ctypes).

Each function carries the name of the C entry point it calls and only
marshals arguments: it checks tensor placement/dtype/contiguity, passes raw
pointers, sizes and the current CUDA stream, and raises :class:`TVError` on a
non-zero status.  Every step of the computation runs in the library's
kernels; there is no Python or CPU fallback, and a missing library raises.
"""

from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtreeverify.so")

TV_F32, TV_BF16 = 0, 1
TV_ATTN_AUTO, TV_ATTN_SIMT, TV_ATTN_TCGEN05 = 0, 1, 2
TV_ATTN_PUBLISH_ALL = 4
TV_ATTN_ROPE_Q = 8
TV_ATTN_CTA_PAIRS = 16
TV_ATTN_WORKSPACE_ZEROED = 32
TV_SAMPLE_AUTO, TV_SAMPLE_CLUSTER, TV_SAMPLE_SINGLE_CTA, TV_SAMPLE_STREAM, TV_SAMPLE_GRID = 0, 1, 2, 3, 4
TV_DEV_BAD_TOPOLOGY, TV_DEV_BAD_TOKEN, TV_DEV_OUT_OVERFLOW, TV_DEV_BAD_POSITION, TV_DEV_TIMEOUT = 1, 2, 4, 8, 16
TV_DEV_BAD_BLOCK = 32
STATUS_NAMES = {0: "TV_OK", -1: "TV_ERR_INVALID_ARG", -2: "TV_ERR_MISSING_PARENT", -3: "TV_ERR_TOO_MANY_NODES",
                -4: "TV_ERR_UNSUPPORTED", -5: "TV_ERR_WORKSPACE", -6: "TV_ERR_CUDA"}

# exported symbol -> (restype, argtypes)
_I32, _I64, _P, _SZ, _F, _D = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float, ctypes.c_double
SIGNATURES = {
    "tv_last_error": (ctypes.c_char_p, []),
    "tv_version": (ctypes.c_int, []),
    "tv_tree_build": (ctypes.c_int, [_P, _P, _I32, _I32, _P, _P, _P, _P, _P]),
    "tv_tree_mask": (ctypes.c_int, [_P, _I64, _P, _P, _I32, _I32, _P, _P, _P, _P, _P]),
    "tv_rope_table": (ctypes.c_int, [_P, _I32, _I32, _D, _P]),
    "tv_rope_apply": (ctypes.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P]),
    "tv_tree_attn_workspace_size": (ctypes.c_int, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _P]),
    "tv_tree_attn_verify": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _P, _I32, _P, _P, _P, _P, _I64, _I32, _I32,
                                           _I32, _I32, _I32, _I32, _F, _P, _P, _P, _SZ, _I32, _I32, _P, _P]),
    "tv_tree_attn_verify_static": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _P, _I32, _P, _P, _P, _P, _I64, _I32,
                                                  _I32, _I32, _I32, _I32, _I32, _F, _P, _P, _I32, _I32, _P, _P]),
    "tv_tree_attn_static_workspace_bytes": (ctypes.c_size_t, []),
    "tv_tree_attn_verify_rope": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _P, _I32, _P, _P, _P, _P, _I64, _P, _I32,
                                                _I32, _I32, _I32, _I32, _I32, _I32, _F, _P, _P, _P, _SZ, _I32, _I32,
                                                _P, _P]),
    "tv_tree_prepare": (ctypes.c_int, [_P, _I64, _P, _P, _I32, _I32, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                       _P, _I32, _P, _P]),
    "tv_tree_accept_greedy": (ctypes.c_int, [_P, _P, _P, _P, _I64, _P, _I32, _I32, _I32, _P, _P, _P, _I32, _P, _P]),
    "tv_tree_accept_sample": (ctypes.c_int, [_P, _P, _P, _P, _I64, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _I32,
                                             _I32, _P, _SZ, _P, _P]),
    "tv_accept_sample_workspace_size": (ctypes.c_size_t, [_I32, _I32, _I32]),
    "tv_accept_sample_uses_grid": (ctypes.c_int, [_I32, _I32, _I32, _I32, _SZ, _P]),
    "tv_chain_accept_sample": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _I32, _I32, _P, _SZ,
                                              _P, _P]),
    "tv_kv_commit": (ctypes.c_int, [_P, _P, _I64, _I32, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                    _I32, _I32, _P, _P]),
}


class TVError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def lib():
    """The loaded library (raises if it was not built).  The environment
    variable TREEVERIFY_LIB names another build to load instead (the
    development build with test hooks)."""
    global _lib
    if _lib is None:
        path = os.environ.get("TREEVERIFY_LIB") or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with speculative_decoding_tree_attn_gb300.build")
        h = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(h, name)
            f.restype, f.argtypes = res, args
        _lib = h
    return _lib


def _check(fn, code):
    if code != 0:
        raise TVError(fn, code, lib().tv_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dev(t, name, dtypes):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _code(dtype):
    if dtype == torch.float32:
        return TV_F32
    if dtype == torch.bfloat16:
        return TV_BF16
    raise ValueError(f"unsupported dtype {dtype}")


def tv_version():
    return lib().tv_version()


def tv_tree_build(paths, max_nodes=64):
    """Rank paths -> (parent, depth, mask (uint64), path_to_node, n_nodes) on the host."""
    ranks = np.array([r for p in paths for r in p], dtype=np.int32)
    offsets = np.zeros(len(paths) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum([len(p) for p in paths])
    parent = np.zeros(max_nodes, dtype=np.int32)
    depth = np.zeros(max_nodes, dtype=np.int32)
    mask = np.zeros(max_nodes, dtype=np.uint64)
    p2n = np.zeros(max(len(paths), 1), dtype=np.int32)
    n = np.zeros(1, dtype=np.int32)
    _check("tv_tree_build", lib().tv_tree_build(_ptr(ranks) if ranks.size else None, _ptr(offsets), len(paths),
                                                max_nodes, _ptr(parent), _ptr(depth), _ptr(mask), _ptr(p2n), _ptr(n)))
    k = int(n[0])
    return parent[:k].copy(), depth[:k].copy(), mask[:k].copy(), p2n[:len(paths)].copy(), k


def tv_tree_mask(parent, seq_lens, status=None, mask=None, depth=None, pos=None, stream=None, n_nodes=None):
    """parent int32 [N] (shared) or [B, N]; seq_lens int32 [B]; n_nodes int32 [B]
    (optional, ragged trees: nodes >= n_nodes[b] absent) -> (mask int64 [B, N]
    holding the uint64 rows, depth int32 [B, N], pos int32 [B, N])."""
    _dev(parent, "parent", (torch.int32,))
    _dev(seq_lens, "seq_lens", (torch.int32,))
    if n_nodes is not None:
        _dev(n_nodes, "n_nodes", (torch.int32,))
    B = seq_lens.numel()
    N = parent.shape[-1]
    bstride = 0 if parent.dim() == 1 else parent.stride(0)
    dev = seq_lens.device
    mask = torch.empty(B, N, dtype=torch.int64, device=dev) if mask is None else mask
    depth = torch.empty(B, N, dtype=torch.int32, device=dev) if depth is None else depth
    pos = torch.empty(B, N, dtype=torch.int32, device=dev) if pos is None else pos
    _check("tv_tree_mask", lib().tv_tree_mask(_ptr(parent), bstride, _ptr(seq_lens), _ptr(n_nodes), B, N, _ptr(mask),
                                              _ptr(depth), _ptr(pos), _ptr(status), _stream(stream)))
    return mask, depth, pos


def tv_rope_table(max_pos, head_dim, base=10000.0, device="cuda", stream=None):
    cs = torch.empty(max_pos, 2, head_dim // 2, dtype=torch.float32, device=device)
    _check("tv_rope_table", lib().tv_rope_table(_ptr(cs), max_pos, head_dim, float(base), _stream(stream)))
    return cs


def tv_rope_apply(q, k_tree, pos, cos_sin, status=None, stream=None):
    """Rotates q [B, N, Hq, D] and k_tree [B, N, Hkv, D] in place at pos [B, N]."""
    _dev(q, "q", (torch.float32, torch.bfloat16))
    if k_tree is not None:
        _dev(k_tree, "k_tree", (q.dtype,))
    _dev(pos, "pos", (torch.int32,))
    _dev(cos_sin, "cos_sin", (torch.float32,))
    B, N, Hq, D = q.shape
    Hkv = k_tree.shape[2] if k_tree is not None else 1
    _check("tv_rope_apply", lib().tv_rope_apply(_ptr(q), _ptr(k_tree), _ptr(pos), _ptr(cos_sin), cos_sin.shape[0],
                                                B, N, Hq, Hkv, D, _code(q.dtype), _ptr(status), _stream(stream)))


def tv_tree_attn_workspace_size(B, N, Hq, Hkv, head_dim, dtype, block_size, num_ctas=0, flags=0):
    out = ctypes.c_size_t(0)
    _check("tv_tree_attn_workspace_size",
           lib().tv_tree_attn_workspace_size(B, N, Hq, Hkv, head_dim, _code(dtype), block_size, num_ctas, flags,
                                             ctypes.addressof(out)))
    return out.value


def alloc_workspace(nbytes, device="cuda"):
    """A 256-byte aligned workspace tensor of at least nbytes, zeroed (so it
    can be passed with TV_ATTN_WORKSPACE_ZEROED until a call times out)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def tv_tree_attn_verify(q, k_cache, v_cache, block_table, seq_lens, k_tree, v_tree, mask, *, scale=None,
                        out=None, lse=None, workspace=None, num_ctas=0, flags=0, status=None, stream=None):
    """Tree attention; returns out [B, N, Hq, D].  mask is int64 [B, N] (uint64 rows)
    or [N] (shared)."""
    dts = (torch.float32, torch.bfloat16)
    _dev(q, "q", dts)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_tree", k_tree), ("v_tree", v_tree)):
        _dev(t, name, (q.dtype,))
    _dev(block_table, "block_table", (torch.int32,))
    _dev(seq_lens, "seq_lens", (torch.int32,))
    _dev(mask, "mask", (torch.int64,))
    B, N, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    num_blocks, _, block_size, _ = k_cache.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(tv_tree_attn_workspace_size(B, N, Hq, Hkv, D, q.dtype, block_size, num_ctas,
                                                                flags), q.device)
    mstride = 0 if mask.dim() == 1 else mask.stride(0)
    _check("tv_tree_attn_verify",
           lib().tv_tree_attn_verify(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, block_size, _ptr(block_table),
                                     block_table.shape[1], _ptr(seq_lens), _ptr(k_tree), _ptr(v_tree), _ptr(mask),
                                     mstride, B, N, Hq, Hkv, D, _code(q.dtype), scale, _ptr(out), _ptr(lse),
                                     _ptr(workspace), workspace.numel(), num_ctas, flags, _ptr(status),
                                     _stream(stream)))
    return out


def tv_tree_attn_verify_rope(q, k_cache, v_cache, block_table, seq_lens, k_tree, v_tree, mask, cos_sin, *,
                             scale=None, out=None, lse=None, workspace=None, num_ctas=0, flags=0, status=None,
                             stream=None):
    """Tree attention with Q rotated as it is loaded (q unrotated and left as
    it is; k_tree already rotated); returns out [B, N, Hq, D], the same bits as
    tv_rope_apply followed by tv_tree_attn_verify."""
    dts = (torch.float32, torch.bfloat16)
    _dev(q, "q", dts)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_tree", k_tree), ("v_tree", v_tree)):
        _dev(t, name, (q.dtype,))
    _dev(block_table, "block_table", (torch.int32,))
    _dev(seq_lens, "seq_lens", (torch.int32,))
    _dev(mask, "mask", (torch.int64,))
    _dev(cos_sin, "cos_sin", (torch.float32,))
    B, N, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    num_blocks, _, block_size, _ = k_cache.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(tv_tree_attn_workspace_size(B, N, Hq, Hkv, D, q.dtype, block_size, num_ctas,
                                                                flags | TV_ATTN_ROPE_Q), q.device)
    mstride = 0 if mask.dim() == 1 else mask.stride(0)
    _check("tv_tree_attn_verify_rope",
           lib().tv_tree_attn_verify_rope(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, block_size,
                                          _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(k_tree),
                                          _ptr(v_tree), _ptr(mask), mstride, _ptr(cos_sin), cos_sin.shape[0], B, N,
                                          Hq, Hkv, D, _code(q.dtype), scale, _ptr(out), _ptr(lse), _ptr(workspace),
                                          workspace.numel(), num_ctas, flags, _ptr(status), _stream(stream)))
    return out


def tv_tree_prepare(parent, seq_lens, k_tree=None, cos_sin=None, *, q=None, n_nodes=None, status=None, mask=None,
                    depth=None, pos=None, stream=None):
    """tv_tree_mask plus the rotation of k_tree [B, N, Hkv, D] and/or q
    [B, N, Hq, D] in place at pos, in one launch; returns (mask, depth, pos)
    like tv_tree_mask."""
    _dev(parent, "parent", (torch.int32,))
    _dev(seq_lens, "seq_lens", (torch.int32,))
    if n_nodes is not None:
        _dev(n_nodes, "n_nodes", (torch.int32,))
    B = seq_lens.numel()
    N = parent.shape[-1]
    bstride = 0 if parent.dim() == 1 else parent.stride(0)
    dev = seq_lens.device
    mask = torch.empty(B, N, dtype=torch.int64, device=dev) if mask is None else mask
    depth = torch.empty(B, N, dtype=torch.int32, device=dev) if depth is None else depth
    pos = torch.empty(B, N, dtype=torch.int32, device=dev) if pos is None else pos
    Hq = Hkv = D = dt = max_pos = 0
    for t, nm in ((q, "q"), (k_tree, "k_tree")):
        if t is not None:
            _dev(t, nm, (torch.float32, torch.bfloat16))
            _dev(cos_sin, "cos_sin", (torch.float32,))
            D, dt, max_pos = t.shape[3], _code(t.dtype), cos_sin.shape[0]
    if q is not None:
        Hq = q.shape[2]
    if k_tree is not None:
        Hkv = k_tree.shape[2]
    _check("tv_tree_prepare",
           lib().tv_tree_prepare(_ptr(parent), bstride, _ptr(seq_lens), _ptr(n_nodes), B, N, _ptr(mask),
                                 _ptr(depth), _ptr(pos), _ptr(q), Hq, _ptr(k_tree), Hkv, D, dt, _ptr(cos_sin),
                                 max_pos, _ptr(status), _stream(stream)))
    return mask, depth, pos


def tv_tree_attn_static_workspace_bytes():
    return lib().tv_tree_attn_static_workspace_bytes()


def tv_tree_attn_verify_static(q, k_cache, v_cache, block_table, seq_lens, k_tree, v_tree, mask, *, scale=None,
                               out=None, lse=None, num_ctas=0, flags=0, status=None, stream=None):
    """Tree attention without a caller workspace (the library's fixed scratch
    array is used); same arguments and result as tv_tree_attn_verify."""
    dts = (torch.float32, torch.bfloat16)
    _dev(q, "q", dts)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_tree", k_tree), ("v_tree", v_tree)):
        _dev(t, name, (q.dtype,))
    _dev(block_table, "block_table", (torch.int32,))
    _dev(seq_lens, "seq_lens", (torch.int32,))
    _dev(mask, "mask", (torch.int64,))
    B, N, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    num_blocks, _, block_size, _ = k_cache.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    mstride = 0 if mask.dim() == 1 else mask.stride(0)
    _check("tv_tree_attn_verify_static",
           lib().tv_tree_attn_verify_static(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, block_size,
                                            _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(k_tree),
                                            _ptr(v_tree), _ptr(mask), mstride, B, N, Hq, Hkv, D, _code(q.dtype),
                                            scale, _ptr(out), _ptr(lse), num_ctas, flags, _ptr(status),
                                            _stream(stream)))
    return out


def _accept_outputs(B, out_cols, device, out, n_out, path):
    if out is None:
        out = torch.empty(B, out_cols, dtype=torch.int32, device=device)
    if n_out is None:
        n_out = torch.empty(B, dtype=torch.int32, device=device)
    if path is None:
        path = torch.empty(B, out_cols, dtype=torch.int32, device=device)
    return out, n_out, path


def tv_tree_accept_greedy(tokens, parent, *, logits=None, target_argmax=None, n_nodes=None, out_cols=None,
                          out=None, n_out=None, path=None, status=None, stream=None):
    """Greedy walk; returns (out [B, out_cols], n_out [B], path [B, out_cols])."""
    _dev(tokens, "tokens", (torch.int32,))
    _dev(parent, "parent", (torch.int32,))
    B, N = tokens.shape
    if logits is not None:
        _dev(logits, "logits", (torch.float32,))
        V = logits.shape[-1]
    else:
        _dev(target_argmax, "target_argmax", (torch.int32,))
        V = 1
    out_cols = N if out_cols is None else out_cols
    out, n_out, path = _accept_outputs(B, out_cols, tokens.device, out, n_out, path)
    bstride = 0 if parent.dim() == 1 else parent.stride(0)
    _check("tv_tree_accept_greedy",
           lib().tv_tree_accept_greedy(_ptr(logits), _ptr(target_argmax), _ptr(tokens), _ptr(parent), bstride,
                                       _ptr(n_nodes), B, N, V, _ptr(out), _ptr(n_out), _ptr(path), out_cols,
                                       _ptr(status), _stream(stream)))
    return out, n_out, path


def tv_accept_sample_workspace_size(B, N, V):
    """Bytes of the grid sampler's workspace (tv_tree_accept_sample and
    tv_chain_accept_sample with N = K + 1)."""
    return int(lib().tv_accept_sample_workspace_size(B, N, V))


def tv_accept_sample_uses_grid(B, N, V, flags=0, workspace_bytes=0):
    """Whether a sampler call with these sizes, flags and workspace size takes
    the grid sampler (queries the current device)."""
    g = ctypes.c_int32(0)
    _check("tv_accept_sample_uses_grid",
           lib().tv_accept_sample_uses_grid(B, N, V, int(flags), int(workspace_bytes), ctypes.addressof(g)))
    return bool(g.value)


def _ws(workspace):
    if workspace is None:
        return None, 0
    _dev(workspace, "workspace", (torch.uint8,))
    return workspace, workspace.numel()


def tv_tree_accept_sample(p, q, tokens, parent, u_accept, u_final, *, n_nodes=None, out_cols=None, out=None,
                          n_out=None, path=None, flags=0, workspace=None, status=None, stream=None):
    """Stochastic walk; returns (out [B, out_cols], n_out [B], path [B, out_cols]).
    flags: TV_SAMPLE_AUTO / TV_SAMPLE_CLUSTER / TV_SAMPLE_SINGLE_CTA / TV_SAMPLE_STREAM /
    TV_SAMPLE_GRID; workspace: uint8 device tensor of
    tv_accept_sample_workspace_size(B, N, V) bytes (alloc_workspace), or None."""
    _dev(p, "p", (torch.float32,))
    _dev(q, "q", (torch.float32,))
    _dev(tokens, "tokens", (torch.int32,))
    _dev(parent, "parent", (torch.int32,))
    _dev(u_accept, "u_accept", (torch.float32,))
    _dev(u_final, "u_final", (torch.float32,))
    B, N, V = p.shape
    out_cols = N if out_cols is None else out_cols
    out, n_out, path = _accept_outputs(B, out_cols, p.device, out, n_out, path)
    bstride = 0 if parent.dim() == 1 else parent.stride(0)
    ws, ws_bytes = _ws(workspace)
    _check("tv_tree_accept_sample",
           lib().tv_tree_accept_sample(_ptr(p), _ptr(q), _ptr(tokens), _ptr(parent), bstride, _ptr(n_nodes),
                                       _ptr(u_accept), _ptr(u_final), B, N, V, _ptr(out), _ptr(n_out), _ptr(path),
                                       out_cols, int(flags), _ptr(ws), ws_bytes, _ptr(status), _stream(stream)))
    return out, n_out, path


def tv_chain_accept_sample(p, q, draft, u, u_final, *, num_draft=None, out_cols=None, out=None, n_out=None,
                           flags=0, workspace=None, status=None, stream=None):
    """The verifier page's chain walk, read in place: p float32 [B, K + 1, V],
    q float32 [B, K, V], draft int32 [B, K], u float32 [B, K], u_final float32
    [B], num_draft int32 [B] (optional), workspace as in tv_tree_accept_sample
    (N = K + 1).  Returns (out [B, out_cols] -1 padded, n_out [B] =
    accepted + 1); allocates nothing when out and n_out are given."""
    _dev(p, "p", (torch.float32,))
    _dev(q, "q", (torch.float32,))
    _dev(draft, "draft", (torch.int32,))
    _dev(u, "u", (torch.float32,))
    _dev(u_final, "u_final", (torch.float32,))
    if num_draft is not None:
        _dev(num_draft, "num_draft", (torch.int32,))
    B, K1, V = p.shape
    K = K1 - 1
    if tuple(q.shape) != (B, K, V) or tuple(draft.shape) != (B, K) or tuple(u.shape) != (B, K):
        raise ValueError("tv_chain_accept_sample: q [B, K, V], draft and u [B, K] with p [B, K + 1, V]")
    out_cols = K1 if out_cols is None else out_cols
    out, n_out, _ = _accept_outputs(B, out_cols, p.device, out, n_out, False)
    ws, ws_bytes = _ws(workspace)
    _check("tv_chain_accept_sample",
           lib().tv_chain_accept_sample(_ptr(p), _ptr(q), _ptr(draft), _ptr(num_draft), _ptr(u), _ptr(u_final), B,
                                        K, V, _ptr(out), _ptr(n_out), out_cols, int(flags), _ptr(ws), ws_bytes,
                                        _ptr(status), _stream(stream)))
    return out, n_out


def verify_chain(draft, q, p, num_draft, u, u_final, *, flags=0, out=None, n_out=None, workspace=None, status=None,
                 stream=None):
    """The verifier page's verify(draft, q, p, num_draft, u, u_final) call:
    draft int32 [B, K] (draft j drawn from q[:, j]); q float32 [B, K, V]; p
    float32 [B, K + 1, V] (the target after each prefix, the last row for the
    bonus); num_draft int32 [B] (ragged); u float32 [B, K] (one uniform per
    test); u_final float32 [B].  Returns (out int32 [B, K + 1] -1 padded,
    n_out int32 [B] = accepted + 1).  Marshalling only, through
    tv_chain_accept_sample: the arrays are read in place, and with out and
    n_out given nothing is allocated."""
    return tv_chain_accept_sample(p, q, draft, u, u_final, num_draft=num_draft, out=out, n_out=n_out, flags=flags,
                                  workspace=workspace, status=status, stream=stream)


def accept_greedy(parent, tokens, target_argmax, *, n_nodes=None, status=None, stream=None):
    """The mask page's accept_greedy(parent, tokens, target_argmax) on top of
    tv_tree_accept_greedy: parent int32 [N] or [B, N], tokens int32 [B, N],
    target_argmax int32 [B, N] (the target's choice after each node).  Returns
    (out, n_out, path) like tv_tree_accept_greedy."""
    return tv_tree_accept_greedy(tokens, parent, target_argmax=target_argmax, n_nodes=n_nodes, status=status,
                                 stream=stream)


def tv_kv_commit(k_cache, v_cache, block_table, seq_lens, k_tree, v_tree, path, n_out, *, new_seq_lens=None,
                 status=None, stream=None):
    """Copy the accepted path's tree K/V rows into the paged cache (in place);
    returns new_seq_lens int32 [B] = seq_lens + n_out."""
    for t, nm in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_tree, "k_tree"), (v_tree, "v_tree")):
        _dev(t, nm, (torch.float32, torch.bfloat16))
    for t, nm in ((block_table, "block_table"), (seq_lens, "seq_lens"), (path, "path"), (n_out, "n_out")):
        _dev(t, nm, (torch.int32,))
    num_blocks, Hkv, bs, D = k_cache.shape
    B, N = k_tree.shape[0], k_tree.shape[1]
    if new_seq_lens is None:
        new_seq_lens = torch.empty_like(seq_lens)
    _check("tv_kv_commit",
           lib().tv_kv_commit(_ptr(k_cache), _ptr(v_cache), num_blocks, bs, _ptr(block_table), block_table.shape[1],
                              _ptr(seq_lens), _ptr(new_seq_lens), _ptr(k_tree), _ptr(v_tree), _ptr(path),
                              path.shape[1], _ptr(n_out), B, N, Hkv, D, _code(k_cache.dtype), _ptr(status),
                              _stream(stream)))
    return new_seq_lens
