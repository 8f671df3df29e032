#!/usr/bin/env python3
"""Benchmark of one draft-tree verification step on a GB300.

A step is one pass of the whole path over one batch: tree mask and positions
(tv_tree_mask), depth-indexed RoPE of the tree queries and keys
(tv_rope_apply), tree attention over the paged KV cache (tv_tree_attn_verify:
one persistent tcgen05 kernel, or plan + CUDA-core kernel + combine) and tree
acceptance (tv_tree_accept_greedy from the target logits, or
tv_tree_accept_sample).  The static tree's rank paths are built once with
tv_tree_build, as a static tree is in serving.

Reported (one JSON line on rank 0):
  value       tree-verify nodes/s (B * N per step) over the timed steps with
              every input resident in HBM, max over ranks; the step is
              captured once as a CUDA graph and replayed (--eager: direct
              calls, host work between the launches included);
  roofline    the tree-attention call: algorithmic bytes (prefix K+V + tree
              K+V + Q + O) / its CUDA-event time (graph replays of that call
              alone), against the measured HBM peak;
  e2e         the same metric through the public API, called directly (no
              graph), with the step's inputs copied from pinned host memory
              (on a copy stream, overlapping the previous step's kernels)
              and the accepted tokens read back;
  cpu_baseline the CPU oracle timed on a bounded sample of the same workload.
With --impl reference the CPU oracle itself is timed (the reference arm).
"""

from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_tree_attn_gb300 import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "b64_l1k_8k_n64_greedy"
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
ATTN_SOURCES = ["attn.cu", "attn_tc.cu", "attn_common.cuh", "attn_tc.h", "rope_math.cuh"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--flags", type=int, default=0, help="tree attention kernel selection (0 auto, 1 CUDA-core, 2 tcgen05)")
    ap.add_argument("--num-ctas", type=int, default=0)
    ap.add_argument("--requests", type=int, default=0,
                    help="run the workload's shapes with this many requests (a small case for profiler captures; "
                         "0: the workload's own batch)")
    ap.add_argument("--rope", default="auto", choices=["auto", "fused", "separate"],
                    help="fused: tree-key RoPE inside the mask kernel and Q RoPE inside the attention kernel's Q load; "
                         "separate: tv_tree_prepare rotating Q and the tree keys, then tv_tree_attn_verify; auto: fused where it "
                         "measured faster (the one-M-tile kernel, G*N <= 128, with B*Hkv >= 2 x SMs), else separate")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other target configurations after the headline")
    ap.add_argument("--eager", action="store_true", help="time eager calls instead of CUDA-graph replays")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--oracle-single-core", default=None, metavar="LENS",
                    help="internal (run by the cpu_baseline leg with one BLAS/OpenMP thread): time the oracle on "
                         "requests of these comma-separated prefix lengths and print one JSON line")
    ap.add_argument("--oracle-worker", action="store_true",
                    help="internal: with --oracle-single-core, build the inputs, run --warmup requests, print "
                         "'ready', wait for a line on stdin, then time the requests in turn (cycling) for "
                         "--cpu-seconds, or for exactly --steps requests when --cpu-seconds is 0")
    return ap.parse_args()


# --------------------------------------------------------------------------- helpers

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available() and args.impl == "ours":
        torch.cuda.set_device(0)
    return world, rank, local


def rank_workload(w, rank):
    """The batch one rank runs: rank 0 the workload itself, rank r > 0 the
    same shapes and distributions with its own seed (its own requests)."""
    return w if rank == 0 else dataclasses.replace(w, seed=w.seed + 7919 * rank)


def max_over_ranks(x, world, device="cpu"):
    """The largest of the ranks' values (the slowest rank sets the time)."""
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def attn_source_hash():
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        p = os.path.join(ROOT, "speculative_decoding_tree_attn_gb300", "csrc", f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current attention sources for this workload (else None)."""
    path = os.path.join(ROOT, "profiles", "attn_traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    for r in rec if isinstance(rec, list) else [rec]:
        if r.get("workload") == workload and r.get("source_sha") == attn_source_hash():
            return r.get("dram_bytes_per_call")
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(device_index)
        self.cmd = ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "100"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for r in csv.reader(f):
                if len(r) >= 7:
                    rows.append([x.strip() for x in r])
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[3 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def attention_bytes(w, lens, N, esize, counts=None):
    """Algorithmic bytes of one attention call: prefix K+V, then the tree K+V
    and Q+O rows of the nodes present (all N, or n_b per ragged request)."""
    nodes = w.B * N if counts is None else int(np.sum(counts))
    kv = int(np.sum(lens)) * w.Hkv * w.D * 2 * esize
    tree = nodes * w.Hkv * w.D * 2 * esize
    qo = 2 * nodes * w.Hq * w.D * esize
    return kv + tree + qo


# --------------------------------------------------------------------------- CPU oracle

def request_paths(w):
    """Rank paths of every request's tree: one best-first tree per request for
    a dynamic workload, else the workload's static tree for all."""
    return W.dynamic_rank_paths(w) if w.dynamic else [w.paths()] * w.B


def oracle_sample_run(w, inp_cpu, req_paths, greedy, sample, requests, counts):
    """The oracle on a list of requests (every present node, all heads) plus
    acceptance."""
    from oracle import accept as OA
    from oracle import attention as OAt
    from oracle import tree as OT

    for b in requests:
        parent, depth, rows, _ = OT.build_tree(req_paths[b])
        n_b = counts[b:b + 1]
        OT.tree_mask_batch(parent[None], inp_cpu["seq_lens"][b:b + 1], n_b)
        sl = slice(b, b + 1)
        OAt.tree_attention(inp_cpu["q"][sl], inp_cpu["k_cache"], inp_cpu["v_cache"], inp_cpu["block_table"][sl],
                           inp_cpu["seq_lens"][sl], inp_cpu["k_tree"][sl], inp_cpu["v_tree"][sl], parent,
                           nodes=[(0, i) for i in range(int(n_b[0]))], n_nodes=n_b)
        if greedy is not None:
            am = OA.argmax_rows(greedy["logits"][b])
            OA.tree_accept_greedy(am[None], greedy["tokens"][sl], parent, n_b)
        if sample is not None:
            OA.tree_accept_sample(sample["p"][sl], sample["q"][sl], sample["tokens"][sl], sample["parent"],
                                  sample["n_nodes"][sl], sample["u_accept"][sl], sample["u_final"][sl])


def cpu_inputs(w, device_inp, greedy, sample):
    def c(t):
        return (t.float() if t.dtype == torch.bfloat16 else t).cpu().numpy()
    inp = {k: c(v) for k, v in device_inp.items()}
    g = {k: c(v) for k, v in greedy.items()} if greedy else None
    s = {k: c(v) for k, v in sample.items()} if sample else None
    return inp, g, s


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def time_oracle(w, inp_cpu, req_paths, greedy, sample, seconds, order, counts, cycle=False, max_requests=None):
    """Times the oracle request by request until `seconds` elapse (or
    max_requests are done); with `cycle` the order repeats.  Returns
    (nodes/s, requests used, elapsed)."""
    done, t0 = [], time.perf_counter()
    while True:
        for b in order:
            oracle_sample_run(w, inp_cpu, req_paths, greedy, sample, [b], counts)
            done.append(int(b))
            if (max_requests is not None and len(done) >= max_requests) or \
                    (max_requests is None and time.perf_counter() - t0 >= seconds):
                el = time.perf_counter() - t0
                return int(np.sum(counts[done])) / el, done, el
        if not cycle:
            break
    el = time.perf_counter() - t0
    return int(np.sum(counts[done])) / el, done, el


def sample_order(lens, seed=0):
    rng = np.random.default_rng(seed)
    first = [int(np.argmin(lens)), int(np.argmax(lens))]
    rest = [int(b) for b in rng.permutation(len(lens)) if b not in first]
    return first + rest


# --------------------------------------------------------------------------- GPU step

class Step:
    def __init__(self, w, dev, flags, num_ctas, rope="fused"):
        from speculative_decoding_tree_attn_gb300 import capi
        self.capi, self.w, self.dev = capi, w, dev
        self.paths = w.paths()
        self.req_paths = request_paths(w)
        # blocks placed for max_depth + 1 positions past each prefix: room to
        # commit the accepted path (timed separately, see kv_commit)
        self.inp = W.attention_inputs(w, device=dev, reserve=w.max_depth + 1)
        if w.dynamic:  # one tree per request: parent [B, N]
            parent = np.stack([capi.tv_tree_build(p)[0] for p in self.req_paths]).astype(np.int32)
            n = parent.shape[1]
        else:
            parent, depth, rows, _, n = capi.tv_tree_build(self.paths)
        self.N = n
        self.parent = torch.from_numpy(parent).to(dev)
        B = w.B
        self.seq_lens = self.inp["seq_lens"]
        self.lens = self.seq_lens.cpu().numpy()
        self.mask = torch.empty(B, n, dtype=torch.int64, device=dev)
        self.depth = torch.empty(B, n, dtype=torch.int32, device=dev)
        self.pos = torch.empty(B, n, dtype=torch.int32, device=dev)
        self.table = capi.tv_rope_table(int(self.lens.max()) + n + 1, w.D, device=dev)
        self.out = torch.empty_like(self.inp["q"])
        dt = self.inp["q"].dtype
        self.flags, self.num_ctas = flags, num_ctas
        # the workspace is allocated zeroed and every completed call leaves its
        # arrival counters zero, so the calls skip clearing them
        self.call_flags = flags | capi.TV_ATTN_WORKSPACE_ZEROED
        # auto: fused where it measured faster -- the one-M-tile kernel with
        # enough (request, KV head) units for two busy CTAs per SM
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.fused_rope = rope == "fused" or (rope == "auto" and (w.Hq // w.Hkv) * n <= 128
                                              and B * w.Hkv >= 2 * sms)
        ws_flags = flags | (capi.TV_ATTN_ROPE_Q if self.fused_rope else 0)
        self.ws = capi.alloc_workspace(capi.tv_tree_attn_workspace_size(B, n, w.Hq, w.Hkv, w.D, dt, w.block_size,
                                                                         num_ctas, ws_flags), dev)
        self.greedy = self.sample = None
        if w.accept == "greedy":
            self.greedy = W.greedy_inputs(w, parent, device=dev)
        elif w.accept == "sample":
            self.sample = (W.sample_tree_inputs(w, parent, device=dev) if w.sample_tree
                           else W.sample_chain_inputs(w, device=dev))
        cols = n if self.sample is None else self.sample["p"].shape[1]
        # the sampler's workspace: with it TV_SAMPLE_AUTO may take the grid
        # sampler (walk, pass and draw kernels, then the single-launch walk
        # of the requests they leave)
        self.sample_ws, acc_launches = None, 1
        if self.sample is not None:
            sB, sN, sV = self.sample["p"].shape
            ws_bytes = capi.tv_accept_sample_workspace_size(sB, sN, sV)
            self.sample_ws = capi.alloc_workspace(ws_bytes, dev)
            acc_launches = 4 if capi.tv_accept_sample_uses_grid(sB, sN, sV, 0, ws_bytes) else 1
        self.acc_out = torch.empty(B, cols, dtype=torch.int32, device=dev)
        self.acc_n = torch.empty(B, dtype=torch.int32, device=dev)
        self.acc_path = torch.empty(B, cols, dtype=torch.int32, device=dev)
        self.esize = 2 if dt == torch.bfloat16 else 4
        self.counts = W.node_counts(w)  # nodes present per request (all n unless ragged)
        self.n_nodes = torch.from_numpy(self.counts).to(dev) if w.ragged else None
        self.attn_bytes = attention_bytes(w, self.lens, n, self.esize, self.counts)
        # tree_mask, rope_apply, the attention kernel(s), the acceptance kernel;
        # the tcgen05 path is one kernel, the CUDA-core path plan + attention +
        # combine
        uses_tc = flags == capi.TV_ATTN_TCGEN05
        if flags == capi.TV_ATTN_AUTO:
            try:
                capi.tv_tree_attn_workspace_size(B, n, w.Hq, w.Hkv, w.D, dt, w.block_size, num_ctas,
                                                 capi.TV_ATTN_TCGEN05 | (ws_flags & capi.TV_ATTN_ROPE_Q))
                uses_tc = True
            except capi.TVError:
                uses_tc = False
        # mask + rope, the attention kernel(s), the acceptance kernel
        self.launches = 1 + (1 if uses_tc else 3) + (acc_launches if w.accept != "none" else 0)

    def run_attn(self):
        i = self.inp
        if self.fused_rope:
            self.capi.tv_tree_attn_verify_rope(i["q"], i["k_cache"], i["v_cache"], i["block_table"], self.seq_lens,
                                               i["k_tree"], i["v_tree"], self.mask, self.table, out=self.out,
                                               workspace=self.ws, num_ctas=self.num_ctas, flags=self.call_flags)
        else:
            self.capi.tv_tree_attn_verify(i["q"], i["k_cache"], i["v_cache"], i["block_table"], self.seq_lens,
                                          i["k_tree"], i["v_tree"], self.mask, out=self.out, workspace=self.ws,
                                          num_ctas=self.num_ctas, flags=self.call_flags)

    def run(self, ev_attn=None):
        c, i = self.capi, self.inp
        if self.fused_rope:  # mask + tree-key rotation in one kernel; Q is rotated inside the attention kernel
            c.tv_tree_prepare(self.parent, self.seq_lens, i["k_tree"], self.table, n_nodes=self.n_nodes,
                              mask=self.mask, depth=self.depth, pos=self.pos)
        else:  # mask + rotation of the queries and tree keys in one kernel, before the attention kernel
            c.tv_tree_prepare(self.parent, self.seq_lens, i["k_tree"], self.table, q=i["q"], n_nodes=self.n_nodes,
                              mask=self.mask, depth=self.depth, pos=self.pos)
        if ev_attn:
            ev_attn[0].record()
        self.run_attn()
        if ev_attn:
            ev_attn[1].record()
        self.run_accept()

    def run_accept(self):
        c = self.capi
        if self.greedy is not None:
            c.tv_tree_accept_greedy(self.greedy["tokens"], self.parent, logits=self.greedy["logits"],
                                    n_nodes=self.n_nodes, out=self.acc_out,
                                    n_out=self.acc_n, path=self.acc_path)
        elif self.sample is not None:
            s = self.sample
            c.tv_tree_accept_sample(s["p"], s["q"], s["tokens"], s["parent"], s["u_accept"], s["u_final"],
                                    n_nodes=s["n_nodes"], out=self.acc_out, n_out=self.acc_n, path=self.acc_path,
                                    workspace=self.sample_ws)

    def commit_path(self):
        """The accepted path of the last step (the deepest chain when the
        workload has no acceptance) as (path int32 [B, cols], n_out int32 [B])."""
        if self.greedy is not None or self.sample is not None:
            return self.acc_path, self.acc_n
        par_all = self.parent.cpu().numpy().reshape(-1, self.N)
        chains = []
        for b in range(self.w.B):
            par = par_all[b % par_all.shape[0]][:int(self.counts[b])]
            depth = np.zeros(par.size, dtype=np.int64)
            for i in range(1, par.size):
                depth[i] = depth[par[i]] + 1
            chain = [int(np.argmax(depth))]
            while chain[-1] != 0:
                chain.append(int(par[chain[-1]]))
            chains.append(chain[::-1])
        cols = max(len(c) for c in chains)
        path = torch.tensor([c + [0] * (cols - len(c)) for c in chains], dtype=torch.int32, device=self.dev)
        n = torch.tensor([len(c) for c in chains], dtype=torch.int32, device=self.dev)
        return path, n

    def run_commit(self, path, n_out, new_lens):
        i = self.inp
        self.capi.tv_kv_commit(i["k_cache"], i["v_cache"], i["block_table"], self.seq_lens, i["k_tree"], i["v_tree"],
                               path, n_out, new_seq_lens=new_lens)

    def bind(self, t):
        """Points the step at another set of per-step input tensors (the names
        and shapes of per_step_inputs)."""
        self.inp = dict(self.inp, q=t["q"], k_tree=t["k_tree"], v_tree=t["v_tree"], block_table=t["block_table"],
                        seq_lens=t["seq_lens"])
        self.seq_lens, self.parent = t["seq_lens"], t["parent"]
        if self.greedy is not None:
            self.greedy = dict(self.greedy, tokens=t["tokens"], logits=t["logits"])
        if self.sample is not None:
            self.sample = {k: t[f"s_{k}"] for k in self.sample}

    def per_step_inputs(self):
        """Tensors a caller supplies fresh every step (the KV cache is resident state)."""
        t = {"q": self.inp["q"], "k_tree": self.inp["k_tree"], "v_tree": self.inp["v_tree"],
             "block_table": self.inp["block_table"], "seq_lens": self.seq_lens, "parent": self.parent}
        if self.greedy is not None:
            t.update(tokens=self.greedy["tokens"], logits=self.greedy["logits"])
        if self.sample is not None:
            t.update({f"s_{k}": v for k, v in self.sample.items()})
        return t


def l2_flush_buffer(st, dev):
    """A buffer larger than L2 to overwrite between timed iterations when a
    step's data would otherwise stay in L2 (None when it cannot)."""
    ws_bytes = st.attn_bytes + sum(t.numel() * t.element_size() for t in st.per_step_inputs().values())
    flush = torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device=dev) if ws_bytes < 2 * L2_BYTES else None
    return flush, ws_bytes


def measure_step(st, args, flush, world=1):
    """W warm-up steps, then K timed steps and K timed attention calls (CUDA
    graph replays unless --eager), CUDA events on the launching stream, SM
    clocks sampled during the timed region.  Returns (step_ms, attn_ms,
    clocks, graphs)."""
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    eva = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    graphs = None
    if not args.eager:
        # The step (and, for the roofline, the attention call alone) captured
        # once as CUDA graphs and replayed: the same kernels as an eager call,
        # without the per-call host work between them.
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            st.run()
        torch.cuda.current_stream().wait_stream(side)
        g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            st.run()
        with torch.cuda.graph(g_attn):
            st.run_attn()
        for _ in range(args.warmup):
            g_step.replay()
        graphs = (g_step, g_attn)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    with sampler:
        for k in range(args.steps):
            if flush is not None:
                flush.zero_()
            evs[k][0].record()
            if graphs:
                graphs[0].replay()
            else:
                st.run(eva[k])
            evs[k][1].record()
        if graphs:
            for k in range(args.steps):
                if flush is not None:
                    flush.zero_()
                eva[k][0].record()
                graphs[1].replay()
                eva[k][1].record()
        torch.cuda.synchronize()
    clocks = sampler.summary()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    attn_ms = [a.elapsed_time(b) for a, b in eva]
    return step_ms, attn_ms, clocks, graphs


def roofline_of(st, w, attn_ms):
    peak, peak_kind = measured_hbm_peak()
    attn_mean_ms = statistics.mean(attn_ms)
    achieved = st.attn_bytes / (attn_mean_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": recorded_traffic(w.name),
            "kernel": ("tv_tree_attn_verify_rope" if st.fused_rope else "tv_tree_attn_verify")
                      + " (tcgen05: one persistent kernel; the arrival counters are left zero by each call)",
            "algorithmic_bytes_per_call": int(st.attn_bytes), "peak_kind": f"{peak_kind} hbm_gbs",
            "attn_ms_mean": round(attn_mean_ms, 4)}


# Every target configuration, timed after the headline in the same run and
# reported under "per_config" (the headline workload included, as measured
# there).
PER_CONFIG = ["gqa_b8_l512_2048_n26", "b64_l1k_8k_n64_greedy", "long_b16_l32k_n33", "b256_l2k_4k_n10_sample"]


def measure_accept(st, w, args, flush, dev):
    """The acceptance call alone (graph replays, L2 flushed before each):
    time per call, tokens emitted and the row bytes the walk reads -- the
    lazy greedy walk one logits row per emitted token; the chain sampler the
    p row of its stop node, plus its q row when the stop was a rejection."""
    if st.greedy is None and st.sample is None:
        return None
    g_acc = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_acc):
        st.run_accept()
    fl = flush if flush is not None else torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    evc = []
    for k in range(args.warmup + args.steps):
        fl.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g_acc.replay()
        b.record()
        if k >= args.warmup:
            evc.append((a, b))
    torch.cuda.synchronize()
    us = statistics.mean(a.elapsed_time(b) for a, b in evc) * 1e3
    emitted = int(st.acc_n.sum().item())
    accept = {"call": "tv_tree_accept_greedy" if st.greedy is not None else "tv_tree_accept_sample",
              "us_per_call": round(us, 2), "tokens_out": emitted}
    rows_b = None
    if st.greedy is not None:
        rows_b = emitted * w.vocab * 4
        accept["all_rows_bytes"] = w.B * st.N * w.vocab * 4
    elif not w.sample_tree:
        n_out = st.acc_n.cpu().numpy().astype(np.int64)
        n_nodes = st.sample["n_nodes"].cpu().numpy().astype(np.int64)
        V = st.sample["p"].shape[-1]
        rejected = n_out < n_nodes  # the stop node still had its child to test
        rows_b = int(np.sum(np.where(rejected, 2, 1))) * V * 4
    if rows_b is not None:
        accept.update(bytes_read=rows_b, gbs=round(rows_b / (us * 1e-6) / 1e9, 1))
    del g_acc
    return accept


def measure_config(name, args, dev):
    """One workload's attention call and step, measured as the headline is."""
    w = W.WORKLOADS[name]
    st = Step(w, dev, args.flags, args.num_ctas, args.rope)
    flush, ws_bytes = l2_flush_buffer(st, dev)
    step_ms, attn_ms, clocks, graphs = measure_step(st, args, flush)
    roof = roofline_of(st, w, attn_ms)
    nodes = int(np.sum(st.counts))
    ms = statistics.mean(step_ms)
    res = {"attn_ms_mean": roof["attn_ms_mean"], "frac": roof["frac"], "achieved_gbs": roof["achieved"],
           "algorithmic_bytes": roof["algorithmic_bytes_per_call"], "traffic": roof["traffic"],
           "ms_per_step": round(ms, 4), "nodes_per_s": nodes / (ms / 1e3), "nodes_per_step": nodes,
           "accept": w.accept, "rope": "fused" if st.fused_rope else "separate",
           "l2": "flushed between steps" if flush is not None else "inputs larger than L2",
           "clocks": clocks}
    acc = measure_accept(st, w, args, flush, dev) if graphs else None
    if acc is not None:
        res["accept_us_per_call"] = acc["us_per_call"]
        if "gbs" in acc:
            res["accept_bytes_read"], res["accept_gbs"] = acc["bytes_read"], acc["gbs"]
    del st, graphs, flush
    torch.cuda.empty_cache()
    return res


def run_ours(args, world, rank, local):
    base = W.WORKLOADS[args.workload]
    if args.requests:
        base = dataclasses.replace(base, B=args.requests)
    w = rank_workload(base, rank)
    dev = torch.device("cuda", torch.cuda.current_device())
    st = Step(w, dev, args.flags, args.num_ctas, args.rope)
    flush, ws_bytes = l2_flush_buffer(st, dev)
    step_ms, attn_ms, clocks, graphs = measure_step(st, args, flush, world)
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, world, dev)
    if world > 1:
        torch.distributed.barrier()
    nodes = int(np.sum(st.counts))
    value = world * nodes * args.steps / (total_ms / 1e3)

    # end to end through the public API: pinned host inputs in, accepted tokens
    # out.  Two sets of device input buffers: step k + 1's host-to-device
    # copies run on a copy stream while step k's kernels run.
    e2e = None
    if not args.no_e2e:
        base = st.per_step_inputs()
        host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) for k, v in base.items()}
        sets = [base, {k: torch.empty_like(v) for k, v in base.items()}]
        h_out = torch.empty(st.acc_out.shape, dtype=torch.int32, pin_memory=True)
        h_n = torch.empty(st.acc_n.shape, dtype=torch.int32, pin_memory=True)
        bi = sum(v.numel() * v.element_size() for v in host.values())
        bo = h_out.numel() * 4 + h_n.numel() * 4
        comp, copy_s = torch.cuda.current_stream(), torch.cuda.Stream()
        copied = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        copy_s.wait_event(e0)
        for k in range(args.steps):
            j = k % 2
            with torch.cuda.stream(copy_s):
                if k >= 2:
                    copy_s.wait_event(freed[j])  # step k - 2 is done with this set
                for name, v in host.items():
                    sets[j][name].copy_(v, non_blocking=True)
                copied[j].record(copy_s)
            comp.wait_event(copied[j])
            st.bind(sets[j])
            st.run()
            h_out.copy_(st.acc_out, non_blocking=True)
            h_n.copy_(st.acc_n, non_blocking=True)
            freed[j].record(comp)
        e1.record(comp)
        torch.cuda.synchronize()
        st.bind(base)
        e_ms = e0.elapsed_time(e1)
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": world * nodes * args.steps / (e_ms / 1e3), "unit": "nodes/s",
               "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
               "pipelining": "two input buffer sets; step k + 1's host-to-device copies overlap step k's kernels"}

    # the accepted path's K/V committed to the cache (a separate call, not in the step)
    commit = None
    if graphs:
        path, n_commit = st.commit_path()
        new_lens = torch.empty_like(st.seq_lens)
        g_commit = torch.cuda.CUDAGraph()
        st.run_commit(path, n_commit, new_lens)
        with torch.cuda.graph(g_commit):
            st.run_commit(path, n_commit, new_lens)
        for _ in range(args.warmup):
            g_commit.replay()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        c0.record()
        for _ in range(args.steps):
            g_commit.replay()
        c1.record()
        torch.cuda.synchronize()
        us = c0.elapsed_time(c1) * 1e3 / args.steps
        rows = int(n_commit.sum().item())
        moved = rows * w.Hkv * w.D * st.esize * 2 * 2  # K and V rows, read and written
        commit = {"us_per_call": round(us, 2), "rows": rows, "bytes": moved, "gbs": round(moved / (us * 1e-6) / 1e9, 1)}

    accept = measure_accept(st, w, args, flush, dev) if graphs else None

    roofline = roofline_of(st, w, attn_ms)
    achieved, peak = roofline["achieved"], roofline["peak"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on every host core: one single-threaded process per core
        # (os.cpu_count()), each on a rotation of the workload's prefix
        # lengths (the shortest and longest first), started together
        lens_s = [int(st.lens[b]) for b in sample_order(st.lens)[:8]]
        try:
            nps, procs, res = oracle_all_cores(w, lens_s, seconds=args.cpu_seconds)
            cpu = {"value": nps, "unit": "nodes/s", "cores": procs, "kind": "oracle",
                   "sample": f"{procs} single-threaded processes started together, each timing the oracle "
                             f"(all nodes and heads of a request, acceptance incl.) on a rotation of prefix "
                             f"lengths {lens_s} for {args.cpu_seconds:.0f} s: {sum(r['requests'] for r in res)} "
                             f"requests, {sum(r['nodes'] for r in res)} nodes in "
                             f"{max(r['seconds'] for r in res):.1f} s (inputs regenerated on the CPU with the "
                             f"workload's recipe)",
                   "blas_threads_per_process": 1,
                   "single_core": oracle_single_core(w, lens_s[:6], min(8.0, args.cpu_seconds))}
        except (RuntimeError, OSError, subprocess.SubprocessError, ValueError) as e:
            cpu = {"value": None, "unit": "nodes/s", "cores": os.cpu_count(), "kind": "oracle",
                   "error": f"{type(e).__name__}: {e}"[:200]}

    per_config = None
    if rank == 0 and world == 1 and not args.no_per_config:
        del graphs
        torch.cuda.empty_cache()
        per_config = {}
        for name in PER_CONFIG:
            per_config[name] = (measure_config(name, args, dev) if name != w.name else
                                {"attn_ms_mean": roofline["attn_ms_mean"], "frac": roofline["frac"],
                                 "achieved_gbs": roofline["achieved"],
                                 "algorithmic_bytes": roofline["algorithmic_bytes_per_call"],
                                 "traffic": roofline["traffic"], "ms_per_step": round(total_ms / args.steps, 4),
                                 "nodes_per_s": value, "nodes_per_step": nodes, "accept": w.accept,
                                 "rope": "fused" if st.fused_rope else "separate", "clocks": clocks,
                                 "l2": "flushed between steps" if flush is not None else "inputs larger than L2",
                                 "note": "the headline measurement"})

    if rank == 0:
        line = {
            "metric": "tree-verify nodes/s and KV-read HBM GB/s (% of GB300 peak), 1 GPU",
            "value": value, "unit": "nodes/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if st.esize == 2 else "f32",
            "data": "synthetic (seeded; no model weights)",
            "config": {"workload": w.name, "B": w.B, "N": st.N, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "prefix": list(w.prefix), "block_size": w.block_size, "accept": w.accept, "vocab": w.vocab,
                       "tree": "one per request" if w.dynamic else "shared",
                       "nodes_present": int(np.sum(st.counts)),
                       "l2": ("L2 flushed between steps" if flush is not None
                              else f"inputs larger than L2 ({ws_bytes / 2**30:.2f} GiB per step)"),
                       "kernel_flags": args.flags, "parallelism": f"dp{world}: one batch of {w.B} requests per GPU, no collective on the data path",
                       "timing": "eager calls" if args.eager else "CUDA graph replays of the step",
                       "rope": "fused" if st.fused_rope else "separate"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": st.launches * args.steps,
            "kv_commit": commit, "accept": accept,
            "kv_read_gbs": round(achieved, 1), "kv_read_frac_of_peak": round(achieved / peak, 4),
            "per_config": per_config,
        }
        print(json.dumps(line))


def cpu_workload(w, seq_lens=None):
    """The workload's inputs generated on the CPU (the recipe's generators on
    the CPU device), as the oracle takes them."""
    inp = W.attention_inputs(w, device="cpu", seq_lens=seq_lens)
    from oracle import tree as OT
    req_paths = request_paths(w)
    parent = (np.stack([OT.build_tree(p)[0] for p in req_paths]) if w.dynamic else OT.build_tree(w.paths())[0])
    greedy = W.greedy_inputs(w, parent, device="cpu") if w.accept == "greedy" else None
    sample = None
    if w.accept == "sample":
        sample = W.sample_tree_inputs(w, parent, device="cpu") if w.sample_tree else W.sample_chain_inputs(w, device="cpu")
    inp_cpu, g, s = cpu_inputs(w, inp, greedy, sample)
    return inp_cpu, g, s, req_paths, W.node_counts(w)


def run_oracle_single_core(args):
    """One-core oracle timing (the parent starts this process with one BLAS and
    OpenMP thread): requests of the given prefix lengths, generated on the CPU
    with the workload's recipe, timed one by one until --cpu-seconds.  With
    --oracle-worker it is one of several such processes started together
    (all-core figure, reference arm)."""
    lens = np.array([int(x) for x in args.oracle_single_core.split(",")], dtype=np.int32)
    w = dataclasses.replace(W.WORKLOADS[args.workload], B=len(lens))
    inp_cpu, g, s, req_paths, counts = cpu_workload(w, seq_lens=lens)
    order = list(range(len(lens)))
    if args.oracle_worker:
        for k in range(args.warmup):
            oracle_sample_run(w, inp_cpu, req_paths, g, s, [order[k % len(order)]], counts)
        print("ready", flush=True)
        sys.stdin.readline()
        if args.cpu_seconds > 0:
            nps, used, el = time_oracle(w, inp_cpu, req_paths, g, s, args.cpu_seconds, order, counts, cycle=True)
        else:
            nps, used, el = time_oracle(w, inp_cpu, req_paths, g, s, 0, order, counts, cycle=True,
                                        max_requests=args.steps)
    else:
        nps, used, el = time_oracle(w, inp_cpu, req_paths, g, s, args.cpu_seconds, order, counts)
    print(json.dumps({"value": nps, "requests": len(used), "nodes": int(np.sum(counts[used])),
                      "seconds": round(el, 3), "threads": blas_threads()}))


def one_thread_env():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "LOCAL_WORLD_SIZE")}
    env.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    return env


def oracle_all_cores(w, lens, seconds=None, steps=None, warmup=0, timeout=900):
    """One single-threaded oracle process per host core (os.cpu_count()),
    each on its own rotation of the sampled prefix lengths.  Every process
    builds its inputs and runs its warm-up requests, then all are released
    together; each times its requests for `seconds` (cycling), or exactly
    `steps` requests.  Returns (nodes/s over all processes = total nodes /
    longest elapsed time, processes, per-process results)."""
    n = os.cpu_count() or 1
    cmds = []
    for k in range(n):
        mine = [int(lens[(k + j) % len(lens)]) for j in range(min(len(lens), 4))]
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", w.name, "--oracle-single-core",
               ",".join(map(str, mine)), "--oracle-worker", "--warmup", str(warmup),
               "--cpu-seconds", str(seconds if seconds is not None else 0), "--steps", str(steps or 1)]
        cmds.append(cmd)
    procs = [subprocess.Popen(c, env=one_thread_env(), stdin=subprocess.PIPE, stdout=subprocess.PIPE,
                              stderr=subprocess.DEVNULL, text=True) for c in cmds]
    try:
        for pr in procs:  # every process ready (inputs built, warm-up done)
            line = pr.stdout.readline()
            if line.strip() != "ready":
                raise RuntimeError(f"oracle worker did not start ({line.strip()[:80]})")
        for pr in procs:
            pr.stdin.write("go\n")
            pr.stdin.flush()
        res = []
        for pr in procs:
            out, _ = pr.communicate(timeout=timeout)
            res.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for pr in procs:
            if pr.poll() is None:
                pr.kill()
    nodes = sum(r["nodes"] for r in res)
    el = max(r["seconds"] for r in res)
    return nodes / el, n, res


def oracle_single_core(w, lens, seconds):
    """cpu_baseline's one-core figure: run_oracle_single_core in a child
    process with the thread counts pinned to 1."""
    env = one_thread_env()
    cmd = [sys.executable, os.path.abspath(__file__), "--workload", w.name, "--cpu-seconds", str(seconds),
           "--oracle-single-core", ",".join(str(int(x)) for x in lens)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
        out = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"error": f"{type(e).__name__}: {e}"[:200]}
    return {"value": out["value"], "unit": "nodes/s", "cores": out["threads"],
            "sample": f"{out['requests']} requests of prefix lengths {list(map(int, lens))[:out['requests']]}, "
                      f"inputs regenerated on the CPU with the same recipe, {out['seconds']} s"}


def run_reference(args, world, rank):
    """The reference arm: the oracle on every host core.  One single-threaded
    process per core (os.cpu_count()) builds its requests' inputs with the
    workload's recipe and runs --warmup requests; all are then released
    together and each runs --steps requests, one per step (a step is one
    request on every core at once).  value = nodes / the longest process
    time; ms_per_step = that time / steps."""
    if rank != 0:
        return
    w = W.WORKLOADS[args.workload]
    lens = W.prefix_lengths(w)
    lens_s = [int(lens[b]) for b in sample_order(lens)[:8]]
    value, procs, res = oracle_all_cores(w, lens_s, steps=args.steps, warmup=args.warmup)
    el = max(r["seconds"] for r in res)
    line = {
        "impl": "reference",
        "metric": "tree-verify nodes/s and KV-read HBM GB/s (% of GB300 peak), 1 GPU",
        "value": value, "unit": "nodes/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded; no model weights)",
        "config": {"workload": w.name, "B": w.B, "N": w.n_nodes, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "prefix": list(w.prefix), "block_size": w.block_size, "accept": w.accept, "vocab": w.vocab,
                   "tree": "one per request" if w.dynamic else "shared"},
        "cpu_baseline": {"value": value, "unit": "nodes/s", "cores": procs, "kind": "oracle",
                         "blas_threads_per_process": 1,
                         "sample": f"{procs} single-threaded processes, one request each per step (all "
                                   f"{w.n_nodes} nodes, all heads, acceptance incl.), prefix lengths {lens_s} in "
                                   f"rotation; {sum(r['nodes'] for r in res)} nodes in {el:.2f} s"},
        "e2e": {"value": value, "unit": "nodes/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse_args()
    if args.oracle_single_core:
        run_oracle_single_core(args)
        return
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            if not torch.cuda.is_available():
                raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
