// Tree acceptance on the device: one CTA of 1024 threads per request.
//
// Greedy ("Build the tree attention mask that verifies a draft tree in one
// pass", "The mask."; "Encode branch histories in masks and positions"): from
// the root, the target's choice after the current node (largest logit, ties to
// the lowest index -- computed only for the nodes the walk visits) is emitted;
// the walk moves to the lowest-index child carrying that token, else stops.
//
// Stochastic ("Implement the lossless speculative sampling verifier for a
// batch with ragged draft lengths", "A strong answer", "Details that matter in
// review" and "What interviewers probe next"; "Tree Verification", "Accepting
// on a Tree"): children are tested in index order, the first with
// u * q(x) < p(x) is accepted; after each rejection the node's target becomes
// the normalised residual max(0, target - q); when every child is rejected, or
// at a leaf, one token is drawn from the node's current distribution.  The
// residuals and the final inverse-CDF draw use integer images of the rows
// (round(r * 2^40)) so that prefix sums are exact in any summation order:
//
//   level 0            : target p; accept iff (double)u * q(x) < (double)p(x)
//   w_0 = P            : P = rint(2^40 p), Q = rint(2^40 q)
//   w_{m+1}            : max(0, w_m - floor((S_m * Q + 2^39) / 2^40)),
//                        S_0 = 2^40, S_m = W_m = sum(w_m); kept only if W_{m+1} > 0
//   level m >= 1       : accept iff fl64(fl64(u * q(x)) * W_m) < w_m(x)
//   final draw         : min(#{x : prefix_sum(w)(x) < ceil(fl64(u_final * W))}, V - 1)
//
// The row of a level is split into 32 contiguous segments, one per warp; a
// pass over the row leaves each warp's segment total in shared memory, so the
// draw only re-reads the one segment that holds the crossing.
#include <cooperative_groups.h>

#include <climits>

#include "common.h"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

struct AcceptOut {
  int32_t* out;
  int32_t* n_out;
  int32_t* path;
  int out_cols;
  int32_t* status;
};

__device__ __forceinline__ int clamp_nodes(const int32_t* n_nodes, int b, int N) {
  if (!n_nodes) return N;
  int n = n_nodes[b];
  return n < 1 ? 1 : (n > N ? N : n);
}

// Loads parent and token rows of request b into shared memory.
__device__ __forceinline__ void load_tree(const int32_t* parent, int64_t pstride, const int32_t* tokens, int b,
                                          int N, int32_t* s_par, int32_t* s_tok) {
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    s_par[c] = parent[(int64_t)b * pstride + c];
    s_tok[c] = tokens[(int64_t)b * N + c];
  }
}

// Lowest-index valid child of `node` with token `tok` (all threads get it).
__device__ int find_child(const int32_t* s_par, const int32_t* s_tok, int node, int n, int tok, int* s_best) {
  if (threadIdx.x == 0) *s_best = INT_MAX;
  __syncthreads();
  const int c = node + 1 + threadIdx.x;
  if (c < n && s_par[c] == node && s_tok[c] == tok) atomicMin(s_best, c);
  __syncthreads();
  const int r = *s_best;
  __syncthreads();
  return r;
}

__device__ void finish_walk(const AcceptOut& o, int b, int k) {
  for (int j = k + threadIdx.x; j < o.out_cols; j += blockDim.x) {
    o.out[(int64_t)b * o.out_cols + j] = -1;
    if (o.path) o.path[(int64_t)b * o.out_cols + j] = -1;
  }
  if (threadIdx.x == 0) o.n_out[b] = k;
}

__device__ __forceinline__ void emit(const AcceptOut& o, int b, int k, int token, int node) {
  if (threadIdx.x == 0) {
    o.out[(int64_t)b * o.out_cols + k] = token;
    if (o.path) o.path[(int64_t)b * o.out_cols + k] = node;
  }
}

// ------------------------------------------------------------------ greedy

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Block argmax of row[0..V): largest value, lowest index among equals.
__device__ int block_argmax(const float* __restrict__ row, int V, bool vec, float* s_v, int* s_i) {
  float bv = -INFINITY;
  int bi = INT_MAX;
  if (vec) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = V / 4;
#pragma unroll 4
    for (int t = threadIdx.x; t < n4; t += blockDim.x) {
      const float4 x = __ldg(r4 + t);
      const int i = 4 * t;
      if (better(x.x, i, bv, bi)) { bv = x.x; bi = i; }
      if (better(x.y, i + 1, bv, bi)) { bv = x.y; bi = i + 1; }
      if (better(x.z, i + 2, bv, bi)) { bv = x.z; bi = i + 2; }
      if (better(x.w, i + 3, bv, bi)) { bv = x.w; bi = i + 3; }
    }
  } else {
    for (int i = threadIdx.x; i < V; i += blockDim.x) {
      const float x = __ldg(row + i);
      if (better(x, i, bv, bi)) { bv = x; bi = i; }
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  if (lane == 0) { s_v[warp] = bv; s_i[warp] = bi; }
  __syncthreads();
  if (warp == 0) {
    bv = lane < (int)(blockDim.x / 32) ? s_v[lane] : -INFINITY;
    bi = lane < (int)(blockDim.x / 32) ? s_i[lane] : INT_MAX;
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) s_i[0] = bi;
  }
  __syncthreads();
  const int r = s_i[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads) greedy_kernel(const float* __restrict__ logits,
                                                          const int32_t* __restrict__ target_argmax,
                                                          const int32_t* __restrict__ tokens,
                                                          const int32_t* __restrict__ parent, int64_t pstride,
                                                          const int32_t* __restrict__ n_nodes, int N, int V,
                                                          AcceptOut o) {
  __shared__ int32_t s_par[TV_MAX_NODES], s_tok[TV_MAX_NODES];
  __shared__ float s_v[kWarps];
  __shared__ int s_i[kWarps];
  __shared__ int s_best;
  const int b = blockIdx.x;
  load_tree(parent, pstride, tokens, b, N, s_par, s_tok);
  __syncthreads();
  const int n = clamp_nodes(n_nodes, b, N);
  const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  int node = 0, k = 0;
  while (true) {
    int choice;
    if (logits) choice = block_argmax(logits + ((int64_t)b * N + node) * V, V, vec, s_v, s_i);
    else choice = target_argmax[(int64_t)b * N + node];
    emit(o, b, k, choice, node);
    ++k;
    const int nxt = find_child(s_par, s_tok, node, n, choice, &s_best);
    if (nxt == INT_MAX) break;
    if (k == o.out_cols) {
      if (threadIdx.x == 0 && o.status) atomicOr(o.status, TV_DEV_OUT_OVERFLOW);
      break;
    }
    node = nxt;
  }
  finish_walk(o, b, k);
}

// Greedy walk from logits by a cluster of kGreedyCtas CTAs per request: each
// CTA takes the argmax of its contiguous slice of the visited row, the slices'
// results are exchanged through distributed shared memory, and every CTA of
// the cluster continues the walk with the same choice (CTA rank 0 writes the
// outputs).  A row is 128 KB at a 32000-token vocabulary: split eight ways,
// one load per thread fetches a slice, so a step of the walk costs about one
// memory round trip instead of several.
constexpr int kGreedyCtas = 8;
constexpr int kGreedyThreads = 256;

__global__ void __cluster_dims__(kGreedyCtas, 1, 1) __launch_bounds__(kGreedyThreads)
    greedy_cluster_kernel(const float* __restrict__ logits, const int32_t* __restrict__ tokens,
                          const int32_t* __restrict__ parent, int64_t pstride, const int32_t* __restrict__ n_nodes,
                          int N, int V, AcceptOut o) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ int32_t s_par[TV_MAX_NODES], s_tok[TV_MAX_NODES];
  __shared__ float s_v[kGreedyThreads / 32];
  __shared__ int s_i[kGreedyThreads / 32];
  __shared__ float s_res_v[2];  // this CTA's slice result, by step parity (read by the peers)
  __shared__ int s_res_i[2];
  __shared__ int s_choice, s_best;
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / kGreedyCtas;
  load_tree(parent, pstride, tokens, b, N, s_par, s_tok);
  __syncthreads();
  const int n = clamp_nodes(n_nodes, b, N);
  const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  int seg = (V + kGreedyCtas - 1) / kGreedyCtas;
  seg = (seg + 3) / 4 * 4;
  const int lo = rank * seg, hi = min(lo + seg, V);
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int node = 0, k = 0;
  for (int step = 0;; ++step) {
    const float* row = logits + ((int64_t)b * N + node) * V;
    float bv = -INFINITY;
    int bi = INT_MAX;
    if (vec) {
      // kBatch float4 per thread requested together, then compared
      constexpr int kBatch = 4;
      const float4* r4 = reinterpret_cast<const float4*>(row) + lo / 4;
      const int n4 = (hi - lo) / 4;
      for (int base = threadIdx.x; base < n4; base += kBatch * kGreedyThreads) {
        float4 x[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int t = base + u * kGreedyThreads;
          if (t < n4) x[u] = __ldg(r4 + t);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (base + u * kGreedyThreads >= n4) break;
          const int i = lo + 4 * (base + u * kGreedyThreads);
          if (better(x[u].x, i, bv, bi)) { bv = x[u].x; bi = i; }
          if (better(x[u].y, i + 1, bv, bi)) { bv = x[u].y; bi = i + 1; }
          if (better(x[u].z, i + 2, bv, bi)) { bv = x[u].z; bi = i + 2; }
          if (better(x[u].w, i + 3, bv, bi)) { bv = x[u].w; bi = i + 3; }
        }
      }
    } else {
      for (int i = lo + threadIdx.x; i < hi; i += kGreedyThreads) {
        const float x = __ldg(row + i);
        if (better(x, i, bv, bi)) { bv = x; bi = i; }
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) { s_v[warp] = bv; s_i[warp] = bi; }
    __syncthreads();
    const int par = step & 1;
    if (warp == 0) {
      bv = lane < kGreedyThreads / 32 ? s_v[lane] : -INFINITY;
      bi = lane < kGreedyThreads / 32 ? s_i[lane] : INT_MAX;
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) { s_res_v[par] = bv; s_res_i[par] = bi; }
    }
    cluster.sync();  // every slice result of this step is visible cluster-wide
    if (warp == 0) {
      bv = -INFINITY;
      bi = INT_MAX;
      if (lane < kGreedyCtas) {
        bv = *cluster.map_shared_rank(&s_res_v[par], lane);
        bi = *cluster.map_shared_rank(&s_res_i[par], lane);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) s_choice = bi;
    }
    __syncthreads();
    const int choice = s_choice;
    if (rank == 0) emit(o, b, k, choice, node);
    ++k;
    const int nxt = find_child(s_par, s_tok, node, n, choice, &s_best);
    if (nxt == INT_MAX) break;
    if (k == o.out_cols) {
      if (rank == 0 && threadIdx.x == 0 && o.status) atomicOr(o.status, TV_DEV_OUT_OVERFLOW);
      break;
    }
    node = nxt;
  }
  cluster.sync();  // no CTA leaves while a peer may still read its slice result
  if (rank == 0) finish_walk(o, b, k);
}

// ------------------------------------------------------------------ stochastic

__device__ __forceinline__ int64_t fix40(float x) { return __float2ll_rn(x * 1099511627776.0f); }

// floor((S * Q + 2^39) / 2^40) for S < 2^53, 0 <= Q <= 2^42, exactly.
__device__ __forceinline__ int64_t scaled_round(uint64_t S, uint64_t Q) {
  const uint64_t lo = S * Q;
  uint64_t hi = __umul64hi(S, Q);
  const uint64_t lo2 = lo + (1ull << 39);
  hi += (lo2 < lo) ? 1ull : 0ull;
  return (int64_t)((hi << 24) | (lo2 >> 40));
}

// Weight of one element at level m given the scale history S[0..m).
__device__ __forceinline__ int64_t level_weight(float p, float q, const uint64_t* S, int m) {
  int64_t w = fix40(p);
  if (m == 0) return w < 0 ? 0 : w;
  const int64_t Q = fix40(q);
  for (int j = 0; j < m; ++j) {
    const int64_t sub = (j == 0) ? Q : scaled_round(S[j], (uint64_t)(Q < 0 ? 0 : Q));
    w -= sub;
    if (w < 0) w = 0;
  }
  return w;
}

struct RowView {
  const float* p;
  const float* q;
  int V;
  int seg;    // elements per warp segment (multiple of 128 when vec)
  bool vec;
};

// Sum of the level-m weights over the calling warp's segment (all lanes get it).
__device__ uint64_t segment_total(const RowView& r, const uint64_t* S, int m, int warp, int lane) {
  const int lo = warp * r.seg;
  const int hi = min(lo + r.seg, r.V);
  uint64_t acc = 0;
  if (r.vec) {
    for (int base = lo + 4 * lane; base < hi; base += 128) {
      const float4 pv = __ldg(reinterpret_cast<const float4*>(r.p + base));
      float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m) qv = __ldg(reinterpret_cast<const float4*>(r.q + base));
      acc += (uint64_t)level_weight(pv.x, qv.x, S, m) + (uint64_t)level_weight(pv.y, qv.y, S, m) +
             (uint64_t)level_weight(pv.z, qv.z, S, m) + (uint64_t)level_weight(pv.w, qv.w, S, m);
    }
  } else {
    for (int x = lo + lane; x < hi; x += 32)
      acc += (uint64_t)level_weight(__ldg(r.p + x), m ? __ldg(r.q + x) : 0.f, S, m);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

// One pass: every warp's segment total into seg[], returns the row total.
__device__ uint64_t row_pass(const RowView& r, const uint64_t* S, int m, uint64_t* seg, uint64_t* s_total) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const uint64_t t = segment_total(r, S, m, warp, lane);
  if (lane == 0) seg[warp] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t w = 0;
    for (int i = 0; i < kWarps; ++i) w += seg[i];
    *s_total = w;
  }
  __syncthreads();
  const uint64_t w = *s_total;
  __syncthreads();
  return w;
}

// Index of the first element whose inclusive prefix sum reaches thr (V if none).
__device__ int find_crossing(const RowView& r, const uint64_t* S, int m, const uint64_t* seg, uint64_t thr,
                             int* s_idx) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  __shared__ int s_seg;
  __shared__ uint64_t s_base;
  if (threadIdx.x == 0) {
    uint64_t base = 0;
    int s = kWarps;
    for (int i = 0; i < kWarps; ++i) {
      if (base + seg[i] >= thr && seg[i] > 0) { s = i; break; }
      base += seg[i];
    }
    if (thr == 0) { s = 0; base = 0; }
    s_seg = s;
    s_base = base;
    *s_idx = r.V;
  }
  __syncthreads();
  const int s = s_seg;
  if (s < kWarps && warp == s) {
    uint64_t base = s_base;
    const int lo = s * r.seg, hi = min(lo + r.seg, r.V);
    const int per = r.vec ? 4 : 1;
    for (int cbase = lo; cbase < hi; cbase += 32 * per) {
      int64_t w[4] = {0, 0, 0, 0};
      const int x0 = cbase + lane * per;
      if (r.vec) {
        if (x0 < hi) {
          const float4 pv = __ldg(reinterpret_cast<const float4*>(r.p + x0));
          float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
          if (m) qv = __ldg(reinterpret_cast<const float4*>(r.q + x0));
          w[0] = level_weight(pv.x, qv.x, S, m);
          w[1] = level_weight(pv.y, qv.y, S, m);
          w[2] = level_weight(pv.z, qv.z, S, m);
          w[3] = level_weight(pv.w, qv.w, S, m);
        }
      } else if (x0 < hi) {
        w[0] = level_weight(__ldg(r.p + x0), m ? __ldg(r.q + x0) : 0.f, S, m);
      }
      const uint64_t mine = (uint64_t)(w[0] + w[1] + w[2] + w[3]);
      uint64_t incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint64_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const uint64_t chunk = __shfl_sync(0xffffffffu, incl, 31);
      const unsigned hit = __ballot_sync(0xffffffffu, base + incl >= thr);
      if (hit) {
        const int l = __ffs(hit) - 1;
        if (lane == l) {
          uint64_t run = base + incl - mine;
          int x = x0;
          for (int e = 0; e < per; ++e) {
            run += (uint64_t)w[e];
            if (run >= thr) { x = x0 + e; break; }
          }
          *s_idx = x;
        }
        break;
      }
      base += chunk;
    }
  }
  __syncthreads();
  const int x = *s_idx;
  __syncthreads();
  return x;
}

__global__ void __launch_bounds__(kThreads) sample_kernel(const float* __restrict__ p, const float* __restrict__ q,
                                                          const int32_t* __restrict__ tokens,
                                                          const int32_t* __restrict__ parent, int64_t pstride,
                                                          const int32_t* __restrict__ n_nodes,
                                                          const float* __restrict__ u_accept,
                                                          const float* __restrict__ u_final, int N, int V,
                                                          AcceptOut o) {
  __shared__ int32_t s_par[TV_MAX_NODES], s_tok[TV_MAX_NODES];
  __shared__ uint64_t S[TV_MAX_NODES + 1];
  __shared__ uint64_t seg_cur[kWarps], seg_tmp[kWarps];
  __shared__ uint64_t s_total;
  __shared__ int s_flag, s_idx;
  const int b = blockIdx.x;
  load_tree(parent, pstride, tokens, b, N, s_par, s_tok);
  __syncthreads();
  const int n = clamp_nodes(n_nodes, b, N);
  const bool vec = (V % 4 == 0) && (((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(q)) & 15) == 0);
  int seg = (V + kWarps - 1) / kWarps;
  if (vec) seg = (seg + 127) / 128 * 128;
  int node = 0, k = 0;
  while (true) {
    RowView row{p + ((int64_t)b * N + node) * V, q + ((int64_t)b * N + node) * V, V, seg, vec};
    int m = 0;
    uint64_t Wm = 0;     // total of the current level (valid for m >= 1)
    if (threadIdx.x == 0) S[0] = 1ull << 40;
    __syncthreads();
    int taken = -1;
    for (int c = node + 1; c < n; ++c) {
      if (s_par[c] != node) continue;
      const int x = s_tok[c];
      if (x < 0 || x >= V) {
        if (threadIdx.x == 0 && o.status) atomicOr(o.status, TV_DEV_BAD_TOKEN);
        continue;
      }
      if (threadIdx.x == 0) {
        const float px = row.p[x], qx = row.q[x];
        const double uq = __dmul_rn((double)u_accept[(int64_t)b * N + c], (double)qx);
        bool ok;
        if (m == 0) ok = uq < (double)px;
        else ok = __dmul_rn(uq, (double)Wm) < (double)level_weight(px, qx, S, m);
        s_flag = ok;
      }
      __syncthreads();
      const bool ok = s_flag;
      __syncthreads();
      if (ok) { taken = c; break; }
      // rejected: the target moves to the residual of the current level
      const uint64_t Wn = row_pass(row, S, m + 1, seg_tmp, &s_total);
      if (Wn > 0) {
        ++m;
        Wm = Wn;
        if (threadIdx.x == 0) S[m] = Wn;
        if (threadIdx.x < kWarps) seg_cur[threadIdx.x] = seg_tmp[threadIdx.x];
        __syncthreads();
      }
    }
    if (taken >= 0) {
      emit(o, b, k, s_tok[taken], node);
      ++k;
      if (k == o.out_cols) {
        if (threadIdx.x == 0 && o.status) atomicOr(o.status, TV_DEV_OUT_OVERFLOW);
        break;
      }
      node = taken;
      continue;
    }
    // replacement (after rejections) or bonus (leaf / all children absent)
    if (m == 0) Wm = row_pass(row, S, 0, seg_cur, &s_total);
    const double t = __dmul_rn((double)u_final[b], (double)Wm);
    const uint64_t thr = (uint64_t)ceil(t);
    int x = find_crossing(row, S, m, seg_cur, thr, &s_idx);
    if (x > V - 1) x = V - 1;
    emit(o, b, k, x, node);
    ++k;
    break;
  }
  finish_walk(o, b, k);
}

int check_accept_args(int B, int N, int V, const void* tokens, const void* parent, int64_t pstride,
                      const void* out, const void* n_out, int out_cols) {
  if (B < 0 || N < 1 || N > TV_MAX_NODES || V < 1 || pstride < 0 || out_cols < 1)
    return tv::fail(TV_ERR_INVALID_ARG, "tree accept: bad sizes B=%d N=%d V=%d out_cols=%d", B, N, V, out_cols);
  if (B > 0 && (!tokens || !parent || !out || !n_out))
    return tv::fail(TV_ERR_INVALID_ARG, "tree accept: null pointer");
  return TV_OK;
}

}  // namespace

extern "C" int tv_tree_accept_greedy(const float* logits, const int32_t* target_argmax, const int32_t* tokens,
                                     const int32_t* parent, int64_t parent_bstride, const int32_t* n_nodes,
                                     int32_t B, int32_t N, int32_t V, int32_t* out, int32_t* n_out, int32_t* path,
                                     int32_t out_cols, int32_t* status, void* stream) {
  tv::clear_error();
  int st = check_accept_args(B, N, V, tokens, parent, parent_bstride, out, n_out, out_cols);
  if (st) return st;
  if (B == 0) return TV_OK;
  if (!logits && !target_argmax)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_accept_greedy: need logits or target_argmax");
  AcceptOut o{out, n_out, path, out_cols, status};
  if (logits) {
    greedy_cluster_kernel<<<B * kGreedyCtas, kGreedyThreads, 0, (cudaStream_t)stream>>>(
        logits, tokens, parent, parent_bstride, n_nodes, N, V, o);
    TV_LAUNCH_CHECK("greedy_cluster_kernel");
    return TV_OK;
  }
  greedy_kernel<<<B, kThreads, 0, (cudaStream_t)stream>>>(logits, target_argmax, tokens, parent, parent_bstride,
                                                           n_nodes, N, V, o);
  TV_LAUNCH_CHECK("greedy_kernel");
  return TV_OK;
}

extern "C" int tv_tree_accept_sample(const float* p, const float* q, const int32_t* tokens, const int32_t* parent,
                                     int64_t parent_bstride, const int32_t* n_nodes, const float* u_accept,
                                     const float* u_final, int32_t B, int32_t N, int32_t V, int32_t* out,
                                     int32_t* n_out, int32_t* path, int32_t out_cols, int32_t* status,
                                     void* stream) {
  tv::clear_error();
  int st = check_accept_args(B, N, V, tokens, parent, parent_bstride, out, n_out, out_cols);
  if (st) return st;
  if (B == 0) return TV_OK;
  if (!p || !q || !u_accept || !u_final) return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_accept_sample: null pointer");
  AcceptOut o{out, n_out, path, out_cols, status};
  sample_kernel<<<B, kThreads, 0, (cudaStream_t)stream>>>(p, q, tokens, parent, parent_bstride, n_nodes, u_accept,
                                                           u_final, N, V, o);
  TV_LAUNCH_CHECK("sample_kernel");
  return TV_OK;
}
