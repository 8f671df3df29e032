// Tree acceptance on the device: one thread-block cluster per request (one
// CTA per request for target choices given directly, and for stochastic
// verification over vocabularies too large for the cluster's shared memory).
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
// The cluster sampler keeps each CTA's vocabulary slice of the current
// level's weights in shared memory; the single-CTA sampler streams the row
// and leaves the weight total of every chunk in shared memory, so its draw
// re-reads only the chunk that holds the crossing.
#include <cooperative_groups.h>

#include <climits>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "common.h"

namespace {

#ifdef TV_TC_TRACE
// Development aid: globaltimer stamps of the sampler's phases per request.
__device__ unsigned long long g_sample_t[4096][8];
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define TV_SAMPLE_T(k) do { if (threadIdx.x == 0 && blockIdx.x < 4096) g_sample_t[blockIdx.x][k] = gtimer(); } while (0)
// Cluster sampler, per request (rank 0, thread 0): start, end, passes, pass
// compute time, exchange time, node-entry time, final-draw time, nodes.
__device__ unsigned long long g_sc_t[4096][8];
#define TV_SC_DECL unsigned long long sc_tr[8] = {0, 0, 0, 0, 0, 0, 0, 0}, sc_t0 = 0
#define TV_SC_MARK() do { sc_t0 = gtimer(); } while (0)
#define TV_SC_ADD(k) do { const unsigned long long t_ = gtimer(); sc_tr[k] += t_ - sc_t0; sc_t0 = t_; } while (0)
#define TV_SC_SET(k, v) do { sc_tr[k] = (v); } while (0)
#define TV_SC_STORE(b) do { if (threadIdx.x == 0 && rank == 0 && (b) < 4096) \
    for (int i_ = 0; i_ < 8; ++i_) g_sc_t[b][i_] = sc_tr[i_]; } while (0)
#else
#define TV_SAMPLE_T(k) do { } while (0)
#define TV_SC_DECL do { } while (0)
#define TV_SC_MARK() do { } while (0)
#define TV_SC_ADD(k) do { } while (0)
#define TV_SC_SET(k, v) do { } while (0)
#define TV_SC_STORE(b) do { } while (0)
#endif

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

// Where request b's per-node inputs of the stochastic walk live.  The tree
// call keeps them at entry b * N + c (tokens, u_accept, rows of q); the
// chain call (the verifier page's verify shape: draft j is node j + 1) reads
// its own arrays in place: tokens and u of node c >= 1 at entry b * K + c - 1,
// q of node c at row b * K + c (the last node has no children, so its q row
// is never read), and num_draft[b] + 1 nodes.
struct NodeIdx {
  int64_t bs;  // entries (rows of q) between requests: N (tree) or K (chain)
  int shift;   // tokens / u of node c: entry b * bs + c - shift
  int n_add;   // request b has n_nodes[b] + n_add nodes
  __device__ __forceinline__ int64_t tu(int b, int c) const { return (int64_t)b * bs + c - shift; }
  __device__ __forceinline__ int64_t qrow(int b, int c) const { return (int64_t)b * bs + c; }
  __device__ __forceinline__ int nodes(const int32_t* n_nodes, int b, int N) const {
    if (!n_nodes) return N;
    const int n = n_nodes[b] + n_add;
    return n < 1 ? 1 : (n > N ? N : n);
  }
};

// A request's state after the grid sampler's walk (see gc_walk_kernel): its
// stop node is drawn from, its walk was truncated, or it needs another
// kernel's walk.  The other kernels take an optional state array and walk
// only the requests marked kGcOther.
enum : int { kGcDraw = 0, kGcDone = 1, kGcOther = 2 };

// The tree of request b for the stochastic walk (node 0's token is never
// used), with every node's acceptance-test inputs: p(x) and q(x) from its
// parent's rows at its token x, and its uniform (a test after rejections at
// the parent computes the residual's weight from the same p(x) and q(x)).
// They depend on the tree alone (the walk only chooses which it reads), so
// all of them are requested at once: one memory round trip for the whole
// walk instead of one per level.  Nodes whose parent does not precede them,
// or whose token is outside the vocabulary, are never tested and load
// nothing.
__device__ __forceinline__ void load_walk(const float* p, const float* q, const float* u_accept,
                                          const int32_t* parent, int64_t pstride, const int32_t* tokens,
                                          const NodeIdx& ix, int b, int N, int V, int32_t* s_par, int32_t* s_tok,
                                          float* s_tp, float* s_tq, float* s_tu) {
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    const int par = parent[(int64_t)b * pstride + c];
    const int x = c >= ix.shift ? tokens[ix.tu(b, c)] : -1;
    s_par[c] = par;
    s_tok[c] = x;
    const bool test = c >= 1 && par >= 0 && par < c && x >= 0 && x < V;
    s_tu[c] = c >= 1 && c >= ix.shift ? u_accept[ix.tu(b, c)] : 0.f;
    s_tp[c] = test ? p[((int64_t)b * N + par) * V + x] : 0.f;
    s_tq[c] = test ? q[ix.qrow(b, par) * V + x] : 0.f;
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

// Orderable key of a float (no NaN): key(a) > key(b) exactly when a > b, and
// -0 and +0 share a key, as they compare equal.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(__fadd_rn(v, 0.f));  // -0 + 0 = +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp argmax of (key, index) pairs: the largest key, the lowest index among
// equal keys (the order of `better`); every lane gets the result.
__device__ __forceinline__ void warp_argmax_key(uint32_t& key, uint32_t& idx) {
  const uint32_t km = __reduce_max_sync(0xffffffffu, key);
  idx = __reduce_min_sync(0xffffffffu, key == km ? idx : 0xffffffffu);
  key = km;
}

// One-way exchange of the slice results: each CTA stores its packed result
// into slot [rank] of every peer's shared memory with st.async, which counts
// the 8 bytes against the peer's mbarrier for that step parity; a CTA waits
// on its own mbarrier (armed for 8 results per step) instead of a cluster
// barrier.  Waits are bounded (TV_DEV_TIMEOUT).
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void gx_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(bar)) : "memory");
}
__device__ __forceinline__ void gx_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void gx_send(uint64_t* slot, uint64_t* bar, unsigned peer, uint64_t v) {
  uint32_t rs, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rs) : "r"((uint32_t)__cvta_generic_to_shared(slot)), "r"(peer));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"((uint32_t)__cvta_generic_to_shared(bar)), "r"(peer));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u64 [%0], %1, [%2];" ::"r"(rs), "l"(v), "r"(rb)
               : "memory");
}
// true once the phase of the given parity has completed; false after about 2 s
__device__ __forceinline__ bool gx_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  const uint64_t t0 = gtime();
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(a), "r"(parity)
                 : "memory");
    if (done) return true;
    if ((it & 255u) == 255u && gtime() - t0 > 2000000000ull) return false;
  }
}

__global__ void __cluster_dims__(kGreedyCtas, 1, 1) __launch_bounds__(kGreedyThreads)
    greedy_cluster_kernel(const float* __restrict__ logits, const int32_t* __restrict__ tokens,
                          const int32_t* __restrict__ parent, int64_t pstride, const int32_t* __restrict__ n_nodes,
                          int N, int V, AcceptOut o) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ int32_t s_par[TV_MAX_NODES], s_tok[TV_MAX_NODES];
  __shared__ uint32_t s_key[kGreedyThreads / 32], s_idx[kGreedyThreads / 32];
  __shared__ uint64_t s_slot[2][kGreedyCtas];  // the CTAs' packed slice results, by step parity
  __shared__ uint64_t s_bar[2];                 // their arrival, by step parity
  __shared__ int s_choice, s_next;
  const int rank = (int)cluster.block_rank();
  if (threadIdx.x == 0) {
    gx_init(&s_bar[0]);
    gx_init(&s_bar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster.sync();  // every CTA's barriers are initialised before any result is sent
  const int b = blockIdx.x / kGreedyCtas;
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
      // kBatch float4 per thread requested together, then compared; the
      // first batch of the root row goes out before the tree is loaded
      constexpr int kBatch = 4;
      const float4* r4 = reinterpret_cast<const float4*>(row) + lo / 4;
      const int n4 = (hi - lo) / 4;
      for (int base = threadIdx.x; base < n4 || (step == 0 && base == (int)threadIdx.x);
           base += kBatch * kGreedyThreads) {
        float4 x[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int t = base + u * kGreedyThreads;
          if (t < n4) x[u] = __ldg(r4 + t);
        }
        if (step == 0 && base == (int)threadIdx.x) load_tree(parent, pstride, tokens, b, N, s_par, s_tok);
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
      if (step == 0) load_tree(parent, pstride, tokens, b, N, s_par, s_tok);
      for (int i = lo + threadIdx.x; i < hi; i += kGreedyThreads) {
        const float x = __ldg(row + i);
        if (better(x, i, bv, bi)) { bv = x; bi = i; }
      }
    }
    uint32_t key = order_key(bv), idx = (uint32_t)bi;
    warp_argmax_key(key, idx);
    if (lane == 0) { s_key[warp] = key; s_idx[warp] = idx; }
    __syncthreads();  // also publishes the tree rows at step 0
    const int par = step & 1;
    if (warp == 0) {
      key = lane < kGreedyThreads / 32 ? s_key[lane] : 0u;
      idx = lane < kGreedyThreads / 32 ? s_idx[lane] : 0xffffffffu;
      warp_argmax_key(key, idx);
      // (key, ~index) packed: the largest value is the largest key, then the lowest index
      if (lane == 0) gx_expect(&s_bar[par], 8u * kGreedyCtas);
      __syncwarp();
      if (lane < kGreedyCtas)
        gx_send(&s_slot[par][rank], &s_bar[par], (unsigned)lane, ((uint64_t)key << 32) | (uint64_t)(~idx));
      const bool late = __any_sync(0xffffffffu, !gx_wait(&s_bar[par], (step >> 1) & 1));
      if (late && lane == 0 && o.status) atomicOr(o.status, TV_DEV_TIMEOUT);
      uint64_t v = lane < kGreedyCtas ? s_slot[par][lane] : 0ull;
#pragma unroll
      for (int off = 4; off; off >>= 1) {
        const uint64_t w = __shfl_xor_sync(0xffffffffu, v, off);
        v = w > v ? w : v;
      }
      v = __shfl_sync(0xffffffffu, v, 0);
      const int choice = (int)(~(uint32_t)v);
      // lowest-index valid child of `node` carrying the choice (children
      // follow their parent and N <= 64: two 32-node windows)
      int nxt = INT_MAX;
#pragma unroll
      for (int w0 = 1; w0 <= 33; w0 += 32) {
        const int c = node + w0 + lane;
        const unsigned hit = __ballot_sync(0xffffffffu, c < n && s_par[c] == node && s_tok[c] == choice);
        if (hit && nxt == INT_MAX) nxt = node + w0 + __ffs(hit) - 1;
      }
      if (lane == 0) {
        s_choice = choice;
        s_next = late ? INT_MAX : nxt;  // a peer's result never came: end the walk
      }
    }
    __syncthreads();
    const int choice = s_choice, nxt = s_next;
    if (rank == 0) emit(o, b, k, choice, node);
    ++k;
    if (nxt == INT_MAX) break;
    if (k == o.out_cols) {
      if (rank == 0 && threadIdx.x == 0 && o.status) atomicOr(o.status, TV_DEV_OUT_OVERFLOW);
      break;
    }
    node = nxt;
  }
  cluster.sync();  // no CTA leaves while a peer's result may still be on its way to it
  if (rank == 0) finish_walk(o, b, k);
}

// ------------------------------------------------------------------ stochastic

// rint(x * 2^40) as an integer using only float32 additions and integer
// arithmetic on the bit patterns: float-to-integer conversions run on the
// double-precision pipe, which is slow on this GPU and would bound the
// sampler.  With a = |x| < 8:
//   H   = floor(a * 2^20)            (a * 2^20 + 2^23 added toward zero: the
//                                     sum's low mantissa bits hold H)
//   rem = a * 2^40 - H * 2^20        in [0, 2^20), exact (fused multiply-add
//                                     of values that are multiples of ulp(a*2^40))
//   L   = rint(rem)                  (rem + 1.5 * 2^23 rounded to nearest even)
//   rint(a * 2^40) = H * 2^20 + L    since H * 2^20 is an integer.
// Rows are probability rows (no negative entries): an entry below zero is
// taken as 0, which gives it weight 0 at every level as its rint image would.
// The two parts of fix40(x): rint(max(x, 0) * 2^40) = H * 2^20 + L with
// 0 <= H, L <= 2^20 (the same arithmetic as fix40, kept in 32 bits).
__device__ __forceinline__ void fix40_parts(float x, int32_t& H, int32_t& L) {
  const float a = fmaxf(x, 0.f);
  const float y = a * 1099511627776.0f;
  float hf;
  asm("add.rz.f32 %0, %1, %2;" : "=f"(hf) : "f"(a * 1048576.0f), "f"(8388608.0f));
  const float h = hf - 8388608.0f;
  const float rem = fmaf(h, -1048576.0f, y);
  const float lt = rem + 12582912.0f;
  H = (int32_t)(__float_as_uint(hf) - 0x4B000000u);
  L = (int32_t)(__float_as_uint(lt) - 0x4B400000u);
}

__device__ __forceinline__ int64_t fix40(float x) {
  const float a = fmaxf(x, 0.f);  // probabilities; a negative entry weighs 0 like its clamped image
  const float y = a * 1099511627776.0f;
  float hf;
  asm("add.rz.f32 %0, %1, %2;" : "=f"(hf) : "f"(a * 1048576.0f), "f"(8388608.0f));
  const float h = hf - 8388608.0f;
  const float rem = fmaf(h, -1048576.0f, y);
  const float lt = rem + 12582912.0f;
  const uint32_t H = __float_as_uint(hf) - 0x4B000000u;
  const uint32_t L = __float_as_uint(lt) - 0x4B400000u;
  return (int64_t)(((uint64_t)H << 20) + L);
}

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
  const int64_t P = fix40(p);
  if (m == 0) return P;
  const int64_t Q = fix40(q);
  int64_t w = P > Q ? P - Q : 0;
  for (int j = 1; j < m; ++j) {
    const int64_t sub = scaled_round(S[j], (uint64_t)Q);
    w = w > sub ? w - sub : 0;
  }
  return w;
}

// A row is cut into chunks of ch = 128 * k consecutive elements (k chosen so
// that there are at most kMaxChunks chunks); chunk c belongs to warp
// c % kSampleWarps.
// A pass over the row leaves every chunk's weight total in shared memory, so
// the final draw finds the chunk holding the crossing with one block-wide
// prefix scan and re-reads only that chunk.
constexpr int kMaxChunks = 1024;
constexpr int kChunkBatch = 2;  // chunks a warp loads together (their loads in flight at once)
constexpr int kSampleThreads = 512;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kScanPer = kMaxChunks / kSampleThreads;  // chunk totals per thread in the prefix scan

struct RowView {
  const float* p;
  const float* q;
  int V;
  int k;      // float4 groups of 32 lanes per chunk: chunk = 128 * k elements
  int nc;     // number of chunks
  bool vec;   // rows 16-byte aligned and V % 4 == 0
};

// Elements e .. e + 3 of the row (4 * lane + 128 * i within a chunk), zero
// past the end.
__device__ __forceinline__ void load4(const RowView& r, int e, int m, float4& pv, float4& qv) {
  pv = make_float4(0.f, 0.f, 0.f, 0.f);
  qv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (e >= r.V) return;
  if (r.vec) {
    pv = __ldg(reinterpret_cast<const float4*>(r.p + e));
    if (m) qv = __ldg(reinterpret_cast<const float4*>(r.q + e));
  } else {
    pv.x = __ldg(r.p + e);
    if (e + 1 < r.V) pv.y = __ldg(r.p + e + 1);
    if (e + 2 < r.V) pv.z = __ldg(r.p + e + 2);
    if (e + 3 < r.V) pv.w = __ldg(r.p + e + 3);
    if (m) {
      qv.x = __ldg(r.q + e);
      if (e + 1 < r.V) qv.y = __ldg(r.q + e + 1);
      if (e + 2 < r.V) qv.z = __ldg(r.q + e + 2);
      if (e + 3 < r.V) qv.w = __ldg(r.q + e + 3);
    }
  }
}

// Level-m weights of elements e .. e + 3 (zero past the end of the row).
__device__ __forceinline__ void weights4(const RowView& r, int e, const float4& pv, const float4& qv,
                                         const uint64_t* S, int m, int64_t (&w)[4]) {
  w[0] = e < r.V ? level_weight(pv.x, qv.x, S, m) : 0;
  w[1] = e + 1 < r.V ? level_weight(pv.y, qv.y, S, m) : 0;
  w[2] = e + 2 < r.V ? level_weight(pv.z, qv.z, S, m) : 0;
  w[3] = e + 3 < r.V ? level_weight(pv.w, qv.w, S, m) : 0;
}

// One pass at level m: every chunk's weight total into cs[], returns the row
// total (all threads).
__device__ uint64_t row_pass(const RowView& r, const uint64_t* S, int m, uint64_t* cs, uint64_t* s_red) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  for (int c0 = warp; c0 < r.nc; c0 += kSampleWarps * kChunkBatch) {
    uint64_t sum[kChunkBatch];
#pragma unroll
    for (int j = 0; j < kChunkBatch; ++j) sum[j] = 0;
    for (int i = 0; i < r.k; ++i) {
      float4 pv[kChunkBatch], qv[kChunkBatch];
#pragma unroll
      for (int j = 0; j < kChunkBatch; ++j) {
        const int c = c0 + kSampleWarps * j;
        load4(r, c < r.nc ? c * 128 * r.k + 128 * i + 4 * lane : r.V, m, pv[j], qv[j]);
      }
#pragma unroll
      for (int j = 0; j < kChunkBatch; ++j) {
        const int c = c0 + kSampleWarps * j;
        int64_t w[4];
        weights4(r, c < r.nc ? c * 128 * r.k + 128 * i + 4 * lane : r.V, pv[j], qv[j], S, m, w);
        sum[j] += (uint64_t)(w[0] + w[1] + w[2] + w[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < kChunkBatch; ++j) {
      uint64_t v = sum[j];
#pragma unroll
      for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      const int c = c0 + kSampleWarps * j;
      if (lane == 0 && c < r.nc) cs[c] = v;
    }
  }
  __syncthreads();
  uint64_t t = 0;
  for (int c = threadIdx.x; c < r.nc; c += kSampleThreads) t += cs[c];
#pragma unroll
  for (int off = 16; off; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  if (lane == 0) s_red[warp] = t;
  __syncthreads();
  uint64_t w = 0;
#pragma unroll
  for (int i = 0; i < kSampleWarps; ++i) w += s_red[i];
  __syncthreads();
  return w;
}

// The same pass with the row streamed through a ring of shared-memory stages
// by cp.async copies, so a CTA keeps far more of the row in flight than its
// registers could hold.  Stage = kStageElems elements of p (and q), one
// 256-element chunk per warp.  Needs 16-byte aligned rows, V % 4 == 0 and
// 256-element chunks (k == 2).
constexpr int kStreamStages = 2;  // (a third stage measured no faster: the pass is issue-bound)
constexpr int kChunkElems = 256;                  // a chunk: two float4 per lane of one warp
constexpr int kStageElems = kChunkElems * kSampleWarps;  // 4096: one chunk per warp and stage
static_assert(kStageElems % (4 * kSampleThreads) == 0, "whole float4 copies per thread");

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Level 0/1 weights of four in-row elements added into (h, l), the sum being
// h * 2^20 + l: w0 = P, w1 = max(0, P - Q) with P - Q = dH * 2^20 + dL and
// |dL| <= 2^20, so P - Q > 0 iff dH > 0, or dH == 0 and dL > 0.
__device__ __forceinline__ void add_weights4(const float4& pv, const float4& qv, int m, int32_t& h, int32_t& l) {
  const float ps[4] = {pv.x, pv.y, pv.z, pv.w};
  const float qs[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int32_t Hp, Lp;
    fix40_parts(ps[i], Hp, Lp);
    if (m == 0) {
      h += Hp;
      l += Lp;
    } else {
      int32_t Hq, Lq;
      fix40_parts(qs[i], Hq, Lq);
      const int32_t dH = Hp - Hq, dL = Lp - Lq;
      const bool pos = dH > 0 || (dH == 0 && dL > 0);
      h += pos ? dH : 0;
      l += pos ? dL : 0;
    }
  }
}

__device__ uint64_t row_pass_stream(const RowView& r, const uint64_t* S, int m, uint64_t* cs, uint64_t* s_red,
                                    float4* ring) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  constexpr int kRow4 = kStageElems / 4;  // float4 per row and stage
  const int nst = (r.V + kStageElems - 1) / kStageElems;
  auto issue = [&](int st) {
    if (st < nst) {
      const int slot = st % kStreamStages;
#pragma unroll
      for (int j = 0; j < kRow4 / kSampleThreads; ++j) {
        const int i4 = j * kSampleThreads + threadIdx.x;
        const int e = st * kStageElems + 4 * i4;
        if (e < r.V) {
          cp_async16(&ring[(2 * slot) * kRow4 + i4], r.p + e);
          if (m) cp_async16(&ring[(2 * slot + 1) * kRow4 + i4], r.q + e);
        }
      }
    }
    cp_async_commit();  // an empty group past the end keeps the group count uniform
  };
#pragma unroll
  for (int st = 0; st < kStreamStages - 1; ++st) issue(st);
  for (int g = 0; g < nst; ++g) {
    issue(g + kStreamStages - 1);
    asm volatile("cp.async.wait_group %0;" ::"n"(kStreamStages - 1) : "memory");  // stage g has landed
    __syncthreads();
    const int slot = g % kStreamStages;
    const int c = g * kSampleWarps + warp;  // this warp's chunk
    uint64_t v;
    if ((g + 1) * kStageElems <= r.V && m <= 1) {  // the whole stage lies inside the row
      int32_t h = 0, l = 0;
#pragma unroll
      for (int j = 0; j < kChunkElems / 128; ++j) {
        const int i4 = warp * (kChunkElems / 4) + j * 32 + lane;
        const float4 pv = ring[(2 * slot) * kRow4 + i4];
        const float4 qv = m ? ring[(2 * slot + 1) * kRow4 + i4] : make_float4(0.f, 0.f, 0.f, 0.f);
        add_weights4(pv, qv, m, h, l);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        h += __shfl_xor_sync(0xffffffffu, h, off);
        l += __shfl_xor_sync(0xffffffffu, l, off);
      }
      v = (uint64_t)(((int64_t)h << 20) + l);
    } else {
      uint64_t acc = 0;
#pragma unroll
      for (int j = 0; j < kChunkElems / 128; ++j) {
        const int i4 = warp * (kChunkElems / 4) + j * 32 + lane;
        const int e = g * kStageElems + 4 * i4;
        const float4 pv = ring[(2 * slot) * kRow4 + i4];
        const float4 qv = m ? ring[(2 * slot + 1) * kRow4 + i4] : make_float4(0.f, 0.f, 0.f, 0.f);
        int64_t w[4];
        weights4(r, e, pv, qv, S, m, w);  // zero past the end of the row
        acc += (uint64_t)(w[0] + w[1] + w[2] + w[3]);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      v = acc;
    }
    if (lane == 0 && c < r.nc) cs[c] = v;
    __syncthreads();  // every warp is done with this slot before it is refilled
  }
  uint64_t t = 0;
  for (int c = threadIdx.x; c < r.nc; c += kSampleThreads) t += cs[c];
#pragma unroll
  for (int off = 16; off; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  if (lane == 0) s_red[warp] = t;
  __syncthreads();
  uint64_t w = 0;
#pragma unroll
  for (int i = 0; i < kSampleWarps; ++i) w += s_red[i];
  __syncthreads();
  return w;
}

// Index of the first element whose inclusive prefix sum of level-m weights
// reaches thr (V if none), from the chunk totals cs[] of the same level.
__device__ int find_crossing(const RowView& r, const uint64_t* S, int m, const uint64_t* cs, uint64_t thr,
                             uint64_t* s_red, int* s_chunk, uint64_t* s_base, int* s_idx) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  if (thr == 0) return 0;
  // block exclusive prefix over the chunk totals, kScanPer consecutive chunks per thread
  const int c_first = kScanPer * threadIdx.x;
  uint64_t v[kScanPer];
  uint64_t mine_sum = 0;
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    v[j] = c_first + j < r.nc ? cs[c_first + j] : 0;
    mine_sum += v[j];
  }
  uint64_t incl = mine_sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint64_t x = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += x;
  }
  if (lane == 31) s_red[warp] = incl;
  if (threadIdx.x == 0) {
    *s_chunk = -1;
    *s_idx = r.V;
  }
  __syncthreads();
  uint64_t ex = incl - mine_sum;
  for (int i = 0; i < warp; ++i) ex += s_red[i];
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    if (v[j] > 0 && ex < thr && thr <= ex + v[j]) { *s_chunk = c_first + j; *s_base = ex; }
    ex += v[j];
  }
  __syncthreads();
  const int c = *s_chunk;
  if (c >= 0 && warp == 0) {
    uint64_t base = *s_base;
    for (int i = 0; i < r.k; ++i) {
      const int e = c * 128 * r.k + 128 * i + 4 * lane;
      float4 pv, qv;
      load4(r, e, m, pv, qv);
      int64_t w[4];
      weights4(r, e, pv, qv, S, m, w);
      const uint64_t mine = (uint64_t)(w[0] + w[1] + w[2] + w[3]);
      uint64_t inc = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint64_t v = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += v;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, base + inc >= thr);
      if (hit) {
        const int l = __ffs(hit) - 1;
        if (lane == l) {
          uint64_t run = base + inc - mine;
          int x = e;
          for (int q4 = 0; q4 < 4; ++q4) {
            run += (uint64_t)w[q4];
            if (run >= thr) { x = e + q4; break; }
          }
          *s_idx = x;
        }
        break;
      }
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  __syncthreads();
  const int x = *s_idx;
  __syncthreads();
  return x;
}

__global__ void __launch_bounds__(kSampleThreads, 2) sample_kernel(const float* __restrict__ p, const float* __restrict__ q,
                                                          const int32_t* __restrict__ tokens,
                                                          const int32_t* __restrict__ parent, int64_t pstride,
                                                          const int32_t* __restrict__ n_nodes,
                                                          const float* __restrict__ u_accept,
                                                          const float* __restrict__ u_final, int N, int V,
                                                          NodeIdx ix, AcceptOut o, const int4* __restrict__ only) {
  if (only && only[blockIdx.x].x != kGcOther) return;  // walked by the grid sampler
  __shared__ int32_t s_par[TV_MAX_NODES], s_tok[TV_MAX_NODES];
  __shared__ float s_tp[TV_MAX_NODES], s_tq[TV_MAX_NODES], s_tu[TV_MAX_NODES];  // acceptance-test inputs by node
  __shared__ uint64_t S[TV_MAX_NODES + 1];
  __shared__ uint64_t s_red[kSampleWarps], s_base;
  extern __shared__ float4 dsm[];  // stream ring, then the chunk totals of the current level
  float4* ring = dsm;
  uint64_t* cs = reinterpret_cast<uint64_t*>(dsm + 2 * kStreamStages * (kStageElems / 4));
  __shared__ int s_flag, s_idx, s_chunk;
  const int b = blockIdx.x;
  TV_SAMPLE_T(0);
  load_walk(p, q, u_accept, parent, pstride, tokens, ix, b, N, V, s_par, s_tok, s_tp, s_tq, s_tu);
  __syncthreads();
  TV_SAMPLE_T(1);
  const int n = ix.nodes(n_nodes, b, N);
  const bool vec = (V % 4 == 0) && (((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(q)) & 15) == 0);
  const int groups = (V + 127) / 128;
  int kk = (groups + kMaxChunks - 1) / kMaxChunks;
  kk = kk < 2 ? 2 : kk;  // chunks of at least 256 elements
  const int nc = (groups + kk - 1) / kk;
  const bool stream = vec && kk == 2;
  auto pass = [&](const RowView& rv, int level, uint64_t* cs) {
    return stream ? row_pass_stream(rv, S, level, cs, s_red, ring) : row_pass(rv, S, level, cs, s_red);
  };
  int node = 0, k = 0;
  while (true) {
    RowView row{p + ((int64_t)b * N + node) * V, q + ix.qrow(b, node) * V, V, kk, nc, vec};
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
        const float px = s_tp[c], qx = s_tq[c];
        const double uq = __dmul_rn((double)s_tu[c], (double)qx);
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
      TV_SAMPLE_T(6);
      const uint64_t Wn = pass(row, m + 1, cs);
      TV_SAMPLE_T(7);
      if (Wn > 0) {
        ++m;
        Wm = Wn;
        if (threadIdx.x == 0) S[m] = Wn;
        __syncthreads();
      } else if (m >= 1) {
        pass(row, m, cs);  // the level is kept: its chunk totals again (level 0's are rebuilt at the draw)
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
    TV_SAMPLE_T(2);
    if (m == 0) Wm = pass(row, 0, cs);
    TV_SAMPLE_T(3);
    const double t = __dmul_rn((double)u_final[b], (double)Wm);
    const uint64_t thr = (uint64_t)ceil(t);
    int x = find_crossing(row, S, m, cs, thr, s_red, &s_chunk, &s_base, &s_idx);
    TV_SAMPLE_T(4);
    if (x > V - 1) x = V - 1;
    emit(o, b, k, x, node);
    ++k;
    break;
  }
  TV_SAMPLE_T(5);
  finish_walk(o, b, k);
}

// ------------------------------------------------------ stochastic, cluster

// The same walk with the vocabulary cut into kScCtas slices, one per CTA of a
// thread-block cluster.  Each CTA keeps its slice of the current level's
// weights w_m (uint64) and of q (float32) in shared memory, so a residual
// pass after the first rejection at a node reads only shared memory and costs
// O(1) per element, where the single-CTA kernel recomputes w_m from p and q
// in O(m).  Slice totals are exchanged through distributed shared memory with
// one cluster barrier per pass; every CTA takes the same accept decisions
// from the same p(x), q(x) and totals, so all CTAs of a cluster follow one
// control flow.
constexpr int kScCtas = 8;
constexpr int kScThreads = 256;
constexpr int kScWarps = kScThreads / 32;
constexpr int kScBatch = 4;                          // float4 of p (and q) a thread requests together
constexpr size_t kScMaxDyn = 200 * 1024;             // shared memory for the slice state, at most

// Slice length (elements, a multiple of 4) of a V-element row cut over csize CTAs.
inline int sc_slice(int V, int csize) { return (int)((tv::ceil_div(V, csize) + 3) / 4 * 4); }

__device__ __forceinline__ uint64_t sc_block_sum(uint64_t v, uint64_t* s_red) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  uint64_t t = 0;
#pragma unroll
  for (int i = 0; i < kScWarps; ++i) t += s_red[i];
  __syncthreads();
  return t;
}

// Level 0 (w = P) or level 1 (w = max(0, P - Q), and q kept) of the slice
// [lo, lo + len) of a row, read from global memory into shared memory.
// Returns this thread's part of the slice total.
__device__ uint64_t sc_fill(const float* __restrict__ prow, const float* __restrict__ qrow, int lo, int len,
                            bool vec, int level, uint64_t* w, float* qs) {
  uint64_t acc = 0;
  if (vec) {  // lo and len are multiples of 4, the row is 16-byte aligned
    const float4* p4 = reinterpret_cast<const float4*>(prow + lo);
    const float4* q4 = reinterpret_cast<const float4*>(qrow + lo);
    const int n4 = len / 4;
    for (int base = threadIdx.x; base < n4; base += kScBatch * kScThreads) {
      float4 pv[kScBatch], qv[kScBatch];
#pragma unroll
      for (int j = 0; j < kScBatch; ++j) {
        const int i = base + j * kScThreads;
        pv[j] = qv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n4) {
          pv[j] = __ldg(p4 + i);
          if (level) qv[j] = __ldg(q4 + i);
        }
      }
#pragma unroll
      for (int j = 0; j < kScBatch; ++j) {
        const int i = base + j * kScThreads;
        if (i >= n4) break;
        const float ps[4] = {pv[j].x, pv[j].y, pv[j].z, pv[j].w};
        const float qq[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
        uint64_t wv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int64_t P = fix40(ps[t]);
          const int64_t Q = level ? fix40(qq[t]) : 0;
          wv[t] = (uint64_t)(P > Q ? P - Q : 0);
          acc += wv[t];
        }
        reinterpret_cast<ulonglong2*>(w)[2 * i] = make_ulonglong2(wv[0], wv[1]);
        reinterpret_cast<ulonglong2*>(w)[2 * i + 1] = make_ulonglong2(wv[2], wv[3]);
        if (level) reinterpret_cast<float4*>(qs)[i] = qv[j];
      }
    }
  } else {
    for (int i = threadIdx.x; i < len; i += kScThreads) {
      const int64_t P = fix40(__ldg(prow + lo + i));
      float qx = 0.f;
      if (level) qx = __ldg(qrow + lo + i);
      const int64_t Q = level ? fix40(qx) : 0;
      const uint64_t v = (uint64_t)(P > Q ? P - Q : 0);
      w[i] = v;
      if (level) qs[i] = qx;
      acc += v;
    }
  }
  return acc;
}

// Level m -> m + 1 in place (m >= 1): w = max(0, w - floor((W_m * Q + 2^39) / 2^40)).
// With Q = H * 2^20 + L (the parts of fix40) the rounded product is
// floor((W_m * H + floor((W_m * L + 2^39) / 2^20)) / 2^20), exactly (nested
// floors of an integer plus a fraction), and both products fit in 64 bits:
// W_m <= sum P <= 2^41 for rows summing to at most 2, H <= 2^21, L <= 2^20.
// A weight that is already 0 stays 0.
__device__ uint64_t sc_residual(int len, uint64_t Wm, uint64_t* w, const float* qs) {
  uint64_t acc = 0;
#pragma unroll 4
  for (int i = threadIdx.x; i < len; i += kScThreads) {
    const uint64_t wv = w[i];
    if (wv == 0) continue;
    int32_t H, L;
    fix40_parts(qs[i], H, L);
    const uint64_t sub = (Wm * (uint64_t)H + ((Wm * (uint64_t)L + (1ull << 39)) >> 20)) >> 20;
    const uint64_t v = wv > sub ? wv - sub : 0;
    w[i] = v;
    acc += v;
  }
  return acc;
}

// Publishes this CTA's slice total in slot `rank` of every CTA's s_tot[par]
// and returns the cluster total.  s_tot is double-buffered by pass parity: a
// CTA writes buffer par again only after the next pass's barrier, which every
// CTA reaches after reading this pass's totals.
__device__ uint64_t sc_exchange(cooperative_groups::cluster_group& cl, uint64_t mine,
                                uint64_t (*s_tot)[kScCtas], int par, int rank, int nct) {
  if ((int)threadIdx.x < nct) *cl.map_shared_rank(&s_tot[par][rank], (unsigned)threadIdx.x) = mine;
  cl.sync();
  uint64_t t = 0;
  for (int r = 0; r < nct; ++r) t += s_tot[par][r];
  return t;
}

// The stateless variant's pass at a level: the CTA's slice [lo, lo + len) in
// 256-element chunks read from global memory (two chunks per warp in
// flight), each chunk's weight total into cs[] for the draw; returns this
// thread's part of the slice total.  Levels 0 and 1 sum the fixed-point
// images in 32-bit parts (add_weights4); deeper levels recompute each weight
// from p and q (level_weight), O(level) per element.
constexpr int kScChunk = 256;
constexpr int kScMaxChunks = 2 * kScThreads;  // chunk totals one block scan covers (find_crossing)

__device__ uint64_t sc_stream(const float* __restrict__ prow, const float* __restrict__ qrow, int lo, int len,
                              bool vec, int level, const uint64_t* S, uint64_t* cs, int nch) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const RowView r{prow + lo, qrow + lo, len, kScChunk / 128, nch, vec};
  for (int c0 = warp; c0 < nch; c0 += 2 * kScWarps) {
    float4 pv[2][2], qv[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = c0 + j * kScWarps;
        load4(r, c < nch ? c * kScChunk + 128 * h + 4 * lane : len, level, pv[j][h], qv[j][h]);
      }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = c0 + j * kScWarps;
      uint64_t v;
      if (level <= 1) {
        int32_t hh = 0, ll = 0;
        add_weights4(pv[j][0], qv[j][0], level, hh, ll);
        add_weights4(pv[j][1], qv[j][1], level, hh, ll);
#pragma unroll
        for (int off = 16; off; off >>= 1) {
          hh += __shfl_xor_sync(0xffffffffu, hh, off);
          ll += __shfl_xor_sync(0xffffffffu, ll, off);
        }
        v = (uint64_t)(((int64_t)hh << 20) + ll);
      } else {
        uint64_t acc = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          int64_t wv[4];
          weights4(r, c < nch ? c * kScChunk + 128 * h + 4 * lane : len, pv[j][h], qv[j][h], S, level, wv);
          acc += (uint64_t)(wv[0] + wv[1] + wv[2] + wv[3]);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        v = acc;
      }
      if (lane == 0 && c < nch) cs[c] = v;
    }
  }
  __syncthreads();
  uint64_t t = 0;
  for (int c = threadIdx.x; c < nch; c += kScThreads) t += cs[c];
  return t;
}

// kState: the slice's weights and q kept in shared memory (one pass from
// global memory per node, later levels from shared memory); otherwise every
// pass streams the slice from global memory and only chunk totals are kept
// (a small footprint, so many requests are resident at once).  The cluster
// size (1 to 8) is a launch parameter.
template <bool kState>
__global__ void __launch_bounds__(kScThreads, 4)
    sample_cluster_kernel(const float* __restrict__ p, const float* __restrict__ q,
                          const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent, int64_t pstride,
                          const int32_t* __restrict__ n_nodes, const float* __restrict__ u_accept,
                          const float* __restrict__ u_final, int N, int V, int Ls, NodeIdx ix, AcceptOut o,
                          const int4* __restrict__ only) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  // walked by the grid sampler: the whole cluster returns before its first barrier
  if (only && only[blockIdx.x / cl.num_blocks()].x != kGcOther) return;
  __shared__ int32_t s_par[TV_MAX_NODES], s_tok[TV_MAX_NODES];
  __shared__ uint64_t S[TV_MAX_NODES + 1];
  __shared__ uint64_t s_tot[2][kScCtas];
  __shared__ uint64_t s_lev[kScCtas];  // slice totals of the current level
  __shared__ uint64_t s_red[kScWarps];
  __shared__ int s_kid[TV_MAX_NODES];  // the current node's children in index order
  __shared__ float s_tp[TV_MAX_NODES], s_tq[TV_MAX_NODES], s_tu[TV_MAX_NODES];  // acceptance-test inputs by node
  __shared__ int s_nk, s_x, s_flag, s_chunk, s_idx;
  __shared__ uint64_t s_thr, s_base;
  extern __shared__ __align__(16) uint64_t sc_dyn[];
  uint64_t* w = sc_dyn;                                // kState: level weights of the slice
  float* qs = reinterpret_cast<float*>(sc_dyn + Ls);   // kState: q of the slice
  uint64_t* cs = sc_dyn;                               // otherwise: chunk totals
  const int rank = (int)cl.block_rank();
  const int nct = (int)cl.num_blocks();
  const int b = blockIdx.x / nct;
  load_walk(p, q, u_accept, parent, pstride, tokens, ix, b, N, V, s_par, s_tok, s_tp, s_tq, s_tu);
  if (threadIdx.x == 0) s_x = V - 1;  // read by rank 0 after the draw's barrier
  __syncthreads();
  const int n = ix.nodes(n_nodes, b, N);
  const int lo = min(rank * Ls, V), len = min(V - lo, Ls);
  const int nch = (len + kScChunk - 1) / kScChunk;
  const bool vec = (V % 4 == 0) && (((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(q)) & 15) == 0);
  int node = 0, k = 0, pass = 0;
  TV_SC_DECL;
  TV_SC_MARK();
  TV_SC_SET(0, sc_t0);
  while (true) {
    const float* prow = p + ((int64_t)b * N + node) * V;
    const float* qrow = q + ix.qrow(b, node) * V;
    int m = 0;
    uint64_t Wm = 0;  // total of the current level (valid for m >= 1)
    TV_SC_MARK();
    TV_SC_SET(7, sc_tr[7] + 1);
    if (threadIdx.x == 0) S[0] = 1ull << 40;
    if (threadIdx.x < 32) {
      // list the node's children in index order
      const int lane = threadIdx.x;
      int cnt = 0;
      for (int base = node + 1; base < n; base += 32) {
        const int c = base + lane;
        const bool is = c < n && s_par[c] == node;
        const unsigned bal = __ballot_sync(0xffffffffu, is);
        if (is) s_kid[cnt + __popc(bal & ((1u << lane) - 1u))] = c;
        cnt += __popc(bal);
      }
      if (lane == 0) s_nk = cnt;
    }
    __syncthreads();
    TV_SC_ADD(5);
    const int nk = s_nk;
    int taken = -1;
    for (int j = 0; j < nk; ++j) {
      const int c = s_kid[j], x = s_tok[c];
      if (x < 0 || x >= V) {
        if (rank == 0 && threadIdx.x == 0 && o.status) atomicOr(o.status, TV_DEV_BAD_TOKEN);
        continue;
      }
      // one thread decides (double precision is slow here) and shares it;
      // the pass after a rejection synchronises before s_flag is written again
      if (threadIdx.x == 0) {
        const float px = s_tp[c], qx = s_tq[c];
        const double uq = __dmul_rn((double)s_tu[c], (double)qx);
        s_flag = m == 0 ? uq < (double)px : __dmul_rn(uq, (double)Wm) < (double)level_weight(px, qx, S, m);
      }
      __syncthreads();
      if (s_flag) { taken = c; break; }
      // rejected: the target moves to the residual of the current level
      TV_SC_MARK();
      uint64_t part;
      if constexpr (kState) part = m == 0 ? sc_fill(prow, qrow, lo, len, vec, 1, w, qs) : sc_residual(len, Wm, w, qs);
      else part = sc_stream(prow, qrow, lo, len, vec, m + 1, S, cs, nch);
      TV_SC_ADD(3);
      const uint64_t Wn = sc_exchange(cl, sc_block_sum(part, s_red), s_tot, pass & 1, rank, nct);
      TV_SC_ADD(4);
      ++pass;
      if (Wn > 0) {
        ++m;
        Wm = Wn;
        if (threadIdx.x == 0) S[m] = Wn;
        if (threadIdx.x < nct) s_lev[threadIdx.x] = s_tot[(pass - 1) & 1][threadIdx.x];
      } else if (m >= 1) {
        // the level is kept: rebuild what the pass overwrote
        if constexpr (kState) {
          for (int i = threadIdx.x; i < len; i += kScThreads)
            w[i] = (uint64_t)level_weight(__ldg(prow + lo + i), __ldg(qrow + lo + i), S, m);
        } else {
          sc_stream(prow, qrow, lo, len, vec, m, S, cs, nch);
        }
      }
      __syncthreads();
    }
    if (taken >= 0) {
      if (rank == 0) emit(o, b, k, s_tok[taken], node);
      ++k;
      if (k == o.out_cols) {
        if (rank == 0 && threadIdx.x == 0 && o.status) atomicOr(o.status, TV_DEV_OUT_OVERFLOW);
        break;
      }
      node = taken;
      continue;
    }
    // replacement (after rejections) or bonus (leaf / all children absent)
    TV_SC_MARK();
    if (m == 0) {
      uint64_t part;
      if constexpr (kState) part = sc_fill(prow, qrow, lo, len, vec, 0, w, qs);
      else part = sc_stream(prow, qrow, lo, len, vec, 0, S, cs, nch);
      Wm = sc_exchange(cl, sc_block_sum(part, s_red), s_tot, pass & 1, rank, nct);
      if (threadIdx.x < nct) s_lev[threadIdx.x] = s_tot[pass & 1][threadIdx.x];
      ++pass;
      __syncthreads();
    }
    if (threadIdx.x == 0) s_thr = (uint64_t)ceil(__dmul_rn((double)u_final[b], (double)Wm));
    __syncthreads();
    const uint64_t thr = s_thr;
    uint64_t E = 0;  // weight of the slices before this one
    for (int r = 0; r < rank; ++r) E += s_lev[r];
    const uint64_t T = s_lev[rank];
    if (thr == 0) {
      if (rank == 0 && threadIdx.x == 0) s_x = 0;
    } else if (!kState && T > 0 && E < thr && thr <= E + T) {
      // the crossing lies in this slice: find its chunk from the totals, then
      // the element, re-reading that chunk
      const RowView r{prow + lo, qrow + lo, len, kScChunk / 128, nch, vec};
      const int x = find_crossing(r, S, m, cs, thr - E, s_red, &s_chunk, &s_base, &s_idx);
      if (threadIdx.x == 0 && x < len) *cl.map_shared_rank(&s_x, 0u) = lo + x;
    } else if (kState && T > 0 && E < thr && thr <= E + T) {
      // the crossing lies in this slice: block scan over contiguous segments
      const uint64_t t = thr - E;
      const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
      const int seg = (len + kScThreads - 1) / kScThreads;
      const int a = min((int)threadIdx.x * seg, len), e = min(a + seg, len);
      uint64_t mine = 0;
      for (int i = a; i < e; ++i) mine += w[i];
      uint64_t incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint64_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      if (lane == 31) s_red[warp] = incl;
      __syncthreads();
      uint64_t ex = incl - mine;
      for (int i = 0; i < warp; ++i) ex += s_red[i];
      if (mine > 0 && ex < t && t <= ex + mine) {
        uint64_t run = ex;
        for (int i = a; i < e; ++i) {
          run += w[i];
          if (run >= t) {
            *cl.map_shared_rank(&s_x, 0u) = lo + i;
            break;
          }
        }
      }
    }
    cl.sync();  // the crossing is in rank 0's s_x
    TV_SC_ADD(6);
    if (rank == 0) {
      int x = s_x;
      if (x > V - 1) x = V - 1;
      emit(o, b, k, x, node);
    }
    ++k;
    break;
  }
  cl.sync();  // no CTA leaves while a peer may still write to its shared memory
  if (rank == 0) finish_walk(o, b, k);
  TV_SC_SET(2, pass);
  TV_SC_MARK();
  TV_SC_SET(1, sc_t0);
  TV_SC_STORE(b);
}

// ------------------------------------------------------- stochastic, grid

// The walk as three kernels over a caller's workspace, for large batches:
// (1) one warp per request walks from the root with the gathered test inputs
// (as load_walk does) until its first rejection or a leaf; (2) the pass that
// the stop node needs -- the residual max(0, P - Q) after a rejection, or P
// for a bonus -- runs over uniform (request, 4096-element chunk) items spread
// over the whole GPU, each leaving its chunk's level-0 and level-1 totals;
// (3) one CTA per request draws from those totals, re-reading the one chunk
// that holds the crossing.  (Drawing in the pass kernel, by the last item of
// a request to finish, measured slower: the last requests' draws then run
// one after another at the end of the pass.)  The same arithmetic as the
// other kernels, so the results match them bit for bit.  A request whose rejected child has a later valid sibling
// needs the next level's total before that sibling's test: the walk marks
// it, and one of the other kernels walks it again (every other request
// returns at once there).
constexpr int kGcChunk = 4096;                     // elements of one pass item
constexpr int kGcThreads = 256;                    // = kScThreads: sc_block_sum serves these kernels too
constexpr int kGcPer = kGcChunk / kGcThreads;      // 16 elements per thread
constexpr int kGcMaxChunks = kGcThreads;           // chunk totals one draw CTA scans (V <= 2^20)
constexpr int kGcWalkWarps = kGcThreads / 32;      // requests per walk CTA
static_assert(kGcThreads == kScThreads, "sc_block_sum");

// per request: {state, stop node, level of the draw (0 bonus, 1 residual), tokens emitted}
struct GcWs {
  int4* state;     // [B]
  uint64_t* tot;   // [B][nch][2]: level-1 and level-0 totals of each chunk
  int nch;
};

__global__ void __launch_bounds__(kGcThreads) gc_walk_kernel(const float* __restrict__ p, const float* __restrict__ q,
                                                            const int32_t* __restrict__ tokens,
                                                            const int32_t* __restrict__ parent, int64_t pstride,
                                                            const int32_t* __restrict__ n_nodes,
                                                            const float* __restrict__ u_accept, int B, int N, int V,
                                                            NodeIdx ix, AcceptOut o, GcWs ws) {
  const int lane = threadIdx.x % 32;
  const int b = blockIdx.x * kGcWalkWarps + threadIdx.x / 32;
  if (b >= B) return;
  const int n = ix.nodes(n_nodes, b, N);
  // nodes lane and lane + 32: parent, token and the test's p(x), q(x), u
  int par[2], tok[2];
  float tp[2], tq[2], tu[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = lane + 32 * h;
    par[h] = -1;
    tok[h] = -1;
    tp[h] = tq[h] = tu[h] = 0.f;
    if (c < N) {
      par[h] = parent[(int64_t)b * pstride + c];
      tok[h] = c >= ix.shift ? tokens[ix.tu(b, c)] : -1;
      if (c >= 1 && c >= ix.shift) tu[h] = u_accept[ix.tu(b, c)];
      if (c >= 1 && par[h] >= 0 && par[h] < c && tok[h] >= 0 && tok[h] < V) {
        tp[h] = p[((int64_t)b * N + par[h]) * V + tok[h]];
        tq[h] = q[ix.qrow(b, par[h]) * V + tok[h]];
      }
    }
  }
  int node = 0, k = 0, state = kGcDraw, level = 0;
  while (true) {
    // the node's children in index order, as bit masks over the two windows
    unsigned kids[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = lane + 32 * h;
      kids[h] = __ballot_sync(0xffffffffu, c > node && c < n && par[h] == node);
    }
    int taken = -1;
    bool rejected = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      unsigned m = kids[h];
      const int tk = h ? tok[1] : tok[0];
      const float pk = h ? tp[1] : tp[0], qk = h ? tq[1] : tq[0], uk = h ? tu[1] : tu[0];
      while (m && taken < 0 && state == kGcDraw) {
        const int l = __ffs(m) - 1;
        m &= m - 1;
        const int x = __shfl_sync(0xffffffffu, tk, l);
        const float px = __shfl_sync(0xffffffffu, pk, l), qx = __shfl_sync(0xffffffffu, qk, l);
        const float u = __shfl_sync(0xffffffffu, uk, l);
        if (x < 0 || x >= V) {
          if (lane == 0 && o.status) atomicOr(o.status, TV_DEV_BAD_TOKEN);
          continue;
        }
        if (rejected) {
          state = kGcOther;  // a later sibling is tested at the next level: another kernel's walk
        } else if (__dmul_rn((double)u, (double)qx) < (double)px) {
          taken = l + 32 * h;
          if (lane == 0) {
            o.out[(int64_t)b * o.out_cols + k] = x;
            if (o.path) o.path[(int64_t)b * o.out_cols + k] = node;
          }
        } else {
          rejected = true;
        }
      }
    }
    if (state != kGcDraw) break;
    if (taken >= 0) {
      ++k;
      if (k == o.out_cols) {
        if (lane == 0 && o.status) atomicOr(o.status, TV_DEV_OUT_OVERFLOW);
        state = kGcDone;
        break;
      }
      node = taken;
      continue;
    }
    level = rejected ? 1 : 0;  // the residual after the rejection, else a bonus from p
    break;
  }
  if (lane == 0) ws.state[b] = make_int4(state, node, level, k);
  if (state == kGcDone) {  // truncated: no draw
    for (int j = k + lane; j < o.out_cols; j += 32) {
      o.out[(int64_t)b * o.out_cols + j] = -1;
      if (o.path) o.path[(int64_t)b * o.out_cols + j] = -1;
    }
    if (lane == 0) o.n_out[b] = k;
  }
}

// The draw of request b after its pass: level 1 when W_1 > 0 after a
// rejection, else level 0; the crossing's chunk from an exclusive scan of
// the chunk totals, then its element from a scan of that chunk re-read
// (thread t: 16 consecutive elements; the one thread holding the crossing
// reads its elements again to find it).
__device__ void gc_draw(const float* __restrict__ p, const float* __restrict__ q, const float* __restrict__ u_final,
                        int N, int V, const NodeIdx& ix, const AcceptOut& o, const GcWs& ws, int b, int4 st,
                        uint64_t* s_red, int* s_chunk, int* s_x, uint64_t* s_base) {
  const int node = st.y, k = st.w;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int t = threadIdx.x;
  const uint64_t* tot = ws.tot + (int64_t)b * ws.nch * 2;
  uint64_t v1 = t < ws.nch ? tot[2 * t] : 0, v0 = t < ws.nch ? tot[2 * t + 1] : 0;
  const uint64_t W1 = sc_block_sum(v1, s_red);
  const int m = st.z == 1 && W1 > 0 ? 1 : 0;
  const uint64_t v = m ? v1 : v0;
  const uint64_t W = m ? W1 : sc_block_sum(v0, s_red);
  const uint64_t thr = (uint64_t)ceil(__dmul_rn((double)u_final[b], (double)W));
  if (t == 0) {
    *s_chunk = -1;
    *s_x = thr == 0 ? 0 : V - 1;
  }
  // exclusive scan of the chosen totals over the chunks (thread t: chunk t)
  uint64_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) s_red[warp] = incl;
  __syncthreads();
  uint64_t ex = incl - v;
  for (int i = 0; i < warp; ++i) ex += s_red[i];
  if (thr > 0 && v > 0 && ex < thr && thr <= ex + v) {
    *s_chunk = t;
    *s_base = ex;
  }
  __syncthreads();
  const int cc = *s_chunk;
  if (cc >= 0) {
    const float* prow = p + ((int64_t)b * N + node) * V;
    const float* qrow = q + ix.qrow(b, node) * V;
    const int e0 = cc * kGcChunk + kGcPer * t;
    // level-m weight of element e (0 past the end of the row)
    auto weight = [&](int e) -> uint64_t {
      if (e >= V) return 0;
      const int64_t P = fix40(__ldg(prow + e));
      if (m == 0) return (uint64_t)P;
      const int64_t Q = fix40(__ldg(qrow + e));
      return P > Q ? (uint64_t)(P - Q) : 0;
    };
    uint64_t mine = 0;
#pragma unroll
    for (int j = 0; j < kGcPer; ++j) mine += weight(e0 + j);
    uint64_t inc = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    __syncthreads();  // s_red's chunk-scan values are no longer read
    if (lane == 31) s_red[warp] = inc;
    __syncthreads();
    uint64_t run = *s_base + inc - mine;
    for (int i = 0; i < warp; ++i) run += s_red[i];
    if (mine > 0 && run < thr && thr <= run + mine) {
      for (int j = 0; j < kGcPer; ++j) {  // the one thread holding the crossing re-reads its elements
        run += weight(e0 + j);
        if (run >= thr) {
          *s_x = e0 + j;
          break;
        }
      }
    }
  }
  __syncthreads();
  if (t == 0) {
    int x = *s_x;
    if (x > V - 1) x = V - 1;
    o.out[(int64_t)b * o.out_cols + k] = x;
    if (o.path) o.path[(int64_t)b * o.out_cols + k] = node;
  }
  finish_walk(o, b, k + 1);
}

// One pass item: chunk c of request b's stop-node row at its level; the
// chunk's level-1 total (w_1 = max(0, P - Q), summed only after a rejection)
// and level-0 total (P: the bonus, or the draw's row when W_1 = 0).
__global__ void __launch_bounds__(kGcThreads) gc_pass_kernel(const float* __restrict__ p, const float* __restrict__ q,
                                                            int N, int V, NodeIdx ix, GcWs ws) {
  __shared__ uint64_t s_red[kScWarps];
  const int b = blockIdx.x / ws.nch, c = blockIdx.x % ws.nch;
  const int4 st = ws.state[b];
  if (st.x != kGcDraw) return;
  const int node = st.y, level = st.z;
  const float* prow = p + ((int64_t)b * N + node) * V;
  const float* qrow = q + ix.qrow(b, node) * V;
  const bool vec = (V % 4 == 0) && (((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(q)) & 15) == 0);
  const int e0 = c * kGcChunk;
  float pv[kGcPer], qv[kGcPer];
  if (vec) {
    // float4 j of the thread: elements e0 + 4 (j * kGcThreads + t) .. + 3
#pragma unroll
    for (int j = 0; j < kGcPer / 4; ++j) {
      const int e = e0 + 4 * (j * kGcThreads + (int)threadIdx.x);
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), d = a;
      if (e < V) {
        a = __ldg(reinterpret_cast<const float4*>(prow + e));
        if (level) d = __ldg(reinterpret_cast<const float4*>(qrow + e));
      }
      pv[4 * j] = a.x; pv[4 * j + 1] = a.y; pv[4 * j + 2] = a.z; pv[4 * j + 3] = a.w;
      qv[4 * j] = d.x; qv[4 * j + 1] = d.y; qv[4 * j + 2] = d.z; qv[4 * j + 3] = d.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kGcPer; ++j) {
      const int e = e0 + j * kGcThreads + (int)threadIdx.x;
      pv[j] = e < V ? __ldg(prow + e) : 0.f;
      qv[j] = e < V && level ? __ldg(qrow + e) : 0.f;
    }
  }
  // sums as h * 2^20 + l in 32-bit parts (16 elements of at most 2 each: no overflow)
  int32_t h0 = 0, l0 = 0, h1 = 0, l1 = 0;
#pragma unroll
  for (int j = 0; j < kGcPer; ++j) {
    int32_t Hp, Lp;
    fix40_parts(pv[j], Hp, Lp);
    h0 += Hp;
    l0 += Lp;
    if (level) {
      int32_t Hq, Lq;
      fix40_parts(qv[j], Hq, Lq);
      const int32_t dH = Hp - Hq, dL = Lp - Lq;
      const bool pos = dH > 0 || (dH == 0 && dL > 0);
      h1 += pos ? dH : 0;
      l1 += pos ? dL : 0;
    }
  }
  const uint64_t t1 = sc_block_sum((uint64_t)(((int64_t)h1 << 20) + l1), s_red);
  const uint64_t t0 = sc_block_sum((uint64_t)(((int64_t)h0 << 20) + l0), s_red);
  if (threadIdx.x == 0) {
    uint64_t* t = ws.tot + ((int64_t)b * ws.nch + c) * 2;
    t[0] = t1;
    t[1] = t0;
  }
}

// One CTA per request: the draw of a request whose walk stopped.
__global__ void __launch_bounds__(kGcThreads) gc_draw_kernel(const float* __restrict__ p, const float* __restrict__ q,
                                                            const float* __restrict__ u_final, int N, int V,
                                                            NodeIdx ix, AcceptOut o, GcWs ws) {
  __shared__ uint64_t s_red[kScWarps];
  __shared__ int s_chunk, s_x;
  __shared__ uint64_t s_base;
  const int4 st = ws.state[blockIdx.x];
  if (st.x != kGcDraw) return;
  gc_draw(p, q, u_final, N, V, ix, o, ws, blockIdx.x, st, s_red, &s_chunk, &s_x, &s_base);
}


// Clusters of a sampler kernel resident on the current device at once for a
// launch configuration (cached per device, kernel, cluster size and shared
// memory).  Also raises the kernel's dynamic shared-memory limit.
template <bool kState>
int sc_capacity(const cudaLaunchConfig_t& cfg, int* out) {
  static std::mutex mu;
  static std::map<std::tuple<int, size_t, unsigned>, int> cache;
  int dev = 0;
  TV_CUDA_TRY(cudaGetDevice(&dev));
  const unsigned csize = cfg.attrs[0].val.clusterDim.x;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(dev, cfg.dynamicSmemBytes, csize);
  const auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return TV_OK;
  }
  TV_CUDA_TRY(cudaFuncSetAttribute(sample_cluster_kernel<kState>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kScMaxDyn));
  cudaLaunchConfig_t c = cfg;
  c.gridDim = dim3(csize);
  int n = 0;
  TV_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, sample_cluster_kernel<kState>, &c));
  cache[key] = n;
  *out = n;
  return TV_OK;
}

struct ScLaunch {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  ScLaunch(int csize, size_t dyn, void* stream) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kScThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = (cudaStream_t)stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

int check_accept_args(int B, int N, int V, const void* tokens, const void* parent, int64_t pstride,
                      const void* out, const void* n_out, int out_cols) {
  if (B < 0 || N < 1 || N > TV_MAX_NODES || V < 1 || pstride < 0 || out_cols < 1)
    return tv::fail(TV_ERR_INVALID_ARG, "tree accept: bad sizes B=%d N=%d V=%d out_cols=%d", B, N, V, out_cols);
  if (B > 0 && (!tokens || !parent || !out || !n_out))
    return tv::fail(TV_ERR_INVALID_ARG, "tree accept: null pointer");
  return TV_OK;
}

}  // namespace

#ifdef TV_TC_TRACE
extern "C" int tv_debug_sc_times(void* dst, size_t bytes) {
  const size_t n = sizeof(g_sc_t) < bytes ? sizeof(g_sc_t) : bytes;
  return cudaMemcpyFromSymbol(dst, g_sc_t, n) == cudaSuccess ? 0 : -1;
}
extern "C" int tv_debug_sample_times(void* dst, size_t bytes) {
  const size_t n = sizeof(g_sample_t) < bytes ? sizeof(g_sample_t) : bytes;
  return cudaMemcpyFromSymbol(dst, g_sample_t, n) == cudaSuccess ? 0 : -1;
}
#endif

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

namespace {

// Parent array of a chain (node c's parent is c - 1), shared by every request
// of the chain call (parent batch stride 0).
struct ChainParent {
  int32_t v[TV_MAX_NODES];
};
constexpr ChainParent make_chain_parent() {
  ChainParent c{};
  for (int i = 0; i < TV_MAX_NODES; ++i) c.v[i] = i - 1;
  return c;
}
__device__ const ChainParent g_chain_parent = make_chain_parent();

// Kernel choice and launch of the single-launch walks; `only` (nullable):
// the grid sampler's request states, of which only kGcOther requests are
// walked.
int launch_walk(const float* p, const float* q, const int32_t* tokens, const int32_t* parent,
                int64_t parent_bstride, const int32_t* n_nodes, const float* u_accept, const float* u_final,
                int32_t B, int32_t N, int32_t V, NodeIdx ix, AcceptOut o, int32_t flags, const int4* only,
                void* stream) {
  int st = TV_OK;
  if (B > INT_MAX / kScCtas && flags != TV_SAMPLE_SINGLE_CTA)
    return tv::fail(TV_ERR_INVALID_ARG, "tree accept sample: B=%d too large", B);
  // 1. one 8-CTA cluster per request keeping the level weights on chip, when
  //    every request's cluster is resident at once (or when asked for)
  const int Ls8 = sc_slice(V, kScCtas);
  const size_t dyn_state = (size_t)Ls8 * (sizeof(uint64_t) + sizeof(float));
  if ((flags == TV_SAMPLE_AUTO || flags == TV_SAMPLE_CLUSTER) && dyn_state <= kScMaxDyn) {
    ScLaunch L(kScCtas, dyn_state, stream);
    int capacity = 0;
    st = sc_capacity<true>(L.cfg, &capacity);
    if (st) return st;
    if (flags == TV_SAMPLE_CLUSTER || B <= capacity) {
      L.cfg.gridDim = dim3((unsigned)(B * kScCtas));
      cudaError_t e = cudaLaunchKernelEx(&L.cfg, sample_cluster_kernel<true>, p, q, tokens, parent, parent_bstride,
                                         n_nodes, u_accept, u_final, (int)N, (int)V, Ls8, ix, o, only);
      if (e != cudaSuccess) return tv::cuda_fail(e, "sample_cluster_kernel<state>");
      return TV_OK;
    }
  } else if (flags == TV_SAMPLE_CLUSTER) {
    return tv::fail(TV_ERR_UNSUPPORTED, "tree accept sample: the cluster kernel needs V <= %d (V=%d)",
                    kScCtas * (int)(kScMaxDyn / 12 / 4 * 4), V);
  }
  // 2. streaming clusters: the largest cluster (8, 4, 2 or 1 CTAs) with which
  //    all B requests are resident at once, each slice within one block scan
  //    of chunk totals
  if (flags == TV_SAMPLE_AUTO || flags == TV_SAMPLE_STREAM) {
    const size_t dyn = sizeof(uint64_t) * kScMaxChunks;
    int pick = 0;
    for (int csize = kScCtas; csize >= 1; csize /= 2) {
      if ((int64_t)sc_slice(V, csize) > (int64_t)kScMaxChunks * kScChunk) break;  // slice too long
      ScLaunch L(csize, dyn, stream);
      int capacity = 0;
      st = sc_capacity<false>(L.cfg, &capacity);
      if (st) return st;
      pick = csize;
      if (B <= capacity) break;
    }
    if (pick > 0) {
      ScLaunch L(pick, dyn, stream);
      L.cfg.gridDim = dim3((unsigned)(B * pick));
      cudaError_t e = cudaLaunchKernelEx(&L.cfg, sample_cluster_kernel<false>, p, q, tokens, parent, parent_bstride,
                                         n_nodes, u_accept, u_final, (int)N, (int)V, sc_slice(V, pick), ix, o,
                                         only);
      if (e != cudaSuccess) return tv::cuda_fail(e, "sample_cluster_kernel<stream>");
      return TV_OK;
    }
    if (flags == TV_SAMPLE_STREAM)
      return tv::fail(TV_ERR_UNSUPPORTED, "tree accept sample: V=%d too large for the streaming clusters", V);
  }
  // one CTA per request, rows streamed and w_m recomputed per pass
  constexpr size_t kDyn = sizeof(float4) * 2 * kStreamStages * (kStageElems / 4) + sizeof(uint64_t) * kMaxChunks;
  static_assert(2 * (kDyn + 2048 + 1024) <= 228 * 1024, "two CTAs per SM");
  cudaError_t e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDyn);
  if (e != cudaSuccess) return tv::cuda_fail(e, "cudaFuncSetAttribute(sample_kernel)");
  sample_kernel<<<B, kSampleThreads, kDyn, (cudaStream_t)stream>>>(p, q, tokens, parent, parent_bstride, n_nodes,
                                                                   u_accept, u_final, N, V, ix, o, only);
  TV_LAUNCH_CHECK("sample_kernel");
  return TV_OK;
}

// Chunks of a row in the grid sampler, and its workspace: request states
// (16 bytes each), then two totals per (request, chunk).
int gc_chunks(int V) { return (V + kGcChunk - 1) / kGcChunk; }
size_t gc_workspace_bytes(int64_t B, int V) { return (size_t)B * 16u * (1u + (size_t)gc_chunks(V)); }

// Whether a call takes the grid sampler: when asked for, or under
// TV_SAMPLE_AUTO when the workspace is large enough and the on-chip-state
// cluster kernel cannot hold every request at once.
int takes_grid(int B, int V, int flags, bool ws_ok, void* stream, bool* grid) {
  *grid = flags == TV_SAMPLE_GRID;
  if (flags == TV_SAMPLE_AUTO && ws_ok && gc_chunks(V) <= kGcMaxChunks) {
    const size_t dyn_state = (size_t)sc_slice(V, kScCtas) * (sizeof(uint64_t) + sizeof(float));
    *grid = dyn_state > kScMaxDyn;
    if (!*grid) {
      ScLaunch L(kScCtas, dyn_state, stream);
      int capacity = 0;
      const int st = sc_capacity<true>(L.cfg, &capacity);
      if (st) return st;
      *grid = B > capacity;
    }
  }
  return TV_OK;
}

// The stochastic walk, both entry points: the grid sampler (three kernels,
// then the single-launch walk of the requests it leaves) when asked for, or
// under TV_SAMPLE_AUTO when a workspace is given and the cluster kernel
// cannot hold every request at once; else one single-launch walk.
int launch_sample(const float* p, const float* q, const int32_t* tokens, const int32_t* parent,
                  int64_t parent_bstride, const int32_t* n_nodes, const float* u_accept, const float* u_final,
                  int32_t B, int32_t N, int32_t V, NodeIdx ix, AcceptOut o, int32_t flags, void* workspace,
                  size_t workspace_bytes, void* stream) {
  const bool ws_ok = workspace != nullptr && workspace_bytes >= gc_workspace_bytes(B, V) &&
                     (int64_t)B * gc_chunks(V) <= INT_MAX;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 15))
    return tv::fail(TV_ERR_INVALID_ARG, "tree accept sample: workspace not 16-byte aligned");
  if (flags == TV_SAMPLE_GRID) {
    if (!ws_ok)
      return tv::fail(TV_ERR_INVALID_ARG, "tree accept sample: TV_SAMPLE_GRID needs a workspace of %zu bytes (%zu)",
                      gc_workspace_bytes(B, V), workspace ? workspace_bytes : (size_t)0);
    if (gc_chunks(V) > kGcMaxChunks)
      return tv::fail(TV_ERR_UNSUPPORTED, "tree accept sample: V=%d too large for the grid sampler", V);
  }
  bool grid = false;
  const int st = takes_grid(B, V, flags, ws_ok, stream, &grid);
  if (st) return st;
  if (!grid)
    return launch_walk(p, q, tokens, parent, parent_bstride, n_nodes, u_accept, u_final, B, N, V, ix, o, flags,
                       nullptr, stream);
  const cudaStream_t s = (cudaStream_t)stream;
  char* base = static_cast<char*>(workspace);
  const GcWs ws{reinterpret_cast<int4*>(base), reinterpret_cast<uint64_t*>(base + (size_t)B * 16u), gc_chunks(V)};
  gc_walk_kernel<<<(B + kGcWalkWarps - 1) / kGcWalkWarps, kGcThreads, 0, s>>>(p, q, tokens, parent, parent_bstride,
                                                                             n_nodes, u_accept, B, N, V, ix, o, ws);
  TV_LAUNCH_CHECK("gc_walk_kernel");
  gc_pass_kernel<<<(unsigned)((int64_t)B * ws.nch), kGcThreads, 0, s>>>(p, q, N, V, ix, ws);
  TV_LAUNCH_CHECK("gc_pass_kernel");
  gc_draw_kernel<<<B, kGcThreads, 0, s>>>(p, q, u_final, N, V, ix, o, ws);
  TV_LAUNCH_CHECK("gc_draw_kernel");
  return launch_walk(p, q, tokens, parent, parent_bstride, n_nodes, u_accept, u_final, B, N, V, ix, o,
                     TV_SAMPLE_AUTO, ws.state, stream);
}

}  // namespace

extern "C" int tv_tree_accept_sample(const float* p, const float* q, const int32_t* tokens, const int32_t* parent,
                                     int64_t parent_bstride, const int32_t* n_nodes, const float* u_accept,
                                     const float* u_final, int32_t B, int32_t N, int32_t V, int32_t* out,
                                     int32_t* n_out, int32_t* path, int32_t out_cols, int32_t flags,
                                     void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  tv::clear_error();
  int st = check_accept_args(B, N, V, tokens, parent, parent_bstride, out, n_out, out_cols);
  if (st) return st;
  if (flags < TV_SAMPLE_AUTO || flags > TV_SAMPLE_GRID)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_accept_sample: unknown flags %d", flags);
  if (B == 0) return TV_OK;
  if (!p || !q || !u_accept || !u_final) return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_accept_sample: null pointer");
  return launch_sample(p, q, tokens, parent, parent_bstride, n_nodes, u_accept, u_final, B, N, V, NodeIdx{N, 0, 0},
                       AcceptOut{out, n_out, path, out_cols, status}, flags, workspace, workspace_bytes, stream);
}

extern "C" int tv_chain_accept_sample(const float* p, const float* q, const int32_t* draft, const int32_t* num_draft,
                                      const float* u, const float* u_final, int32_t B, int32_t K, int32_t V,
                                      int32_t* out, int32_t* n_out, int32_t out_cols, int32_t flags, void* workspace,
                                      size_t workspace_bytes, int32_t* status, void* stream) {
  tv::clear_error();
  if (B < 0 || K < 0 || K + 1 > TV_MAX_NODES || V < 1 || out_cols < 1)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_chain_accept_sample: bad sizes B=%d K=%d V=%d out_cols=%d", B, K, V,
                    out_cols);
  if (flags < TV_SAMPLE_AUTO || flags > TV_SAMPLE_GRID)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_chain_accept_sample: unknown flags %d", flags);
  if (B == 0) return TV_OK;
  if (!p || !u_final || !out || !n_out || (K > 0 && (!q || !draft || !u)))
    return tv::fail(TV_ERR_INVALID_ARG, "tv_chain_accept_sample: null pointer");
  const int32_t* parent = nullptr;
  cudaError_t e = cudaGetSymbolAddress((void**)&parent, g_chain_parent);
  if (e != cudaSuccess) return tv::cuda_fail(e, "cudaGetSymbolAddress(chain parent)");
  // K = 0: no node is read but the root; any valid address stands in
  const float* qq = K > 0 ? q : p;
  const int32_t* tok = K > 0 ? draft : parent;
  const float* uu = K > 0 ? u : u_final;
  return launch_sample(p, qq, tok, parent, 0, num_draft, uu, u_final, B, K + 1, V, NodeIdx{K, 1, 1},
                       AcceptOut{out, n_out, nullptr, out_cols, status}, flags, workspace, workspace_bytes, stream);
}

extern "C" size_t tv_accept_sample_workspace_size(int32_t B, int32_t N, int32_t V) {
  (void)N;
  return B > 0 && V > 0 ? gc_workspace_bytes(B, V) : 0;
}

extern "C" int tv_accept_sample_uses_grid(int32_t B, int32_t N, int32_t V, int32_t flags, size_t workspace_bytes,
                                          int32_t* grid) {
  tv::clear_error();
  (void)N;
  if (!grid || B < 0 || V < 1 || flags < TV_SAMPLE_AUTO || flags > TV_SAMPLE_GRID)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_accept_sample_uses_grid: bad arguments");
  const bool ws_ok = workspace_bytes > 0 && workspace_bytes >= gc_workspace_bytes(B, V) &&
                     (int64_t)B * gc_chunks(V) <= INT_MAX;
  bool g = false;
  const int st = takes_grid(B, V, flags, ws_ok, nullptr, &g);
  if (st) return st;
  *grid = g ? 1 : 0;
  return TV_OK;
}
