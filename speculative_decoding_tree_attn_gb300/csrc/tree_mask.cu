// tv_tree_mask: batched ancestor rows, depths and position ids on the device;
// tv_tree_prepare: the same plus the rotation of the queries and/or tree keys
// at those positions, in one launch.
//
// "Build the tree attention mask that verifies a draft tree in one pass",
// "The mask.": node i sees itself and its ancestors; its position id is the
// prefix length plus its depth, so siblings share a position.  "Tree
// Verification", "Tree Attention": the flattening is parent-before-child.
//
// One warp per request; lane l owns nodes l and l + 32.  A node's row is built
// by climbing parent pointers, which terminates because every parent index was
// first checked to be smaller than its child's.
//
// Ragged trees ("Build the tree attention mask ...", "What interviewers probe
// next": graph capture needs a fixed tree shape per batch bucket): with
// n_nodes, request b holds nodes 0 .. n_b - 1 of the bucket's N; the others
// are absent -- mask row 0, depth 0, position -1 -- and their parents are not
// read.
#include <algorithm>
#include <type_traits>

#include "common.h"
#include "rope_math.cuh"

namespace {

// Rows, depths and positions of request b, computed by one warp (lane l owns
// nodes l and l + 32) and written to mask/depth/pos at row b; positions also
// to s_pos when given.  Returns false (rows zeroed, status flagged) for a
// request whose first n parents are not a parent-before-child tree.
__device__ void request_rows(const int32_t* __restrict__ parent, int64_t pstride,
                             const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ n_nodes, int b,
                             int N, int32_t* sp, uint64_t* __restrict__ mask, int32_t* __restrict__ depth,
                             int32_t* __restrict__ pos, int32_t* s_pos, int32_t* __restrict__ status) {
  const int lane = threadIdx.x % 32;
  const int32_t* par = parent + (int64_t)b * pstride;
  int n = N;
  if (n_nodes) n = min(max(n_nodes[b], 1), N);

  bool ok = true;
  for (int i = lane; i < n; i += 32) {
    int32_t p = par[i];
    sp[i] = p;
    ok &= (i == 0) ? (p == -1) : (p >= 0 && p < i);
  }
  const int32_t L = seq_lens[b];
  const bool topo_ok = __all_sync(0xffffffffu, ok);
  ok = topo_ok && L >= 0;
  __syncwarp();

  for (int i = lane; i < N; i += 32) {
    uint64_t row = 0;
    int32_t d = 0;
    const int64_t o = (int64_t)b * N + i;
    if (i >= n) {  // absent node
      if (mask) {
        mask[o] = 0;
        depth[o] = 0;
        pos[o] = -1;
      }
      if (s_pos) s_pos[i] = -1;
      continue;
    }
    if (ok) {
      int j = i;
      row = 1ull << j;
      while (sp[j] >= 0) {
        j = sp[j];
        row |= 1ull << j;
        ++d;
      }
    }
    if (mask) {
      mask[o] = row;
      depth[o] = ok ? d : 0;
      pos[o] = ok ? L + d : 0;
    }
    if (s_pos) s_pos[i] = ok ? L + d : -1;
  }
  if (!ok && lane == 0 && status && mask)
    atomicOr(status, (topo_ok ? 0 : TV_DEV_BAD_TOPOLOGY) | (L < 0 ? TV_DEV_BAD_POSITION : 0));
}

__global__ void tree_mask_kernel(const int32_t* __restrict__ parent, int64_t pstride,
                                 const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ n_nodes,
                                 int B, int N, uint64_t* __restrict__ mask, int32_t* __restrict__ depth,
                                 int32_t* __restrict__ pos, int32_t* __restrict__ status) {
  const int warps_per_block = blockDim.x / 32;
  const int b = blockIdx.x * warps_per_block + threadIdx.x / 32;
  if (b >= B) return;
  __shared__ int32_t s_par[8][TV_MAX_NODES];
  request_rows(parent, pstride, seq_lens, n_nodes, b, N, s_par[threadIdx.x / 32], mask, depth, pos, nullptr,
               status);
}

// The mask kernel and RoPE in one launch: CTA (b, y) rebuilds request b's
// positions in shared memory (CTA (b, 0) also writes mask, depth and pos) and
// rotates its share of request b's query rows (when q is given) and tree-key
// rows (when k_tree is given) in place at those positions, with the
// arithmetic of tv_rope_apply.  Rows run node by node, the Hq query heads of
// a node first, then its Hkv tree-key heads.
template <typename T, int D>
__global__ void __launch_bounds__(256) tree_prepare_kernel(
    const int32_t* __restrict__ parent, int64_t pstride, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ n_nodes, int N, uint64_t* __restrict__ mask, int32_t* __restrict__ depth,
    int32_t* __restrict__ pos, T* __restrict__ q, int Hq, T* __restrict__ kt, int Hkv, const float* __restrict__ cs,
    int max_pos, int32_t* __restrict__ status) {
  constexpr int half = D / 2;
  constexpr int chunks = half / 8;
  __shared__ int32_t s_par[TV_MAX_NODES], s_pos[TV_MAX_NODES];
  const int b = blockIdx.x;
  if (threadIdx.x < 32)
    request_rows(parent, pstride, seq_lens, n_nodes, b, N, s_par, blockIdx.y == 0 ? mask : nullptr, depth, pos,
                 s_pos, status);
  __syncthreads();
  const int hq = q ? Hq : 0, hk = kt ? Hkv : 0, heads = hq + hk;
  const int items = N * heads * chunks;
  for (int t = blockIdx.y * blockDim.x + threadIdx.x; t < items; t += gridDim.y * blockDim.x) {
    const int c = t % chunks;
    const int r = t / chunks;  // (node, head) row of request b
    const int i = r / heads, h = r - i * heads;
    const int32_t p = s_pos[i];
    if (p < 0 || p >= max_pos) {  // -1: an absent node (or a bad tree), left as it is
      if (status && c == 0 && p != -1) atomicOr(status, TV_DEV_BAD_POSITION);
      continue;
    }
    T* row = h < hq ? q + (((int64_t)b * N + i) * Hq + h) * D : kt + (((int64_t)b * N + i) * Hkv + (h - hq)) * D;
    const float* cosr = cs + (int64_t)p * D + c * 8;
    float x1[8], x2[8], co[8], si[8], y1[8], y2[8];
    Vec8<T>::load(row + c * 8, x1);
    Vec8<T>::load(row + half + c * 8, x2);
    Vec8<float>::load(cosr, co);
    Vec8<float>::load(cosr + half, si);
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_pair(x1[e], x2[e], co[e], si[e], y1[e], y2[e]);
    Vec8<T>::store(row + c * 8, y1);
    Vec8<T>::store(row + half + c * 8, y2);
  }
}

// The same for bf16 rows of D = 128, a node per warp: the warp reads the
// node's cos/sin table row once (each lane the 8 frequencies of its 16-byte
// chunk) and rotates the node's Hq + Hkv rows four at a time (8 lanes per
// row, one 16-byte load from each half), requesting kBatch rows' loads per
// lane before the first rotation.  Same arithmetic and rounding as
// tv_rope_apply, element by element.
constexpr int kPrepWarps = 8;
template <int D>
__global__ void __launch_bounds__(32 * kPrepWarps) tree_prepare_nodes_kernel(
    const int32_t* __restrict__ parent, int64_t pstride, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ n_nodes, int N, uint64_t* __restrict__ mask, int32_t* __restrict__ depth,
    int32_t* __restrict__ pos, __nv_bfloat16* __restrict__ q, int Hq, __nv_bfloat16* __restrict__ kt, int Hkv,
    const float* __restrict__ cs, int max_pos, int32_t* __restrict__ status) {
  constexpr int half = D / 2;
  constexpr int chunks = half / 8;           // lanes per row
  constexpr int rows_per_it = 32 / chunks;   // rows a warp rotates at once
  constexpr int kBatch = 5;                  // loads in flight per lane and half
  static_assert(32 % chunks == 0, "whole rows per warp");
  __shared__ int32_t s_par[TV_MAX_NODES], s_pos[TV_MAX_NODES];
  const int b = blockIdx.x;
  if (threadIdx.x < 32)
    request_rows(parent, pstride, seq_lens, n_nodes, b, N, s_par, blockIdx.y == 0 ? mask : nullptr, depth, pos,
                 s_pos, status);
  __syncthreads();
  const int hq = q ? Hq : 0, hk = kt ? Hkv : 0, heads = hq + hk;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = lane % chunks, sub = lane / chunks;
  for (int i = blockIdx.y * kPrepWarps + warp; i < N; i += gridDim.y * kPrepWarps) {
    const int32_t p = s_pos[i];
    if (p < 0 || p >= max_pos) {  // -1: an absent node (or a bad tree), left as it is
      if (status && lane == 0 && p != -1) atomicOr(status, TV_DEV_BAD_POSITION);
      continue;
    }
    float co[8], si[8];
    Vec8<float>::load(cs + (int64_t)p * D + c * 8, co);
    Vec8<float>::load(cs + (int64_t)p * D + half + c * 8, si);
    for (int h0 = 0; h0 < heads; h0 += rows_per_it * kBatch) {
      uint4 x1[kBatch], x2[kBatch];
      __nv_bfloat16* rows[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int h = h0 + j * rows_per_it + sub;
        rows[j] = nullptr;
        if (h < heads) {
          rows[j] = h < hq ? q + (((int64_t)b * N + i) * Hq + h) * D : kt + (((int64_t)b * N + i) * Hkv + (h - hq)) * D;
          x1[j] = *reinterpret_cast<const uint4*>(rows[j] + c * 8);
          x2[j] = *reinterpret_cast<const uint4*>(rows[j] + half + c * 8);
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (!rows[j]) continue;
        const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&x1[j]);
        const __nv_bfloat162* bb = reinterpret_cast<const __nv_bfloat162*>(&x2[j]);
        uint4 y1, y2;
        __nv_bfloat162* o1 = reinterpret_cast<__nv_bfloat162*>(&y1);
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&y2);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 u = __bfloat1622float2(a[e]), v = __bfloat1622float2(bb[e]);
          float r1a, r2a, r1b, r2b;
          rope_pair(u.x, v.x, co[2 * e], si[2 * e], r1a, r2a);
          rope_pair(u.y, v.y, co[2 * e + 1], si[2 * e + 1], r1b, r2b);
          o1[e] = __floats2bfloat162_rn(r1a, r1b);
          o2[e] = __floats2bfloat162_rn(r2a, r2b);
        }
        *reinterpret_cast<uint4*>(rows[j] + c * 8) = y1;
        *reinterpret_cast<uint4*>(rows[j] + half + c * 8) = y2;
      }
    }
  }
}

template <typename T, int D>
int launch_prepare(const int32_t* parent, int64_t pstride, const int32_t* seq_lens, const int32_t* n_nodes, int B,
                   int N, uint64_t* mask, int32_t* depth, int32_t* pos, void* q, int Hq, void* kt, int Hkv,
                   const float* cs, int max_pos, int32_t* status, cudaStream_t stream) {
  const int heads = (q ? Hq : 0) + (kt ? Hkv : 0);
  if constexpr (std::is_same<T, __nv_bfloat16>::value && D == 128) {
    if (heads) {
      const int ys = (int)std::min<int64_t>(tv::ceil_div(N, kPrepWarps), 32);
      tree_prepare_nodes_kernel<D><<<dim3(B, ys), 32 * kPrepWarps, 0, stream>>>(
          parent, pstride, seq_lens, n_nodes, N, mask, depth, pos, static_cast<__nv_bfloat16*>(q), Hq,
          static_cast<__nv_bfloat16*>(kt), Hkv, cs, max_pos, status);
      TV_LAUNCH_CHECK("tree_prepare_nodes_kernel");
      return TV_OK;
    }
  }
  const int items = N * heads * (D / 16);
  const int ys = heads ? (int)std::min<int64_t>(tv::ceil_div(items, 256 * 4), 32) : 1;
  tree_prepare_kernel<T, D><<<dim3(B, ys), 256, 0, stream>>>(parent, pstride, seq_lens, n_nodes, N, mask, depth,
                                                              pos, static_cast<T*>(q), Hq, static_cast<T*>(kt), Hkv,
                                                              cs, max_pos, status);
  TV_LAUNCH_CHECK("tree_prepare_kernel");
  return TV_OK;
}

}  // namespace

extern "C" int tv_tree_mask(const int32_t* parent, int64_t parent_bstride, const int32_t* seq_lens,
                            const int32_t* n_nodes, int32_t B, int32_t N, uint64_t* mask, int32_t* depth,
                            int32_t* pos, int32_t* status, void* stream) {
  tv::clear_error();
  if (B < 0 || N < 1 || N > TV_MAX_NODES || parent_bstride < 0)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_mask: bad sizes B=%d N=%d stride=%lld", B, N,
                    (long long)parent_bstride);
  if (B == 0) return TV_OK;
  if (!parent || !seq_lens || !mask || !depth || !pos)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_mask: null pointer");
  const int threads = 256;
  const int blocks = (int)tv::ceil_div(B, threads / 32);
  tree_mask_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(parent, parent_bstride, seq_lens, n_nodes, B, N,
                                                                 mask, depth, pos, status);
  TV_LAUNCH_CHECK("tree_mask_kernel");
  return TV_OK;
}

extern "C" int tv_tree_prepare(const int32_t* parent, int64_t parent_bstride, const int32_t* seq_lens,
                               const int32_t* n_nodes, int32_t B, int32_t N, uint64_t* mask, int32_t* depth,
                               int32_t* pos, void* q, int32_t Hq, void* k_tree, int32_t Hkv, int32_t head_dim,
                               int32_t dtype, const float* cos_sin, int32_t max_pos, int32_t* status, void* stream) {
  tv::clear_error();
  if (B < 0 || N < 1 || N > TV_MAX_NODES || parent_bstride < 0 || max_pos < 0)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_prepare: bad sizes B=%d N=%d stride=%lld max_pos=%d", B, N,
                    (long long)parent_bstride, max_pos);
  const bool rot = q || k_tree;
  if (rot && ((q && Hq < 1) || (k_tree && Hkv < 1) || !cos_sin || (dtype != TV_F32 && dtype != TV_BF16)))
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_prepare: rotation needs Hq/Hkv >= 1, a table and dtype f32/bf16");
  if (rot && (int64_t)B * N * ((q ? Hq : 0) + (k_tree ? Hkv : 0)) * head_dim >= (int64_t(1) << 40))
    return tv::fail(TV_ERR_UNSUPPORTED, "tv_tree_prepare: rows too large");
  if (B == 0) return TV_OK;
  if (!parent || !seq_lens || !mask || !depth || !pos)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_prepare: null pointer");
  cudaStream_t s = (cudaStream_t)stream;
#define TV_PREP(T, D) return launch_prepare<T, D>(parent, parent_bstride, seq_lens, n_nodes, B, N, mask, depth, pos, \
                                                  q, Hq, k_tree, Hkv, cos_sin, max_pos, status, s)
  if (!rot) TV_PREP(float, 128);
  switch (head_dim) {
    case 16: if (dtype == TV_BF16) TV_PREP(__nv_bfloat16, 16); TV_PREP(float, 16);
    case 32: if (dtype == TV_BF16) TV_PREP(__nv_bfloat16, 32); TV_PREP(float, 32);
    case 64: if (dtype == TV_BF16) TV_PREP(__nv_bfloat16, 64); TV_PREP(float, 64);
    case 128: if (dtype == TV_BF16) TV_PREP(__nv_bfloat16, 128); TV_PREP(float, 128);
    case 256: if (dtype == TV_BF16) TV_PREP(__nv_bfloat16, 256); TV_PREP(float, 256);
    default: return tv::fail(TV_ERR_UNSUPPORTED, "tv_tree_prepare: head_dim %d not in {16, 32, 64, 128, 256}", head_dim);
  }
#undef TV_PREP
}
