// tv_tree_mask: batched ancestor rows, depths and position ids on the device.
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
#include "common.h"

namespace {

__global__ void tree_mask_kernel(const int32_t* __restrict__ parent, int64_t pstride,
                                 const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ n_nodes,
                                 int B, int N, uint64_t* __restrict__ mask, int32_t* __restrict__ depth,
                                 int32_t* __restrict__ pos, int32_t* __restrict__ status) {
  const int warps_per_block = blockDim.x / 32;
  const int b = blockIdx.x * warps_per_block + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (b >= B) return;
  const int32_t* par = parent + (int64_t)b * pstride;
  __shared__ int32_t s_par[8][TV_MAX_NODES];
  int32_t* sp = s_par[threadIdx.x / 32];
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
      mask[o] = 0;
      depth[o] = 0;
      pos[o] = -1;
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
    mask[o] = row;
    depth[o] = ok ? d : 0;
    pos[o] = ok ? L + d : 0;
  }
  if (!ok && lane == 0 && status)
    atomicOr(status, (topo_ok ? 0 : TV_DEV_BAD_TOPOLOGY) | (L < 0 ? TV_DEV_BAD_POSITION : 0));
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
