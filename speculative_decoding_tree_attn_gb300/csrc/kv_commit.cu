// Commit of the accepted path's tree K/V into the paged KV cache.
//
// "Build the tree attention mask that verifies a draft tree in one pass",
// "What it costs.": the tree's K/V is written to scratch during verification
// and the accepted path is copied into the cache afterwards; "Tree
// Verification", "The Cost Side": the accepted nodes become the next step's
// prefix.  Node path[b, j] of the accepted path sits at depth j, i.e. at
// cache position L_b + j; its tree K/V rows (every KV head, stored rotated at
// that position) are copied into block block_table[b, (L_b + j) / block_size],
// slot (L_b + j) % block_size, and the prefix length becomes L_b + n_out[b].
// A path step that cannot be committed (a node outside the tree, a position
// without a valid block) ends the committed prefix there: the steps before it
// are copied, the prefix length becomes L_b + (that step's index), and the
// step's reason is flagged; nothing past it is written.
//
// Pure copy work: one CTA per request, its threads over the 16-byte chunks of
// the request's (path step, KV head) rows of K and of V; consecutive threads
// take consecutive chunks, so every row is read and written as whole 16-byte
// vectors and no thread is spent on path steps past n_out.
#include <climits>

#include "common.h"

namespace {

__global__ void __launch_bounds__(256) kv_commit_kernel(char* __restrict__ kc, char* __restrict__ vc,
                                                        int64_t num_blocks, int bs, const int32_t* __restrict__ table,
                                                        int max_blocks, const int32_t* __restrict__ seq_lens,
                                                        int32_t* __restrict__ new_lens, const char* __restrict__ kt,
                                                        const char* __restrict__ vt, const int32_t* __restrict__ path,
                                                        int path_cols, const int32_t* __restrict__ n_out, int N, int Hkv,
                                                        int row_bytes, int32_t* __restrict__ status) {
  // one CTA per request: its n_out path rows x Hkv heads x 16-byte chunks
  const int b = blockIdx.x;
  const int chunks = row_bytes / 16;
  const int L = seq_lens[b];
  __shared__ int s_n;
  if (threadIdx.x == 0) {
    // the committed prefix ends at the first step that cannot be committed
    int n = n_out[b];
    n = n < 0 ? 0 : (n > path_cols ? path_cols : n);
    for (int j = 0; j < n; ++j) {
      const int node = path[(int64_t)b * path_cols + j];
      const int64_t col = ((int64_t)L + j) / bs;
      const int64_t blk = (L >= 0 && col < max_blocks) ? table[(int64_t)b * max_blocks + col] : -1;
      const int bad = (node < 0 || node >= N) ? TV_DEV_BAD_TOPOLOGY
                                               : ((blk < 0 || blk >= num_blocks) ? TV_DEV_OUT_OVERFLOW : 0);
      if (bad) {
        if (status) atomicOr(status, bad);
        n = j;
        break;
      }
    }
    s_n = n;
    if (new_lens) new_lens[b] = L + n;
  }
  __syncthreads();
  const int n = s_n;
  const int per_row = Hkv * chunks;
  for (int t = threadIdx.x; t < n * per_row; t += blockDim.x) {
    const int j = t / per_row;
    const int r = t - j * per_row;
    const int h = r / chunks;
    const int c = r - h * chunks;
    const int node = path[(int64_t)b * path_cols + j];
    const int64_t pos = (int64_t)L + j;
    const int64_t blk = table[(int64_t)b * max_blocks + pos / bs];  // checked above for every step < n
    const int64_t src = (((int64_t)b * N + node) * Hkv + h) * row_bytes + c * 16;
    const int64_t dst = ((blk * Hkv + h) * bs + pos % bs) * row_bytes + c * 16;
    *reinterpret_cast<uint4*>(kc + dst) = *reinterpret_cast<const uint4*>(kt + src);
    *reinterpret_cast<uint4*>(vc + dst) = *reinterpret_cast<const uint4*>(vt + src);
  }
}

}  // namespace

extern "C" int tv_kv_commit(void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size,
                            const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                            int32_t* new_seq_lens, const void* k_tree, const void* v_tree, const int32_t* path,
                            int32_t path_cols, const int32_t* n_out, int32_t B, int32_t N, int32_t Hkv,
                            int32_t head_dim, int32_t dtype, int32_t* status, void* stream) {
  tv::clear_error();
  if (B < 0 || N < 1 || Hkv < 1 || head_dim < 1 || path_cols < 1 || block_size < 1 || max_blocks < 1 ||
      num_blocks < 1)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_kv_commit: bad sizes");
  if (dtype != TV_F32 && dtype != TV_BF16) return tv::fail(TV_ERR_UNSUPPORTED, "tv_kv_commit: dtype %d", dtype);
  const int row_bytes = head_dim * (dtype == TV_F32 ? 4 : 2);
  if (row_bytes % 16) return tv::fail(TV_ERR_UNSUPPORTED, "tv_kv_commit: a K/V row must be a multiple of 16 bytes");
  if (B == 0) return TV_OK;
  if (!k_cache || !v_cache || !block_table || !seq_lens || !k_tree || !v_tree || !path || !n_out)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_kv_commit: null pointer");
  if (new_seq_lens && new_seq_lens == seq_lens)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_kv_commit: new_seq_lens must not alias seq_lens");
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(k_tree) | reinterpret_cast<uintptr_t>(v_tree)) & 15)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_kv_commit: K/V buffers must be 16-byte aligned");
  if ((int64_t)path_cols * Hkv * (row_bytes / 16) >= INT32_MAX)
    return tv::fail(TV_ERR_UNSUPPORTED, "tv_kv_commit: path rows too large");
  kv_commit_kernel<<<B, 256, 0, (cudaStream_t)stream>>>(
      static_cast<char*>(k_cache), static_cast<char*>(v_cache), num_blocks, block_size, block_table, max_blocks,
      seq_lens, new_seq_lens, static_cast<const char*>(k_tree), static_cast<const char*>(v_tree), path, path_cols,
      n_out, N, Hkv, row_bytes, status);
  TV_LAUNCH_CHECK("kv_commit_kernel");
  return TV_OK;
}
