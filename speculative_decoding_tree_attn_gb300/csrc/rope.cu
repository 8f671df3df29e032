// Depth-indexed rotary embedding of the tree queries and tree keys.
//
// "Build the tree attention mask that verifies a draft tree in one pass",
// "What interviewers probe next" / "Common mistakes": siblings share a
// position and rotating a node at its flattened index scores it in the wrong
// place; "Encode branch histories in masks and positions": rotary features
// follow the model's position semantics.  The positions come from
// tv_tree_mask (prefix length + depth); the cached prefix keys were rotated
// when they were written.
//
// Layout of the table: cos_sin[p][0][k] = cos(p * base^(-2k/D)),
// cos_sin[p][1][k] = sin(...), k < D/2, computed in float64 and rounded once.
// Rotate-half pairing: element k is paired with element k + D/2.
#include <algorithm>
#include <climits>

#include <cuda_bf16.h>

#include "common.h"
#include "rope_math.cuh"

namespace {

__global__ void rope_table_kernel(float* __restrict__ cs, int max_pos, int D, double base) {
  const int half = D / 2;
  const int64_t n = (int64_t)max_pos * half;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int p = (int)(t / half);
    const int k = (int)(t % half);
    const double inv_freq = pow(base, -2.0 * (double)k / (double)D);
    double s, c;
    sincos((double)p * inv_freq, &s, &c);
    cs[(int64_t)p * D + k] = (float)c;
    cs[(int64_t)p * D + half + k] = (float)s;
  }
}

// One thread rotates 8 pairs (elements k..k+7 and k+D/2..k+D/2+7) of one row.
// Rows are enumerated as (b, i, head) with the Hq query heads first, then the
// Hkv tree-key heads of the same node.  Index arithmetic in 32 bits (the
// launcher checks the item count) with the per-row chunk count a constant.
template <typename T, int D>
__global__ void __launch_bounds__(256) rope_apply_kernel(T* __restrict__ q, T* __restrict__ kt,
                                                         const int32_t* __restrict__ pos, const float* __restrict__ cs,
                                                         int max_pos, int total, int Hq, int Hkv,
                                                         int32_t* __restrict__ status) {
  constexpr int half = D / 2;
  constexpr int chunks = half / 8;
  const int heads = Hq + (kt ? Hkv : 0);
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
    const int c = t % chunks;
    const int r = t / chunks;
    const int bi = r / heads;
    const int h = r - bi * heads;
    const int32_t p = __ldg(pos + bi);
    if (p < 0 || p >= max_pos) {  // -1: an absent node of a ragged tree, left as it is
      if (status && c == 0 && p != -1) atomicOr(status, TV_DEV_BAD_POSITION);
      continue;
    }
    T* row = (h < Hq) ? q + ((int64_t)bi * Hq + h) * D : kt + ((int64_t)bi * Hkv + (h - Hq)) * D;
    const float* cosr = cs + (int64_t)p * D + c * 8;
    const float* sinr = cosr + half;
    float x1[8], x2[8], co[8], si[8];
    Vec8<T>::load(row + c * 8, x1);
    Vec8<T>::load(row + half + c * 8, x2);
    Vec8<float>::load(cosr, co);
    Vec8<float>::load(sinr, si);
    float y1[8], y2[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_pair(x1[e], x2[e], co[e], si[e], y1[e], y2[e]);
    Vec8<T>::store(row + c * 8, y1);
    Vec8<T>::store(row + half + c * 8, y2);
  }
}

template <typename T>
int launch_rope(T* q, T* kt, const int32_t* pos, const float* cs, int max_pos, int total, int Hq, int Hkv, int D,
                int32_t* status, cudaStream_t stream) {
  const int blocks = (int)std::min<int64_t>(tv::ceil_div(total, 256), 152 * 16);
  switch (D) {
    case 16: rope_apply_kernel<T, 16><<<blocks, 256, 0, stream>>>(q, kt, pos, cs, max_pos, total, Hq, Hkv, status); break;
    case 32: rope_apply_kernel<T, 32><<<blocks, 256, 0, stream>>>(q, kt, pos, cs, max_pos, total, Hq, Hkv, status); break;
    case 64: rope_apply_kernel<T, 64><<<blocks, 256, 0, stream>>>(q, kt, pos, cs, max_pos, total, Hq, Hkv, status); break;
    case 128: rope_apply_kernel<T, 128><<<blocks, 256, 0, stream>>>(q, kt, pos, cs, max_pos, total, Hq, Hkv, status); break;
    case 256: rope_apply_kernel<T, 256><<<blocks, 256, 0, stream>>>(q, kt, pos, cs, max_pos, total, Hq, Hkv, status); break;
    default: return tv::fail(TV_ERR_UNSUPPORTED, "tv_rope_apply: head_dim %d not in {16, 32, 64, 128, 256}", D);
  }
  TV_LAUNCH_CHECK("rope_apply_kernel");
  return TV_OK;
}

}  // namespace

extern "C" int tv_rope_table(float* cos_sin, int32_t max_pos, int32_t head_dim, double base, void* stream) {
  tv::clear_error();
  if (!cos_sin || max_pos < 1 || head_dim < 2 || head_dim % 2 || !(base > 0.0))
    return tv::fail(TV_ERR_INVALID_ARG, "tv_rope_table: bad arguments");
  const int64_t n = (int64_t)max_pos * (head_dim / 2);
  const int blocks = (int)std::min<int64_t>(tv::ceil_div(n, 256), 4096);
  rope_table_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(cos_sin, max_pos, head_dim, base);
  TV_LAUNCH_CHECK("rope_table_kernel");
  return TV_OK;
}

extern "C" int tv_rope_apply(void* q, void* k_tree, const int32_t* pos, const float* cos_sin, int32_t max_pos,
                             int32_t B, int32_t N, int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t dtype,
                             int32_t* status, void* stream) {
  tv::clear_error();
  if (B < 0 || N < 1 || Hq < 1 || Hkv < 1 || head_dim % 16 || head_dim < 16 || max_pos < 1)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_rope_apply: bad sizes");
  if (dtype != TV_F32 && dtype != TV_BF16) return tv::fail(TV_ERR_UNSUPPORTED, "tv_rope_apply: dtype %d", dtype);
  if (B == 0) return TV_OK;
  if (!q || !pos || !cos_sin) return tv::fail(TV_ERR_INVALID_ARG, "tv_rope_apply: null pointer");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_tree) |
       reinterpret_cast<uintptr_t>(cos_sin)) & 15)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_rope_apply: buffers must be 16-byte aligned");
  const int64_t BN = (int64_t)B * N;
  const int64_t total = BN * (Hq + (k_tree ? Hkv : 0)) * (head_dim / 16);
  if (total >= INT32_MAX) return tv::fail(TV_ERR_UNSUPPORTED, "tv_rope_apply: %lld rotations exceed 2^31", (long long)total);
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == TV_BF16)
    return launch_rope((__nv_bfloat16*)q, (__nv_bfloat16*)k_tree, pos, cos_sin, max_pos, (int)total, Hq, Hkv,
                       head_dim, status, s);
  return launch_rope((float*)q, (float*)k_tree, pos, cos_sin, max_pos, (int)total, Hq, Hkv, head_dim, status, s);
}
