// The rotate-half rotation of one frequency pair in float32, shared by every
// kernel that applies RoPE (the separate rope kernel, the tree-prepare
// kernel and the attention kernels that rotate Q as they load it), written
// with explicitly rounded products so that no call site can be contracted
// differently and all of them give the same bits:
//   y1 = x1 cos - x2 sin,   y2 = x2 cos + x1 sin.
// "Build the tree attention mask that verifies a draft tree in one pass",
// "What interviewers probe next": a node is rotated at its depth position.
#pragma once

#include <cuda_bf16.h>

__device__ __forceinline__ void rope_pair(float x1, float x2, float c, float s, float& y1, float& y2) {
  y1 = __fmaf_rn(x1, c, -__fmul_rn(x2, s));
  y2 = __fmaf_rn(x2, c, __fmul_rn(x1, s));
}

template <typename T>
struct Vec8;  // eight consecutive elements, one 16- or 32-byte access

template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 raw = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 raw;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = raw;
  }
};

template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[8]) {
    float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

