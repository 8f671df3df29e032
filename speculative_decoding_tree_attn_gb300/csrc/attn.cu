// Tree attention: the plan and combine kernels, the CUDA-core (FP32 FFMA)
// kernel, and the tv_tree_attn_verify / tv_tree_attn_verify_rope entry points
// that dispatch between the CUDA-core kernel and the tcgen05 kernel of
// attn_tc.cu (the _rope variant rotates each query row as it is loaded).
//
// What is computed ("Tree Verification", "Tree Attention"; "Build the tree
// attention mask that verifies a draft tree in one pass", "The mask."): each
// row (request b, node i, query head h) attends to the whole cached prefix of
// b with no mask, then to the tree nodes whose bit is set in the node's
// ancestor row (itself and its ancestors) -- the [prefix all true | tree
// mask] step mask, with the tree part taken as per-node bit rows.  Online
// softmax in the log2 domain with float32 accumulation.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "attn_common.cuh"
#include "rope_math.cuh"
#include "attn_tc.h"

namespace tv {

namespace {

// ---------------------------------------------------------------------------
// plan: tile_start[u] = sum of tile counts of units < u
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_kernel(AttnParams p) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  for (int base = 0; base < p.U; base += blockDim.x) {
    const int u = base + threadIdx.x;
    int n = 0;
    if (u < p.U) {
      int b, kvh, rg;
      unit_coords(p, u, b, kvh, rg);
      n = (clamp_len(p, b) + p.BLK - 1) / p.BLK + 1 + p.unit_cost;
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = (lane < (int)(blockDim.x / 32)) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += v;
      }
      warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (warp ? warp_sums[warp - 1] : 0) + incl - n;
    if (u < p.U) p.tile_start[u] = before;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = before + n;
    __syncthreads();
  }
  if (threadIdx.x == 0) p.tile_start[p.U] = carry;
}

// ---------------------------------------------------------------------------
// element helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// CUDA-core kernel: 8 warps, 32 rows per unit (4 per warp), 64-key tiles in
// shared memory as float32.  Lane j scores keys j and j + 32 of the tile and
// owns output dimensions lane + 32 e.
// ---------------------------------------------------------------------------
constexpr int kSimtBlk = 64;
constexpr int kSimtRows = 32;
constexpr int kSimtWarps = 8;

template <int D>
constexpr size_t simt_smem_bytes() {
  return sizeof(float) * ((size_t)kSimtBlk * (D + 1) + (size_t)kSimtBlk * D + (size_t)kSimtRows * D);
}

template <typename T, int D>
__global__ void __launch_bounds__(kSimtWarps * 32) attn_simt_kernel(AttnParams p) {
  constexpr int RPW = kSimtRows / kSimtWarps;
  constexpr int DPL = D / 32;
  extern __shared__ float smem[];
  float* Ks = smem;                          // [BLK][D + 1]
  float* Vs = Ks + kSimtBlk * (D + 1);       // [BLK][D]
  float* Qs = Vs + kSimtBlk * D;             // [RPG][D]
  __shared__ uint64_t s_rowmask[kSimtRows];

  const T* __restrict__ q = static_cast<const T*>(p.q);
  const T* __restrict__ kc = static_cast<const T*>(p.k_cache);
  const T* __restrict__ vc = static_cast<const T*>(p.v_cache);
  const T* __restrict__ kt = static_cast<const T*>(p.k_tree);
  const T* __restrict__ vt = static_cast<const T*>(p.v_tree);
  T* __restrict__ out = static_cast<T*>(p.out);

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int64_t T_total = p.tile_start[p.U];
  const int64_t c = blockIdx.x;
  const int64_t t0 = cta_start(c, T_total, p.P), t1 = cta_start(c + 1, T_total, p.P);
  if (t0 >= t1) return;

  for (int u = find_unit(p.tile_start, p.U, t0); u < p.U && p.tile_start[u] < t1; ++u) {
    const int64_t us = p.tile_start[u], ue = p.tile_start[u + 1];
    const int a = (int)(max(t0, us) - us), e = (int)(min(t1, ue) - us), n_u = (int)(ue - us);
    int b, kvh, rg;
    unit_coords(p, u, b, kvh, rg);
    const int L = clamp_len(p, b);

    for (int idx = tid; idx < kSimtRows * D; idx += blockDim.x) {
      const int r = idx / D, d = idx % D, gr = rg * kSimtRows + r;
      float v = 0.f;
      if (gr < p.R) {
        const int i = gr / p.G, h = kvh * p.G + gr % p.G;
        const T* qrow = q + (((int64_t)b * p.N + i) * p.Hq + h) * D;
        v = to_f32(qrow[d]);
        if (p.rope_cs) {
          // rotate at L_b + depth (depth from the ancestor row), the
          // arithmetic and rounding of tv_rope_apply; an absent node (row 0)
          // or a position past the table stays as it is
          const uint64_t mr = p.mask[(int64_t)b * p.mask_bstride + i];
          const int ps = mr ? p.seq_lens[b] + __popcll(mr) - 1 : -1;
          if (ps >= 0 && ps < p.rope_max_pos) {
            constexpr int half = D / 2;
            const int k = d % half;
            float y1, y2;
            rope_pair(to_f32(qrow[k]), to_f32(qrow[k + half]), p.rope_cs[(int64_t)ps * D + k],
                      p.rope_cs[(int64_t)ps * D + half + k], y1, y2);
            v = to_f32(from_f32<T>(d < half ? y1 : y2));
          } else if (ps >= p.rope_max_pos && d == 0 && p.status) {
            atomicOr(p.status, TV_DEV_BAD_POSITION);
          }
        }
      }
      Qs[idx] = v;
    }
    for (int r = tid; r < kSimtRows; r += blockDim.x) {
      const int gr = rg * kSimtRows + r;
      s_rowmask[r] = gr < p.R ? p.mask[(int64_t)b * p.mask_bstride + gr / p.G] : 0ull;
    }
    float m[RPW], l[RPW], acc[RPW][DPL];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
      m[rr] = -INFINITY;
      l[rr] = 0.f;
#pragma unroll
      for (int x = 0; x < DPL; ++x) acc[rr][x] = 0.f;
    }
    __syncthreads();

    for (int k = a; k < e; ++k) {
      const bool tree_tile = (k == n_u - 1);
      for (int idx = tid; idx < kSimtBlk * D; idx += blockDim.x) {
        const int j = idx / D, d = idx % D;
        float kv = 0.f, vv = 0.f;
        if (tree_tile) {
          if (j < p.N) {
            const int64_t o = (((int64_t)b * p.N + j) * p.Hkv + kvh) * D + d;
            kv = to_f32(kt[o]);
            vv = to_f32(vt[o]);
          }
        } else {
          const int t = k * kSimtBlk + j;
          if (t < L) {
            const int64_t blk = p.block_table[(int64_t)b * p.max_blocks + t / p.block_size];
            if (blk >= 0 && blk < p.num_blocks) {  // a bad table entry reads as zeros
              const int64_t o = ((blk * p.Hkv + kvh) * p.block_size + t % p.block_size) * D + d;
              kv = to_f32(kc[o]);
              vv = to_f32(vc[o]);
            } else if (d == 0 && p.status) {
              atomicOr(p.status, TV_DEV_BAD_BLOCK);
            }
          }
        }
        Ks[j * (D + 1) + d] = kv;
        Vs[j * D + d] = vv;
      }
      __syncthreads();
#pragma unroll
      for (int rr = 0; rr < RPW; ++rr) {
        const int r = warp * RPW + rr;
        if (rg * kSimtRows + r >= p.R) continue;
        float s0 = 0.f, s1 = 0.f;
        const float* qr = Qs + r * D;
        const float* k0 = Ks + lane * (D + 1);
        const float* k1 = Ks + (lane + 32) * (D + 1);
#pragma unroll 8
        for (int d = 0; d < D; ++d) {
          const float qd = qr[d];
          s0 = fmaf(qd, k0[d], s0);
          s1 = fmaf(qd, k1[d], s1);
        }
        bool ok0, ok1;
        if (tree_tile) {
          const uint64_t row = s_rowmask[r];
          ok0 = lane < p.N && ((row >> lane) & 1ull);
          ok1 = lane + 32 < p.N && ((row >> (lane + 32)) & 1ull);
        } else {
          ok0 = k * kSimtBlk + lane < L;
          ok1 = k * kSimtBlk + lane + 32 < L;
        }
        const float x0 = ok0 ? s0 * p.scale_log2 : -INFINITY;
        const float x1 = ok1 ? s1 * p.scale_log2 : -INFINITY;
        const float m_new = fmaxf(m[rr], warp_max(fmaxf(x0, x1)));
        if (m_new == -INFINITY) continue;
        const float alpha = exp2f(m[rr] - m_new);
        const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
        l[rr] = l[rr] * alpha + warp_sum(p0 + p1);
#pragma unroll
        for (int x = 0; x < DPL; ++x) acc[rr][x] *= alpha;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
          const float pa = __shfl_sync(0xffffffffu, p0, j);
          const float pb = __shfl_sync(0xffffffffu, p1, j);
#pragma unroll
          for (int x = 0; x < DPL; ++x)
            acc[rr][x] = fmaf(pa, Vs[j * D + lane + 32 * x], fmaf(pb, Vs[(j + 32) * D + lane + 32 * x], acc[rr][x]));
        }
        m[rr] = m_new;
      }
      __syncthreads();
    }

    const bool complete = (a == 0 && e == n_u);
    const int slot = (t0 < us) ? 1 : 0;  // 0: the CTA's first unit, 1: its last
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
      const int r = warp * RPW + rr, gr = rg * kSimtRows + r;
      if (gr >= p.R) continue;
      const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;  // no key at all: zero row, lse -inf
      const float lse2 = m[rr] + log2f(l[rr]);
      if (complete) {
        const int i = gr / p.G, h = kvh * p.G + gr % p.G;
        const int64_t row = ((int64_t)b * p.N + i) * p.Hq + h;
#pragma unroll
        for (int x = 0; x < DPL; ++x) out[row * D + lane + 32 * x] = from_f32<T>(acc[rr][x] * inv);
        if (p.lse && lane == 0) p.lse[row] = lse2 * 0.69314718055994530942f;
      } else {
        const int64_t srow = (c * 2 + slot) * p.RPG + r;
#pragma unroll
        for (int x = 0; x < DPL; ++x) p.part_o[srow * D + lane + 32 * x] = acc[rr][x] * inv;
        if (lane == 0) p.part_lse[srow] = lse2;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// combine: O = sum_k 2^(lse_k - lse*) O_k over the pieces of a split unit
// ---------------------------------------------------------------------------
// Only units cut by a slice boundary need merging, and there are fewer such
// boundaries than CTAs: block x handles the boundary between CTA x and x + 1
// (the unit holding CTA x + 1's first tile, when that tile is not the unit's
// first and x is the unit's first CTA); one warp per row, 32 rows per block.
constexpr int kCombineRows = 32;

template <typename T>
__global__ void __launch_bounds__(32 * kCombineRows) combine_kernel(AttnParams p) {
  const int64_t T_total = p.tile_start[p.U];
  const int64_t cut = cta_start(blockIdx.x + 1, T_total, p.P);
  if (cut >= T_total) return;
  const int u = find_unit(p.tile_start, p.U, cut);
  const int64_t us = p.tile_start[u] + p.unit_cost, ue = p.tile_start[u + 1];  // real tiles [us, ue)
  if (cut <= us) return;                                // the boundary does not cut real tiles
  const int64_t c0 = cta_of(us, T_total, p.P), c1 = cta_of(ue - 1, T_total, p.P);
  if (c0 != (int64_t)blockIdx.x) return;                // merged at the unit's first boundary
  int b, kvh, rg;
  unit_coords(p, u, b, kvh, rg);
  const int lane = threadIdx.x % 32;
  const int r = blockIdx.y * kCombineRows + threadIdx.x / 32;
  if (r >= p.RPG || rg * p.RPG + r >= p.R) return;
  T* __restrict__ out = static_cast<T*>(p.out);
  const int gr = rg * p.RPG + r;
  const int i = gr / p.G, h = kvh * p.G + gr % p.G;
  const int64_t orow = ((int64_t)b * p.N + i) * p.Hq + h;
  const int64_t n_all = c1 - c0 + 1;
  const int dpl = p.D / 32;  // output elements per lane (<= 8)
  float mx = -INFINITY, z = 0.f;
  float acc[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) acc[x] = 0.f;
  for (int64_t j0 = 0; j0 < n_all; j0 += 32) {
    // lane k takes piece j0 + k: the slice of CTA c0 + j0 + k (slot 1 only
    // for the first CTA when the unit began inside its slice; empty slices skipped)
    const int64_t j = j0 + lane;
    int32_t slot = -1;
    if (j < n_all) {
      const int64_t c = c0 + j;
      const int64_t s0 = cta_start(c, T_total, p.P), s1 = cta_start(c + 1, T_total, p.P);
      if (s0 < s1) slot = (int32_t)(c * 2 + (s0 < us ? 1 : 0));
    }
    const float l2 = slot >= 0 ? p.part_lse[(int64_t)slot * p.RPG + r] : -INFINITY;
    float cm = l2;
#pragma unroll
    for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
    const float m_new = fmaxf(mx, cm);
    const float alpha = (mx == -INFINITY) ? 0.f : exp2f(mx - m_new);
    const float w = slot >= 0 ? exp2f(l2 - m_new) : 0.f;
    float wz = w;
#pragma unroll
    for (int o = 16; o; o >>= 1) wz += __shfl_xor_sync(0xffffffffu, wz, o);
    z = z * alpha + wz;
    mx = m_new;
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[x] *= alpha;
    const int n_here = (n_all - j0) < 32 ? (int)(n_all - j0) : 32;
    for (int k = 0; k < n_here; ++k) {
      const float wk = __shfl_sync(0xffffffffu, w, k);
      const int32_t sk = __shfl_sync(0xffffffffu, slot, k);
      if (sk < 0) continue;
      const float* src = p.part_o + ((int64_t)sk * p.RPG + r) * p.D;
#pragma unroll
      for (int x = 0; x < 8; ++x)
        if (x < dpl) acc[x] = fmaf(wk, __ldg(src + lane + 32 * x), acc[x]);
    }
  }
  const float inv = 1.f / z;
#pragma unroll
  for (int x = 0; x < 8; ++x)
    if (x < dpl) out[orow * p.D + lane + 32 * x] = from_f32<T>(acc[x] * inv);
  if (p.lse && lane == 0) p.lse[orow] = (mx + log2f(z)) * 0.69314718055994530942f;
}

template <typename T, int D>
int launch_simt_t(const AttnParams& p, cudaStream_t stream) {
  const size_t smem = simt_smem_bytes<D>();
  cudaError_t err = cudaFuncSetAttribute(attn_simt_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute(attn_simt_kernel)");
  attn_simt_kernel<T, D><<<p.P, kSimtWarps * 32, smem, stream>>>(p);
  TV_LAUNCH_CHECK("attn_simt_kernel");
  return TV_OK;
}

template <typename T, int D>
int simt_blocks_per_sm(int* n) {
  const size_t smem = simt_smem_bytes<D>();
  cudaError_t err = cudaFuncSetAttribute(attn_simt_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute(attn_simt_kernel)");
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, attn_simt_kernel<T, D>, kSimtWarps * 32, smem);
  if (err != cudaSuccess) return cuda_fail(err, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  if (*n < 1) *n = 1;
  return TV_OK;
}

int simt_dispatch(const AttnParams& p, int dtype, cudaStream_t stream, int* blocks_per_sm) {
#define TV_SIMT_CASE(TT, DD)                                                   \
  if (p.D == DD) return blocks_per_sm ? simt_blocks_per_sm<TT, DD>(blocks_per_sm) \
                                      : launch_simt_t<TT, DD>(p, stream);
  if (dtype == TV_F32) {
    TV_SIMT_CASE(float, 64) TV_SIMT_CASE(float, 128) TV_SIMT_CASE(float, 256)
  } else {
    TV_SIMT_CASE(__nv_bfloat16, 64) TV_SIMT_CASE(__nv_bfloat16, 128) TV_SIMT_CASE(__nv_bfloat16, 256)
  }
#undef TV_SIMT_CASE
  return fail(TV_ERR_UNSUPPORTED, "tree attention: head_dim %d not in {64, 128, 256}", p.D);
}

// Shape decisions shared by the workspace query and the launch.
struct AttnConfig {
  bool tc;
  bool duo;  // units of 129-256 rows on CTA pairs (P counts pairs)
  int RPG, RG, U, BLK, P;
  int64_t off_arrive, off_part_o, off_part_lse, bytes;
};

// Scratch of one call: the tile plan [U + 1] (CUDA-core path), the arrival
// counters [P][RPG] (tcgen05 path), the partial outputs [P][2][RPG][D] and
// their log2-sum-exps [P][2][RPG].
void layout_workspace(AttnConfig* cfg, int D) {
  const int64_t plan = align256((int64_t)(cfg->U + 1) * 4);
  const int64_t arrive = align256((int64_t)cfg->P * cfg->RPG * 4);
  const int64_t po = align256((int64_t)cfg->P * 2 * cfg->RPG * D * 4);
  const int64_t pl = align256((int64_t)cfg->P * 2 * cfg->RPG * 4);
  cfg->off_arrive = plan;
  cfg->off_part_o = plan + arrive;
  cfg->off_part_lse = plan + arrive + po;
  cfg->bytes = plan + arrive + po + pl;
}

int attn_config(int B, int N, int Hq, int Hkv, int D, int dtype, int block_size, int num_ctas, int flags,
                AttnConfig* cfg) {
  const bool rope = (flags & TV_ATTN_ROPE_Q) != 0;
  const bool pairs = (flags & TV_ATTN_CTA_PAIRS) != 0;
  flags &= ~(TV_ATTN_ROPE_Q | TV_ATTN_CTA_PAIRS | TV_ATTN_WORKSPACE_ZEROED);
  if (B < 0 || N < 1 || N > TV_MAX_NODES || Hq < 1 || Hkv < 1 || Hq % Hkv)
    return fail(TV_ERR_INVALID_ARG, "tree attention: bad sizes B=%d N=%d Hq=%d Hkv=%d", B, N, Hq, Hkv);
  if (D != 64 && D != 128 && D != 256)
    return fail(TV_ERR_UNSUPPORTED, "tree attention: head_dim %d not in {64, 128, 256}", D);
  if (dtype != TV_F32 && dtype != TV_BF16) return fail(TV_ERR_UNSUPPORTED, "tree attention: dtype %d", dtype);
  if (block_size < 1) return fail(TV_ERR_INVALID_ARG, "tree attention: block_size %d", block_size);
  if (num_ctas < 0) return fail(TV_ERR_INVALID_ARG, "tree attention: num_ctas %d", num_ctas);
  const int sel = flags & 3;
  if (sel == 3 || (flags & ~7)) return fail(TV_ERR_INVALID_ARG, "tree attention: bad flags %d", flags);
  DeviceInfo dev;
  int st = current_device_info(&dev);
  if (st) return st;
  const int G = Hq / Hkv, R = G * N;
  const bool tc_ok = tc_supported(dev, dtype, D, R, G, block_size, rope);
  if (sel == TV_ATTN_TCGEN05 && !tc_ok)
    return fail(TV_ERR_UNSUPPORTED, "tcgen05 tree attention: %s (sm_%d%d, opt-in smem %zu B)",
                tc_unsupported_reason(dev, dtype, D, R, G, block_size, rope), dev.cc_major, dev.cc_minor,
                dev.max_smem_optin);
  cfg->tc = (sel == TV_ATTN_TCGEN05) || (sel == TV_ATTN_AUTO && tc_ok);
  int per_sm = 1;
  if (cfg->tc) {
    cfg->RPG = tc_rows_per_unit(R);
    cfg->BLK = kTcBlk;
    per_sm = tc_ctas_per_sm(R);
  } else {
    cfg->RPG = kSimtRows;
    cfg->BLK = kSimtBlk;
    AttnParams dummy{};
    dummy.D = D;
    st = simt_dispatch(dummy, dtype, nullptr, &per_sm);
    if (st) return st;
  }
  cfg->RG = (int)ceil_div(R, cfg->RPG);
  cfg->U = B * Hkv * cfg->RG;
  cfg->duo = cfg->tc && cfg->RPG == kTcMaxRows && pairs;
  cfg->P = num_ctas > 0 ? num_ctas : (cfg->duo ? tc_duo_pairs(dev) : dev.sm_count * per_sm);
  layout_workspace(cfg, D);
  return TV_OK;
}

}  // namespace

int launch_plan(const AttnParams& p, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(p);
  TV_LAUNCH_CHECK("plan_kernel");
  return TV_OK;
}

int launch_combine(const AttnParams& p, int dtype, cudaStream_t stream) {
  if (p.P <= 1) return TV_OK;
  const dim3 grid(p.P - 1, (p.RPG + kCombineRows - 1) / kCombineRows);
  if (dtype == TV_F32) combine_kernel<float><<<grid, 32 * kCombineRows, 0, stream>>>(p);
  else combine_kernel<__nv_bfloat16><<<grid, 32 * kCombineRows, 0, stream>>>(p);
  TV_LAUNCH_CHECK("combine_kernel");
  return TV_OK;
}

}  // namespace tv

extern "C" int tv_tree_attn_workspace_size(int32_t B, int32_t N, int32_t Hq, int32_t Hkv, int32_t head_dim,
                                           int32_t dtype, int32_t block_size, int32_t num_ctas, int32_t flags,
                                           size_t* bytes) {
  tv::clear_error();
  if (!bytes) return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_attn_workspace_size: null output");
  tv::AttnConfig cfg;
  int st = tv::attn_config(B, N, Hq, Hkv, head_dim, dtype, block_size, num_ctas, flags, &cfg);
  if (st) return st;
  *bytes = (size_t)cfg.bytes;
  return TV_OK;
}

namespace tv {
namespace {

int verify_impl(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks, int32_t block_size,
                const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens, const void* k_tree,
                const void* v_tree, const uint64_t* mask, int64_t mask_bstride, int32_t B, int32_t N, int32_t Hq,
                int32_t Hkv, int32_t head_dim, int32_t dtype, float scale, void* out, float* lse, void* workspace,
                size_t workspace_bytes, int32_t num_ctas, int32_t flags, const float* rope_cs, int32_t rope_max_pos,
                int32_t* status, void* stream) {
  AttnConfig cfg;
  int st = attn_config(B, N, Hq, Hkv, head_dim, dtype, block_size, num_ctas, flags, &cfg);
  if (st) return st;
  if (B == 0) return TV_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !k_tree || !v_tree || !mask || !out)
    return fail(TV_ERR_INVALID_ARG, "tv_tree_attn_verify: null pointer");
  if (num_blocks < 1 || max_blocks < 1 || mask_bstride < 0)
    return fail(TV_ERR_INVALID_ARG, "tv_tree_attn_verify: bad num_blocks/max_blocks/mask stride");
  if (cfg.tc && num_blocks * Hkv * block_size >= (int64_t(1) << 31))
    return fail(TV_ERR_UNSUPPORTED, "tv_tree_attn_verify: KV cache rows exceed the tensor-map range");
  // the tensor-core kernels write output rows in 32-byte pieces and read Q
  // rows in 16-byte pieces (and by TMA)
  if (cfg.tc && ((reinterpret_cast<uintptr_t>(out) & 31) || (reinterpret_cast<uintptr_t>(q) & 15)))
    return fail(TV_ERR_INVALID_ARG, "tv_tree_attn_verify: out must be 32-byte and q 16-byte aligned");
  if (!workspace || workspace_bytes < (size_t)cfg.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(TV_ERR_WORKSPACE, "tv_tree_attn_verify: workspace needs %lld bytes, 256-byte aligned",
                (long long)cfg.bytes);
  AttnParams p{};
  p.q = q; p.k_cache = k_cache; p.v_cache = v_cache; p.block_table = block_table; p.seq_lens = seq_lens;
  p.k_tree = k_tree; p.v_tree = v_tree; p.mask = mask; p.mask_bstride = mask_bstride; p.out = out; p.lse = lse;
  char* ws = static_cast<char*>(workspace);
  p.tile_start = reinterpret_cast<int32_t*>(ws);
  p.arrive = reinterpret_cast<uint32_t*>(ws + cfg.off_arrive);
  p.part_o = reinterpret_cast<float*>(ws + cfg.off_part_o);
  p.part_lse = reinterpret_cast<float*>(ws + cfg.off_part_lse);
  p.num_blocks = num_blocks; p.block_size = block_size; p.max_blocks = max_blocks;
  p.B = B; p.N = N; p.Hq = Hq; p.Hkv = Hkv; p.D = head_dim; p.G = Hq / Hkv;
  p.R = p.G * N; p.RPG = cfg.RPG; p.RG = cfg.RG; p.U = cfg.U; p.BLK = cfg.BLK; p.P = cfg.P;
  p.unit_cost = cfg.tc ? tc_unit_cost(cfg.RPG) : 0;
  p.direct_merge = (flags & TV_ATTN_PUBLISH_ALL) ? 0 : 1;
  p.rope_cs = rope_cs;
  p.rope_max_pos = rope_max_pos;
  p.status = status;
  // tile indices of the plan are 32-bit
  const int64_t unit_tiles_max = ((int64_t)max_blocks * block_size + cfg.BLK - 1) / cfg.BLK + 1 + p.unit_cost;
  if ((int64_t)cfg.U * unit_tiles_max >= (int64_t(1) << 31))
    return fail(TV_ERR_UNSUPPORTED, "tv_tree_attn_verify: %d units of up to %lld tiles exceed 2^31 plan tiles", cfg.U,
                (long long)unit_tiles_max);
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = (cudaStream_t)stream;
  if (cfg.tc) {
    // the tcgen05 kernel plans its own slice and merges split units itself;
    // it only needs the arrival counters at zero, and leaves them so
    if (!(flags & TV_ATTN_WORKSPACE_ZEROED)) {
      cudaError_t e = cudaMemsetAsync(p.arrive, 0, (size_t)p.P * p.RPG * sizeof(uint32_t), s);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(arrival counters)");
    }
    return launch_attn_tc(p, status, s, cfg.duo);
  }
  if ((st = launch_plan(p, s))) return st;
  if ((st = simt_dispatch(p, dtype, s, nullptr))) return st;
  return launch_combine(p, dtype, s);
}

}  // namespace
}  // namespace tv

extern "C" int tv_tree_attn_verify(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
                                   int32_t block_size, const int32_t* block_table, int32_t max_blocks,
                                   const int32_t* seq_lens, const void* k_tree, const void* v_tree,
                                   const uint64_t* mask, int64_t mask_bstride, int32_t B, int32_t N, int32_t Hq,
                                   int32_t Hkv, int32_t head_dim, int32_t dtype, float scale, void* out, float* lse,
                                   void* workspace, size_t workspace_bytes, int32_t num_ctas, int32_t flags,
                                   int32_t* status, void* stream) {
  tv::clear_error();
  if (flags & TV_ATTN_ROPE_Q)
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_attn_verify: TV_ATTN_ROPE_Q belongs to tv_tree_attn_verify_rope");
  return tv::verify_impl(q, k_cache, v_cache, num_blocks, block_size, block_table, max_blocks, seq_lens, k_tree,
                         v_tree, mask, mask_bstride, B, N, Hq, Hkv, head_dim, dtype, scale, out, lse, workspace,
                         workspace_bytes, num_ctas, flags, nullptr, 0, status, stream);
}

extern "C" int tv_tree_attn_verify_rope(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
                                        int32_t block_size, const int32_t* block_table, int32_t max_blocks,
                                        const int32_t* seq_lens, const void* k_tree, const void* v_tree,
                                        const uint64_t* mask, int64_t mask_bstride, const float* cos_sin,
                                        int32_t max_pos, int32_t B, int32_t N, int32_t Hq, int32_t Hkv,
                                        int32_t head_dim, int32_t dtype, float scale, void* out, float* lse,
                                        void* workspace, size_t workspace_bytes, int32_t num_ctas, int32_t flags,
                                        int32_t* status, void* stream) {
  tv::clear_error();
  if (B > 0 && (!cos_sin || max_pos < 1))
    return tv::fail(TV_ERR_INVALID_ARG, "tv_tree_attn_verify_rope: needs the rotary table");
  return tv::verify_impl(q, k_cache, v_cache, num_blocks, block_size, block_table, max_blocks, seq_lens, k_tree,
                         v_tree, mask, mask_bstride, B, N, Hq, Hkv, head_dim, dtype, scale, out, lse, workspace,
                         workspace_bytes, num_ctas, flags | TV_ATTN_ROPE_Q, cos_sin, max_pos, status, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of tv_tree_attn_verify.
//
// Some callers cannot obtain device memory at the point where they verify a
// tree: a serving loop that reserves all of its memory at start-up and forbids
// allocation afterwards, a host runtime (another language, an embedded engine)
// that has no device allocator to hand, or code that must not call cudaMalloc
// because it can synchronise the device.  For them the split-KV scratch of the
// attention call (the tile plan and the partial outputs of split units) lives
// in one fixed array in device memory that this library defines, sized
// kStaticWorkspaceBytes on every GPU that loads the library, kept until the
// process exits.
// ---------------------------------------------------------------------------
namespace tv {
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;  // 32 MiB per device
__device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Identity of the current CUDA context (cuCtxGetId through the runtime's
// driver entry-point query), 0 when it cannot be had.  A device reset tears
// the primary context down and loads the module again, possibly at another
// address, and the new context has a new identity.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
unsigned long long current_context_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS) return id;
  return 0;
}

// Device address of g_static_workspace for the current device (the host-side
// name is only a stand-in for the device array), looked up once per device
// with that device current, and again if the device's context was replaced
// since (after a cudaDeviceReset the old address would be stale).
int static_workspace_ptr(void** out) {
  static std::mutex mu;
  static void* cached[64] = {};
  static unsigned long long cached_ctx[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(TV_ERR_UNSUPPORTED, "device id %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (!cached[dev] || (ctx != 0 && ctx != cached_ctx[dev])) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_static_workspace)");
    cached[dev] = ptr;
    cached_ctx[dev] = ctx != 0 ? ctx : current_context_id();
  }
  *out = cached[dev];
  return TV_OK;
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_tree_attn_static_workspace_bytes(void) { return tv::kStaticWorkspaceBytes; }

extern "C" int tv_tree_attn_verify_static(const void* q, const void* k_cache, const void* v_cache,
                                          int64_t num_blocks, int32_t block_size, const int32_t* block_table,
                                          int32_t max_blocks, const int32_t* seq_lens, const void* k_tree,
                                          const void* v_tree, const uint64_t* mask, int64_t mask_bstride, int32_t B,
                                          int32_t N, int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t dtype,
                                          float scale, void* out, float* lse, int32_t num_ctas, int32_t flags,
                                          int32_t* status, void* stream) {
  using namespace tv;
  clear_error();
  AttnConfig cfg;
  int st = attn_config(B, N, Hq, Hkv, head_dim, dtype, block_size, num_ctas, flags, &cfg);
  if (st) return st;
  if (B == 0) return TV_OK;
  if (num_ctas == 0) {
    // the widest grid (at most one wave) whose scratch fits the static array
    const int64_t per_cta = align256((int64_t)2 * cfg.RPG * head_dim * 4) + align256((int64_t)2 * cfg.RPG * 4) +
                            align256((int64_t)cfg.RPG * 4);
    const int64_t room = (int64_t)kStaticWorkspaceBytes - align256((int64_t)(cfg.U + 1) * 4) - 768;
    int fit = room > 0 ? (int)(room / per_cta) : 0;
    if (fit < 1)
      return fail(TV_ERR_WORKSPACE, "tv_tree_attn_verify_static: %d units need more than the %zu-byte static scratch",
                  cfg.U, kStaticWorkspaceBytes);
    num_ctas = cfg.P < fit ? cfg.P : fit;
    if ((st = attn_config(B, N, Hq, Hkv, head_dim, dtype, block_size, num_ctas, flags, &cfg))) return st;
  }
  if ((size_t)cfg.bytes > kStaticWorkspaceBytes)
    return fail(TV_ERR_WORKSPACE,
                "tv_tree_attn_verify_static: this shape and grid need %lld bytes of scratch, above the %zu-byte "
                "static maximum; pass a smaller num_ctas (or 0) or use tv_tree_attn_verify with a workspace",
                (long long)cfg.bytes, kStaticWorkspaceBytes);
  void* ws = nullptr;
  if ((st = static_workspace_ptr(&ws))) return st;
  return tv_tree_attn_verify(q, k_cache, v_cache, num_blocks, block_size, block_table, max_blocks, seq_lens, k_tree,
                             v_tree, mask, mask_bstride, B, N, Hq, Hkv, head_dim, dtype, scale, out, lse, ws,
                             kStaticWorkspaceBytes, num_ctas, flags & ~TV_ATTN_WORKSPACE_ZEROED, status, stream);
}
