// Work decomposition shared by the tree-attention kernels and the combine.
//
// Units also carry `unit_cost` virtual tiles placed before their real ones: a
// kernel pays a fixed cost at every unit it starts or finishes (epilogue,
// loading the next queries), so a CTA whose slice crosses many short units is
// given fewer real tiles.  A unit's real tiles are [tile_start[u] + unit_cost,
// tile_start[u + 1]).
//
// A "unit" is one (request b, KV head, row group): the rows of a unit are the
// (node, query head) pairs of one GQA group, row r = node * G + g.  A unit's
// work is a sequence of KV tiles: ceil(L_b / BLK) prefix tiles followed by one
// tree tile holding the N tree nodes.  All units' tiles are laid end to end
// (exclusive prefix sums in tile_start[]) and the persistent grid of P CTAs
// takes equal contiguous slices [c*T/P, (c+1)*T/P) of that sequence, so every
// CTA streams the same number of KV tiles whatever the prefix lengths.  A unit
// cut by a slice boundary is "split": each CTA writes a normalised partial
// output and its log2-sum-exp to one of its two slots (0 = the CTA's first
// unit, 1 = its last) and the combine kernel merges the pieces.  Units inside
// one slice are written to the output directly.
//
// The CUDA-core kernel reads the plan from tile_start[] (filled by the plan
// kernel) and leaves split units to the combine kernel.  The tcgen05 kernels
// derive their slice from seq_lens themselves (all units of one request have
// the same tile count, so the prefix sums run over requests) and merge split
// units in their own epilogue: each piece counts its real tiles into a per-row
// arrival counter, and the piece that brings the count to the unit's total
// merges that row.
#pragma once

#include <cstdint>

#include "common.h"

namespace tv {

struct AttnParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const void* k_tree;
  const void* v_tree;
  const uint64_t* mask;
  int64_t mask_bstride;
  void* out;
  float* lse;
  int32_t* tile_start;  // [U + 1]
  float* part_o;        // [P][2][RPG][D]
  float* part_lse;      // [P][2][RPG]
  uint32_t* arrive;     // [P][RPG] arrival counters of split units, by first CTA (tcgen05 kernels)
  int64_t num_blocks;
  int block_size;
  int max_blocks;
  int B, N, Hq, Hkv, D, G;
  int R;    // rows per (b, kv head) = G * N
  int RPG;  // rows per unit
  int RG;   // row groups per (b, kv head)
  int U;    // number of units
  int BLK;  // KV positions per tile
  int P;    // persistent CTAs
  int unit_cost;  // extra virtual tiles charged per unit (its fixed start/finish cost)
  int direct_merge;  // tcgen05: the last piece may merge straight from its accumulator
  const float* rope_cs;  // non-null: Q arrives unrotated and is rotated as it is loaded, at
                         // L_b + depth (depth from the ancestor row), with this cos/sin table
  int rope_max_pos;      // rows of rope_cs
  int32_t* status;       // device status word (nullable), TV_DEV_* bits
  float scale_log2;  // softmax scale * log2(e)
};

__host__ __device__ inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Prefix length, clamped to what the block table can address.
__device__ __forceinline__ int clamp_len(const AttnParams& p, int b) {
  int L = p.seq_lens[b];
  const int cap = p.max_blocks * p.block_size;
  return L < 0 ? 0 : (L > cap ? cap : L);
}

__device__ __forceinline__ void unit_coords(const AttnParams& p, int u, int& b, int& kvh, int& rg) {
  rg = u % p.RG;
  kvh = (u / p.RG) % p.Hkv;
  b = u / (p.RG * p.Hkv);
}

// First tile index of CTA c.
__device__ __forceinline__ int64_t cta_start(int64_t c, int64_t T, int64_t P) { return c * T / P; }

// The CTA whose slice contains tile t (largest c with cta_start(c) <= t).
__device__ __forceinline__ int64_t cta_of(int64_t t, int64_t T, int64_t P) { return ((t + 1) * P - 1) / T; }

// Unit containing tile t: largest u with tile_start[u] <= t.
__device__ __forceinline__ int find_unit(const int32_t* tile_start, int U, int64_t t) {
  int lo = 0, hi = U - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Launches the single-CTA plan kernel that fills tile_start.
int launch_plan(const AttnParams& p, cudaStream_t stream);

// Launches the merge of split units (one CTA per unit; unsplit units exit).
int launch_combine(const AttnParams& p, int dtype, cudaStream_t stream);

}  // namespace tv
