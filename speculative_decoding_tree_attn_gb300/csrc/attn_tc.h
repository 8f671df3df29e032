// Interface of the tcgen05 tree-attention kernel (attn_tc.cu) used by the
// dispatcher in attn.cu.
#pragma once

#include "attn_common.cuh"

namespace tv {

constexpr int kTcBlk = 64;       // keys per tile (MMA N of S, K of P V)
constexpr int kTcMaxRows = 256;  // two 128-row M tiles per CTA (more rows: row groups)

// True when the tensor-core kernel can run this shape on this device:
// bf16, head_dim 128, rows = G * N <= 512, G divides 128, block_size a
// multiple of 16 that divides 64 or is a multiple of 64; with rope (Q rotated
// as it is loaded) also G in {4, 8, 16}.
bool tc_supported(const DeviceInfo& dev, int dtype, int head_dim, int rows, int G, int block_size, bool rope);

// Why the shape is rejected (nullptr when it is supported).
const char* tc_unsupported_reason(const DeviceInfo& dev, int dtype, int head_dim, int rows, int G, int block_size,
                                  bool rope);

// Rows per unit for `rows` = G * N query rows per KV head: 128, 256, or all
// of them when they exceed 256 by at most 8 (those tail rows are computed
// beside the two M tiles, so the unit's K/V is read once).
int tc_rows_per_unit(int rows);

// Resident CTAs per SM the kernel is built for at this row count.
int tc_ctas_per_sm(int rows);

// Virtual tiles the plan charges per unit for this kernel (see AttnParams).
int tc_unit_cost(int rows_per_unit);

// CTA pairs the CTA-pair kernel keeps resident at once on this device.
int tc_duo_pairs(const DeviceInfo& dev);

// Launches the persistent tensor-core kernel; with `duo`, units of 129-256
// rows run on CTA pairs (p.P = pairs).
int launch_attn_tc(const AttnParams& p, int32_t* status, cudaStream_t stream, bool duo);

}  // namespace tv
