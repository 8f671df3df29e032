// Host-side parts of libtreeverify: error state, device properties and the
// rank-path tree builder.
//
// tv_tree_build follows "Build the tree attention mask that verifies a draft
// tree in one pass", sections "The tree." and "The mask.": candidates are rank
// paths, duplicates collapse, nodes are numbered by (length, lexicographic)
// order after the root, every path's parent is the node of its one-shorter
// prefix (absent prefix -> rejected), depth is the path length and each node's
// ancestor row has its own bit and its ancestors' bits.
#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.h"

namespace tv {

namespace {
thread_local std::string g_last_error;
std::mutex g_dev_mu;
DeviceInfo g_dev_cache[64];
}  // namespace

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

void clear_error() { g_last_error.clear(); }

int cuda_fail(cudaError_t e, const char* what) {
  return fail(TV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int current_device_info(DeviceInfo* info) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(TV_ERR_UNSUPPORTED, "device id %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& c = g_dev_cache[dev];
  if (c.device != dev) {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.max_smem_optin = (size_t)v;
    c = d;
  }
  *info = c;
  return TV_OK;
}

}  // namespace tv

extern "C" const char* tv_last_error(void) { return tv::g_last_error.c_str(); }

extern "C" int tv_version(void) { return 202; }

extern "C" int tv_tree_build(const int32_t* ranks, const int32_t* offsets, int32_t n_paths,
                             int32_t max_nodes, int32_t* parent, int32_t* depth, uint64_t* mask,
                             int32_t* path_to_node, int32_t* n_nodes) {
  using tv::fail;
  tv::clear_error();
  if (n_paths < 0 || !offsets || !parent || !depth || !mask || !n_nodes)
    return fail(TV_ERR_INVALID_ARG, "tv_tree_build: null output or negative path count");
  if (max_nodes < 1 || max_nodes > TV_MAX_NODES)
    return fail(TV_ERR_INVALID_ARG, "tv_tree_build: max_nodes %d not in [1, %d]", max_nodes, TV_MAX_NODES);
  if (n_paths > 0 && !ranks && offsets[n_paths] > offsets[0])
    return fail(TV_ERR_INVALID_ARG, "tv_tree_build: null ranks");

  // 1. read and validate every path
  std::vector<std::vector<int32_t>> paths((size_t)n_paths);
  for (int32_t k = 0; k < n_paths; ++k) {
    int32_t a = offsets[k], b = offsets[k + 1];
    if (a < 0 || b < a) return fail(TV_ERR_INVALID_ARG, "tv_tree_build: offsets not non-decreasing at %d", k);
    for (int32_t t = a; t < b; ++t) {
      if (ranks[t] < 0) return fail(TV_ERR_INVALID_ARG, "tv_tree_build: negative rank in path %d", k);
      paths[(size_t)k].push_back(ranks[t]);
    }
  }

  // 2. distinct non-empty paths in (length, lexicographic) order
  std::vector<std::vector<int32_t>> order;
  order.reserve(paths.size());
  for (const auto& p : paths)
    if (!p.empty()) order.push_back(p);
  std::sort(order.begin(), order.end(), [](const std::vector<int32_t>& x, const std::vector<int32_t>& y) {
    if (x.size() != y.size()) return x.size() < y.size();
    return x < y;
  });
  order.erase(std::unique(order.begin(), order.end()), order.end());
  const int64_t n = 1 + (int64_t)order.size();
  if (n > max_nodes)
    return fail(TV_ERR_TOO_MANY_NODES, "tv_tree_build: %lld nodes exceed capacity %d", (long long)n, max_nodes);

  // 3. node ids, then parents (a missing prefix is an error)
  std::map<std::vector<int32_t>, int32_t> id;
  id[std::vector<int32_t>()] = 0;
  for (size_t k = 0; k < order.size(); ++k) id[order[k]] = (int32_t)(k + 1);
  parent[0] = -1;
  depth[0] = 0;
  for (size_t k = 0; k < order.size(); ++k) {
    std::vector<int32_t> up(order[k].begin(), order[k].end() - 1);
    auto it = id.find(up);
    if (it == id.end()) return fail(TV_ERR_MISSING_PARENT, "tv_tree_build: missing parent for a path of length %zu", order[k].size());
    parent[k + 1] = it->second;
    depth[k + 1] = (int32_t)order[k].size();
  }

  // 4. ancestor rows: own bit plus the parent's row (parents precede children)
  for (int64_t i = 0; i < n; ++i) mask[i] = (i == 0 ? 0ull : mask[parent[i]]) | (1ull << i);

  if (path_to_node)
    for (int32_t k = 0; k < n_paths; ++k) path_to_node[k] = id[paths[(size_t)k]];
  *n_nodes = (int32_t)n;
  return TV_OK;
}
