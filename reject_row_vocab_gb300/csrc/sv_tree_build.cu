// Tree-verify inputs from parent lists ([E2D] §2.4, §3.4).
//
// One CTA per request builds: positions = seq_len + depth (the path depth, not
// the flattened index), the ancestor-or-self attention mask over the draft
// nodes, the retrieve index (request * N + node), and the first-child /
// next-sibling links that drive the verify walk (siblings in node-index
// order).  Depths come from pointer jumping in shared memory (log2 N rounds);
// each thread writes its node's mask row by walking its ancestor chain; the
// links come from one reverse pass over the nodes (the lowest-index child is
// the last one seen), which keeps the work per request linear in N.
//
//   [E2D] "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理"
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kBuildThreads = 256;

__global__ void __launch_bounds__(kBuildThreads) k_build_tree(const int32_t* parents, const int64_t* seq_lens,
                                                               int32_t N, int64_t* positions, uint8_t* mask,
                                                               int32_t* retrieve_index, int32_t* first_child,
                                                               int32_t* next_sibling, uint32_t* status) {
  __shared__ int32_t s_par[kMaxNodes];
  __shared__ int32_t s_up[kMaxNodes];     // pointer-jumping ancestor
  __shared__ int32_t s_depth[kMaxNodes];
  __shared__ int32_t s_first[kMaxNodes];
  __shared__ int s_bad;
  grid_dependency_wait();
  allow_dependents();
  const int b = blockIdx.x, t = threadIdx.x;
  const int64_t base = static_cast<int64_t>(b) * N;
  if (t == 0) s_bad = 0;
  __syncthreads();
  for (int i = t; i < N; i += kBuildThreads) {
    const int32_t p = parents[base + i];
    s_par[i] = p;
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) s_bad = 1;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  const int64_t sl = seq_lens ? seq_lens[b] : 0;
  // Depth by pointer jumping: after round r every node knows its 2^r-th ancestor
  // and the depth accumulated so far.
  for (int i = t; i < N; i += kBuildThreads) {
    s_up[i] = bad ? -1 : s_par[i];
    s_depth[i] = (bad || i == 0) ? 0 : 1;
  }
  __syncthreads();
  for (int span = 1; span < N && !bad; span <<= 1) {
    int32_t nu[kMaxNodes / kBuildThreads], nd[kMaxNodes / kBuildThreads];
    int k = 0;
    for (int i = t; i < N; i += kBuildThreads, ++k) {
      const int32_t u = s_up[i];
      nu[k] = u >= 0 ? s_up[u] : -1;
      nd[k] = s_depth[i] + (u >= 0 ? s_depth[u] : 0);
    }
    __syncthreads();
    k = 0;
    for (int i = t; i < N; i += kBuildThreads, ++k) {
      s_up[i] = nu[k];
      s_depth[i] = nd[k];
    }
    __syncthreads();
  }
  // Positions, retrieve index, mask rows.
  for (int i = t; i < N; i += kBuildThreads) {
    positions[base + i] = sl + s_depth[i];
    retrieve_index[base + i] = static_cast<int32_t>(base + i);
    uint8_t* row = mask + (base + i) * N;
    for (int j = 0; j < N; ++j) row[j] = 0;
    if (bad) {
      row[i] = 1;
    } else {
      for (int j = i; j != -1; j = s_par[j]) row[j] = 1;
    }
  }
  // Links: one reverse pass (node-index order among siblings).
  if (t == 0) {
    for (int i = 0; i < N; ++i) s_first[i] = -1;
    for (int i = N - 1; i >= 1 && !bad; --i) {
      const int32_t p = s_par[i];
      next_sibling[base + i] = s_first[p];
      s_first[p] = i;
    }
    next_sibling[base] = -1;
    if (bad)
      for (int i = 1; i < N; ++i) next_sibling[base + i] = -1;
    status[b] = bad ? kStBadTree : 0u;
  }
  __syncthreads();
  for (int i = t; i < N; i += kBuildThreads) first_child[base + i] = s_first[i];
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status_t spec_verify_build_tree(const int32_t* parents, const int64_t* seq_lens, int32_t batch,
                                              int32_t nodes, int64_t* positions, uint8_t* mask,
                                              int32_t* retrieve_index, int32_t* first_child,
                                              int32_t* next_sibling, uint32_t* status, cudaStream_t stream) {
  if (batch < 0 || nodes < 1 || nodes > kMaxNodes || batch > 65535) return SV_ERR_BAD_SHAPE;
  if (batch == 0) return SV_OK;
  if (!parents || !positions || !mask || !retrieve_index || !first_child || !next_sibling || !status)
    return SV_ERR_NULL_ARG;
  const cudaError_t e = launch_pdl(k_build_tree, dim3(static_cast<unsigned>(batch)), dim3(kBuildThreads), 0, stream,
                                   parents, seq_lens, nodes, positions, mask, retrieve_index, first_child,
                                   next_sibling, status);
  return e == cudaSuccess ? SV_OK : cuda_failure(e);
}
