// DSpark verify-length scheduling ([E2D] §5.6.3 and §5.6.4).
//
// Host: the extra draft budget K* = argmax_K (R + a_1 + ... + a_K) * SPS(R + K)
// over historical survival scores sorted in descending order (§5.6.3).
// Device: the budget goes to the current best (request, position) candidates,
// ordered by survival descending, then position ascending, then request
// ascending (§5.6.4); verify_len = 1 anchor + the request's selected drafts.
//
// The device ranking counts, for every candidate, how many candidates come
// before it in that order (a strict total order, so ranks are a permutation);
// a candidate is selected when its rank is below the budget.  Each CTA ranks
// 32 candidates: its eight warps split the comparisons and add their counts.
// A second kernel turns the per-request counts into lengths and clears them.
//
//   [E2D] "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理"
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kRankWarps = 8;

// Sort key of a candidate: smaller keys order first.  The high word is the
// survival in descending order (NaN as -inf), the low word position * R +
// request (position first, then request); R * D <= 2^30 keeps it in 32 bits.
__device__ __forceinline__ uint64_t candidate_key(float s, int32_t pos, int32_t req, int32_t R) {
  if (s != s) s = -kInfF;
  const uint32_t b = __float_as_uint(s);
  const uint32_t asc = (b & 0x80000000u) ? ~b : (b | 0x80000000u);  // order-preserving
  return (static_cast<uint64_t>(~asc) << 32) | static_cast<uint32_t>(pos * R + req);
}

__global__ void __launch_bounds__(32 * kRankWarps) k_dspark_rank(const float* survival, int32_t R, int32_t D,
                                                                  int64_t ld, int32_t budget, float eps,
                                                                  uint32_t* count) {
  __shared__ uint32_t s_part[kRankWarps][32];
  grid_dependency_wait();
  allow_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n = static_cast<int64_t>(R) * D;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * 32 + lane;  // this lane's candidate
  const bool valid = e < n;
  const int32_t er = valid ? static_cast<int32_t>(e / D) : 0;
  const int32_t ep = valid ? static_cast<int32_t>(e - static_cast<int64_t>(er) * D) : 0;
  const float es = valid ? survival[er * ld + ep] : 0.0f;
  const uint64_t ek = candidate_key(es, ep, er, R);
  // Warp w compares against candidates [w * n / 8, (w + 1) * n / 8), 32 at a time.
  const int64_t j0 = warp * n / kRankWarps, j1 = (warp + 1) * n / kRankWarps;
  uint32_t before = 0;
  for (int64_t jb = j0; jb < j1; jb += 32) {
    const int64_t j = jb + lane;
    uint64_t jk = ~0ull;  // past the end: orders after everything, never counted
    if (j < j1) {
      const int32_t jr = static_cast<int32_t>(j / D);
      const int32_t jp = static_cast<int32_t>(j - static_cast<int64_t>(jr) * D);
      jk = candidate_key(survival[jr * ld + jp], jp, jr, R);
    }
#pragma unroll 8
    for (int t = 0; t < 32; ++t) before += __shfl_sync(0xffffffffu, jk, t) < ek ? 1u : 0u;
  }
  s_part[warp][lane] = before;
  __syncthreads();
  if (warp == 0 && valid) {
    uint32_t rank = 0;
#pragma unroll
    for (int w = 0; w < kRankWarps; ++w) rank += s_part[w][lane];
    if (rank < static_cast<uint32_t>(budget) && es >= eps) atomicAdd(&count[er], 1u);  // NaN fails >=
  }
}

__global__ void k_dspark_lens(int32_t R, int32_t min_len, int32_t max_len, uint32_t* count, int32_t* verify_lens) {
  grid_dependency_wait();  // the counts of k_dspark_rank
  allow_dependents();
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const int64_t v = 1 + static_cast<int64_t>(count[r]);
  verify_lens[r] = static_cast<int32_t>(v < min_len ? min_len : (v > max_len ? max_len : v));
  count[r] = 0u;  // leave the workspace clean for the next call
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_dspark_workspace_bytes(int32_t num_requests) {
  const size_t n = num_requests > 0 ? static_cast<size_t>(num_requests) : 1;
  return (n * sizeof(uint32_t) + 255) / 256 * 256;
}

sv_status_t spec_verify_dspark_budget(const float* hist_survival, int64_t n, int32_t num_requests, const float* sps,
                                      int32_t sps_len, float eps, int32_t* k_star) {
  if (!k_star || (n > 0 && !hist_survival) || (sps_len > 0 && !sps)) return SV_ERR_NULL_ARG;
  if (n < 0 || num_requests < 0 || sps_len < 0) return SV_ERR_BAD_SHAPE;
  std::vector<double> a;
  a.reserve(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) {
    const float x = hist_survival[i];
    if (!std::isnan(x) && x >= eps) a.push_back(x);
  }
  std::sort(a.begin(), a.end(), [](double x, double y) { return x > y; });
  int32_t best_k = 0;
  double best = -INFINITY, n_hat = num_requests;
  for (size_t k = 0; k <= a.size(); ++k) {
    if (k > 0) n_hat += a[k - 1];
    const int64_t m = static_cast<int64_t>(num_requests) + static_cast<int64_t>(k);
    if (m >= sps_len) break;
    const double score = n_hat * static_cast<double>(sps[m]);
    if (score > best) {
      best = score;
      best_k = static_cast<int32_t>(k);
    }
  }
  *k_star = best_k;
  return SV_OK;
}

sv_status_t spec_verify_dspark_verify_lens(const float* survival, int32_t num_requests, int32_t num_drafts,
                                           int64_t ld, int32_t budget, int32_t min_len, int32_t max_len, float eps,
                                           int32_t* verify_lens, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (num_requests < 0 || num_drafts < 0 || budget < 0 || ld < num_drafts || min_len < 1 || max_len < min_len)
    return SV_ERR_BAD_SHAPE;
  const int64_t n = static_cast<int64_t>(num_requests) * num_drafts;
  if (n > (int64_t{1} << 30)) return SV_ERR_BAD_SHAPE;
  if (num_requests == 0) return SV_OK;
  if (!verify_lens || (n > 0 && !survival)) return SV_ERR_NULL_ARG;
  if (!ws || ws_bytes < spec_verify_dspark_workspace_bytes(num_requests) || (reinterpret_cast<uintptr_t>(ws) & 255))
    return SV_ERR_WORKSPACE_TOO_SMALL;
  uint32_t* count = static_cast<uint32_t*>(ws);
  cudaError_t e = cudaSuccess;
  if (n > 0) {
    e = launch_pdl(k_dspark_rank, dim3(static_cast<unsigned>((n + 31) / 32)), dim3(32 * kRankWarps), 0, stream,
                   survival, num_requests, num_drafts, ld, budget, eps, count);
    if (e != cudaSuccess) return cuda_failure(e);
  }
  e = launch_pdl(k_dspark_lens, dim3(static_cast<unsigned>((num_requests + 255) / 256)), dim3(256), 0, stream,
                 num_requests, min_len, max_len, count, verify_lens);
  return e == cudaSuccess ? SV_OK : cuda_failure(e);
}

}  // extern "C"
