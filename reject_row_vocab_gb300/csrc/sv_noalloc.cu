// p/q rejection chain verification for callers that cannot hand the library
// any scratch memory.
//
// The regular entry points take a caller-allocated workspace.  Some callers
// have no way to provide one: a plugin that its host framework gives only
// input and output buffers, code running after a serving engine has reserved
// all device memory for itself up front, or an embedding where allocating is
// not allowed at call time (a device allocation can synchronise the device).
// For them this file keeps one fixed scratch area in the library's own device
// image and runs the unchanged rejection-chain kernels on it.
//
// Rules that follow from sharing one fixed area:
//   * its size is SV_NOALLOC_SCRATCH_BYTES; larger problems are rejected;
//   * every GPU on which the library is used holds the area until the process
//     exits;
//   * the first call on a device looks up the area's device address
//     (cudaGetSymbolAddress), so make that first call before any stream
//     capture starts;
//   * all calls share the area and it keeps the previous call's contents, so
//     each call clears the counter words it relies on before launching, and
//     calls that overlap on the GPU (other streams, other host threads) race.
#include <cstdint>
#include <mutex>

#include "sv_internal.h"

// The fixed scratch area.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_addr_mu;
void* g_addr[64];
bool g_addr_ready[64];

// Device address of the scratch area on the current device (looked up once per device).
cudaError_t scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  if (!g_addr_ready[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
    g_addr_ready[dev] = true;
  }
  *addr = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" sv_status_t spec_verify_rejection_chain_noalloc(
    const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t m, int32_t vocab,
    const int32_t* verify_ids, const float* q, int64_t ldq, const float* temperature, const float* u_accept,
    const float* u_final, const int64_t* row_slots, const int64_t* seq_lens, const sv_out_t* out,
    cudaStream_t stream) {
  if (batch < 0 || m < 0 || m >= (1 << 20) || vocab < 1) return SV_ERR_BAD_SHAPE;
  const int64_t rows = static_cast<int64_t>(batch) * (m + 1);
  const sv::WsLayout layout = sv::ws_layout(rows, batch, vocab, m + 1);
  if (layout.total > SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SV_ERR_CUDA;
  if (batch > 0 && cudaMemsetAsync(scratch, 0, layout.counters_end, stream) != cudaSuccess) return SV_ERR_CUDA;
  return spec_verify_rejection_chain(logits, dtype, ld, batch, m, vocab, verify_ids, q, ldq, temperature, u_accept,
                                     u_final, row_slots, seq_lens, out, scratch, SV_NOALLOC_SCRATCH_BYTES, stream);
}
