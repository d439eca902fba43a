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
//   * the first call in each CUDA context (per device, and again after a
//     device reset) looks up the area's device address
//     (cudaGetSymbolAddress), so make that first call before any stream
//     capture starts;
//   * all calls share the area and it keeps the previous call's contents, so
//     each call clears the counter words it relies on (after its argument
//     checks, on its stream) before launching, and calls that overlap on the
//     GPU (other streams, other host threads) race.
#include <cuda.h>  // driver types only: the two driver calls below come through the runtime's entry-point query

#include <cstdint>
#include <mutex>

#include "sv_internal.h"

// The fixed scratch area.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Device addresses of the area, one per CUDA context that used it.  A context
// id is unique for the life of the process, so after a device reset (a new
// primary context, the library's module loaded again) the address is looked up
// again instead of reusing one from the destroyed context.
struct AddrEntry {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kMaxContexts = 64;
std::mutex g_addr_mu;
AddrEntry g_addr[kMaxContexts];
int g_addr_n = 0;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

cudaError_t driver_calls() {
  if (g_ctx_current && g_ctx_id) return cudaSuccess;
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q{};
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) return e != cudaSuccess ? e : cudaErrorNotSupported;
  g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f);
  f = nullptr;
  e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) return e != cudaSuccess ? e : cudaErrorNotSupported;
  g_ctx_id = reinterpret_cast<CtxGetIdFn>(f);
  return cudaSuccess;
}

// Id of the calling thread's current context (the runtime's primary context
// of the current device once any runtime call has touched it).
cudaError_t current_context_id(unsigned long long* id) {
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (!ctx) {  // no context made current on this thread yet: let the runtime set up its primary context
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorUnknown;
  }
  return g_ctx_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// Device address of the scratch area in the current context (looked up once per context).
cudaError_t scratch_address(void** addr) {
  std::lock_guard<std::mutex> lock(g_addr_mu);
  cudaError_t e = driver_calls();
  if (e != cudaSuccess) return e;
  unsigned long long id = 0;
  if ((e = current_context_id(&id)) != cudaSuccess) return e;
  for (int i = 0; i < g_addr_n; ++i)
    if (g_addr[i].ctx_id == id) {
      *addr = g_addr[i].addr;
      return cudaSuccess;
    }
  void* p = nullptr;
  if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return e;
  if (g_addr_n == kMaxContexts) g_addr_n = 0;  // many resets: start the table over
  g_addr[g_addr_n++] = AddrEntry{id, p};
  *addr = p;
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
  // Argument errors need no device: answer them before the first CUDA call.  Given no workspace, the shared
  // path stops at its workspace check, which follows every argument check and precedes every CUDA call, so
  // SV_ERR_WORKSPACE_TOO_SMALL here means the arguments passed.
  const sv_status_t pre = sv::rejection_chain_entry(logits, dtype, ld, batch, m, vocab, verify_ids, q, ldq,
                                                    temperature, u_accept, u_final, row_slots, seq_lens, out,
                                                    nullptr, 0, stream, false);
  if (pre != SV_ERR_WORKSPACE_TOO_SMALL) return pre;  // an argument error, or an empty batch (done)
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SV_ERR_CUDA;
  return sv::rejection_chain_entry(logits, dtype, ld, batch, m, vocab, verify_ids, q, ldq, temperature, u_accept,
                                   u_final, row_slots, seq_lens, out, scratch, SV_NOALLOC_SCRATCH_BYTES, stream,
                                   true);
}

extern "C" sv_status_t spec_verify_noalloc_fill_counters(uint32_t value, cudaStream_t stream) {
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SV_ERR_CUDA;
  const size_t n = sv::ws_layout(1, 1, 1, 1).counters_end;
  return cudaMemsetAsync(scratch, static_cast<int>(value & 0xffu), n, stream) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
