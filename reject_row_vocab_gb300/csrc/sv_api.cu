// C ABI of libspecverify: argument validation, workspace carving and the
// launch sequence of each entry point.  Nothing here reads device memory or
// synchronises; every kernel is enqueued on the caller's stream.
//
// Launch sequences (each kernel chained to the previous one by programmatic
// dependent launch):
//   greedy chain / tree:          row stats -> row merge -> accept -> commit
//     (batches of at most 32:     row stats -> row merge -> accept and commit in one CTA)
//   rejection chain / ragged,
//   sparse q, sample-then-match:  row stats -> row merge -> accept -> sample (tile sums; an extra block
//                                 commits) -> draw
//   target-only tree:             row stats -> row merge -> accept (tree walk) -> sample -> draw
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "sv_internal.h"

namespace sv {

cudaError_t device_info(DeviceInfo* info) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    DeviceInfo d{};
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = stats_occupancy(SV_F32, &d.stats_blocks_per_sm[0]);
    if (e != cudaSuccess) return e;
    e = stats_occupancy(SV_BF16, &d.stats_blocks_per_sm[1]);
    if (e != cudaSuccess) return e;
    e = sample_smem_setup();
    if (e != cudaSuccess) return e;
    e = accept_smem_setup();
    if (e != cudaSuccess) return e;
    if (d.stats_blocks_per_sm[0] < 1) d.stats_blocks_per_sm[0] = 1;
    if (d.stats_blocks_per_sm[1] < 1) d.stats_blocks_per_sm[1] = 1;
    cache[dev] = d;
    have[dev] = true;
  }
  *info = cache[dev];
  return cudaSuccess;
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

sv_status_t check_logits(const void* logits, sv_dtype_t dt, int64_t ld, int64_t rows, int32_t vocab) {
  if (!logits) return SV_ERR_NULL_ARG;
  if (dt != SV_F32 && dt != SV_BF16) return SV_ERR_BAD_DTYPE;
  if (vocab < 1 || rows < 0 || rows > INT32_MAX || ld < vocab) return SV_ERR_BAD_SHAPE;
  const int64_t es = dt == SV_BF16 ? 2 : 4;
  if (!aligned(logits, 16) || (ld * es) % 16 != 0) return SV_ERR_MISALIGNED;
  return SV_OK;
}

sv_status_t check_q(const float* q, int64_t ldq, int32_t vocab) {
  if (!q) return SV_ERR_NULL_ARG;
  if (ldq < vocab) return SV_ERR_BAD_SHAPE;
  if (!aligned(q, 16) || (ldq * 4) % 16 != 0) return SV_ERR_MISALIGNED;
  return SV_OK;
}

sv_status_t check_out(const sv_out_t* out, const int64_t* row_slots, const int64_t* seq_lens) {
  if (!out) return SV_ERR_NULL_ARG;
  if (!out->accept_len || !out->num_out || !out->out_tokens || !out->bonus || !out->accept_rows ||
      !out->commit_cu || !out->dev_status)
    return SV_ERR_NULL_ARG;
  if (out->commit_src_slot && !row_slots) return SV_ERR_NULL_ARG;
  if (out->commit_dst_pos && !seq_lens) return SV_ERR_NULL_ARG;
  return SV_OK;
}

sv_status_t carve(void* ws, size_t ws_bytes, int64_t rows, int32_t batch, int32_t vocab, int32_t max_len, Ws* w) {
  const WsLayout L = ws_layout(rows, batch, vocab, max_len);
  if (!ws || ws_bytes < L.total || !aligned(ws, 256)) return SV_ERR_WORKSPACE_TOO_SMALL;
  char* base = static_cast<char*>(ws);
  w->done_cnt = reinterpret_cast<uint32_t*>(base + L.done_cnt);
  w->err = w->done_cnt + 1;
  w->rowstat = reinterpret_cast<RowStat*>(base + L.rowstat);
  w->partial = reinterpret_cast<RowPartial*>(base + L.partial);
  w->psb = reinterpret_cast<float*>(base + L.psb);
  w->ureq = reinterpret_cast<float*>(base + L.ureq);
  w->state = reinterpret_cast<ReqState*>(base + L.state);
  w->excl = reinterpret_cast<int32_t*>(base + L.excl);
  w->tsum = reinterpret_cast<uint64_t*>(base + L.tsum);
  w->ntiles = L.ntiles;
  return SV_OK;
}

OutView out_view(const sv_out_t* o) {
  return OutView{o->accept_len, o->num_out,       o->out_tokens,     o->bonus,     o->accept_rows,
                 o->commit_cu,  o->commit_src_slot, o->commit_dst_pos, o->dev_status};
}

sv_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

// Optional benchmark instrumentation: events recorded around the row-statistics kernel.
thread_local cudaEvent_t t_stats_start = nullptr;
thread_local cudaEvent_t t_stats_stop = nullptr;


cudaError_t row_stats_timed(const LogitsView& lg, const RowMap& map, const Ws& w, int grid, cudaStream_t stream,
                            const int32_t* probe = nullptr, int32_t probe_rpr = 0) {
  cudaError_t e;
  if (t_stats_start && (e = record_event(t_stats_start, stream)) != cudaSuccess) return e;
  return launch_row_stats(lg, map, w, grid, stream, probe, probe_rpr, t_stats_stop);
}

// An empty batch commits nothing: commit_cu = [0].  Every other pointer may be NULL.
sv_status_t empty_batch(const sv_out_t* out, cudaStream_t stream) {
  if (!out || !out->commit_cu) return SV_ERR_NULL_ARG;
  return cuda_status(cudaMemsetAsync(out->commit_cu, 0, sizeof(int32_t), stream));
}

#define SV_TRY(expr)                      \
  do {                                    \
    const sv_status_t _s = (expr);        \
    if (_s != SV_OK) return _s;           \
  } while (0)
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

#define SV_TRY_CUDA(expr)                 \
  do {                                    \
    const cudaError_t _e = (expr);        \
    if (_e != cudaSuccess) {              \
      t_last_cuda_error = _e;             \
      return SV_ERR_CUDA;                 \
    }                                     \
  } while (0)

}  // namespace

// While a stream is being captured into a graph, an external record becomes an
// event node of the graph; otherwise a plain record.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
  return cudaEventRecord(ev, stream);
}

sv_status_t cuda_failure(cudaError_t e) {
  t_last_cuda_error = e;
  return SV_ERR_CUDA;
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_bytes(int64_t rows, int32_t batch, int32_t vocab, int32_t max_len) {
  return ws_layout(rows, batch, vocab, max_len).total;
}

sv_status_t spec_verify_set_stats_events(cudaEvent_t start, cudaEvent_t stop) {
  if ((start == nullptr) != (stop == nullptr)) return SV_ERR_NULL_ARG;
  t_stats_start = start;
  t_stats_stop = stop;
  return SV_OK;
}

const char* spec_verify_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda_error); }

const char* spec_verify_status_string(sv_status_t status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_NULL_ARG: return "a required pointer is NULL";
    case SV_ERR_BAD_SHAPE: return "a size, stride or scalar argument is out of range";
    case SV_ERR_BAD_DTYPE: return "unsupported logits dtype";
    case SV_ERR_MISALIGNED: return "a base pointer or row stride is not 16-byte aligned";
    case SV_ERR_UNSUPPORTED: return "unsupported combination of arguments";
    case SV_ERR_WORKSPACE_TOO_SMALL: return "workspace missing, too small or not 256-byte aligned";
    case SV_ERR_CUDA: return "a CUDA launch or device query failed";
  }
  return "unknown status";
}

sv_status_t spec_verify_greedy_chain(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t m,
                                     int32_t vocab, const int32_t* verify_ids, const int64_t* row_slots,
                                     const int64_t* seq_lens, const sv_out_t* out, void* ws, size_t ws_bytes,
                                     cudaStream_t stream) {
  if (batch < 0 || m < 0 || m >= (1 << 20)) return SV_ERR_BAD_SHAPE;
  if (batch == 0) return empty_batch(out, stream);
  const int64_t rows = static_cast<int64_t>(batch) * (m + 1);
  SV_TRY(check_logits(logits, dtype, ld, rows, vocab));
  if (!verify_ids) return SV_ERR_NULL_ARG;
  SV_TRY(check_out(out, row_slots, seq_lens));
  Ws w{};
  SV_TRY(carve(ws, ws_bytes, rows, batch, vocab, m + 1, &w));
  DeviceInfo dev{};
  SV_TRY_CUDA(device_info(&dev));
  const LogitsView lg{logits, dtype, ld, rows, vocab};
  SV_TRY_CUDA(row_stats_timed(lg, RowMap{kMapGreedy, m + 1, batch, nullptr, nullptr}, w, stats_grid(dev, lg), stream));
  ChainParams p{lg,      batch,   m + 1,   m + 1,   nullptr, verify_ids, nullptr, 0,
                nullptr, nullptr, nullptr, nullptr, nullptr, 0,          0,       0};
  const OutView ov = out_view(out);
  const CommitParams cp{batch, m + 1, row_slots, seq_lens, w.err};
  if (accept_commit_fits(batch, 0)) {  // one CTA finishes and commits a small batch
    SV_TRY_CUDA(launch_accept_commit_chain(p, ov, cp, w, stream));
  } else {
    SV_TRY_CUDA(launch_accept_chain(p, ov, w, stream));
    SV_TRY_CUDA(launch_commit(ov, cp, stream));
  }
  return SV_OK;
}

static sv_status_t rejection_common(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int64_t rows,
                                    int32_t max_len, int32_t fixed_len, int32_t vocab, const int32_t* cu,
                                    const int32_t* verify_ids, const float* q, int64_t ldq,
                                    const float* temperature, const float* u_accept, const float* u_final,
                                    const int64_t* row_slots, const int64_t* seq_lens, const sv_out_t* out,
                                    void* ws, size_t ws_bytes, cudaStream_t stream, const int32_t* cand_ids = nullptr,
                                    const float* cand_probs = nullptr, int32_t num_cands = 0, int64_t ldc = 0,
                                    bool clear_counters = false) {
  if (batch > 65535) return SV_ERR_BAD_SHAPE;  // the sampler's grid has one y-slice per request
  if (batch == 0) return empty_batch(out, stream);
  SV_TRY(check_logits(logits, dtype, ld, rows, vocab));
  if (!verify_ids || !temperature || !u_accept || !u_final) return SV_ERR_NULL_ARG;
  if (fixed_len == 0 && !cu) return SV_ERR_NULL_ARG;
  if (cand_ids) {  // sparse q: candidate lists instead of dense rows
    if (!cand_probs) return SV_ERR_NULL_ARG;
    if (num_cands < 1 || num_cands > kMaxCands || ldc < num_cands) return SV_ERR_BAD_SHAPE;
  } else {
    SV_TRY(check_q(q, ldq, vocab));
  }
  SV_TRY(check_out(out, row_slots, seq_lens));
  Ws w{};
  SV_TRY(carve(ws, ws_bytes, rows, batch, vocab, max_len, &w));
  w.cand_id = cand_ids;  // the final draws read the residual row's list in place
  w.cand_q = cand_probs;
  w.cand_ld = ldc;
  DeviceInfo dev{};
  SV_TRY_CUDA(device_info(&dev));
  if (clear_counters)
    SV_TRY_CUDA(cudaMemsetAsync(w.done_cnt, 0, ws_layout(rows, batch, vocab, max_len).counters_end, stream));
  const LogitsView lg{logits, dtype, ld, rows, vocab};
  const OutView ov = out_view(out);
  if (rows > 0) {
    const RowMap map = fixed_len > 0 ? RowMap{kMapFixed, fixed_len, batch, nullptr, temperature}
                                     : RowMap{kMapCu, 0, batch, cu, temperature};
    SV_TRY_CUDA(row_stats_timed(lg, map, w, stats_grid(dev, lg), stream));
  }
  ChainParams p{lg,       batch,    max_len,  fixed_len, cu,        verify_ids, q,  ldq,
                temperature, u_accept, u_final, cand_ids, cand_probs, num_cands, ldc, 0};
  SV_TRY_CUDA(launch_accept_chain(p, ov, w, stream));
  SV_TRY_CUDA(launch_sample_and_commit(lg, q, ldq, u_final, ov, CommitParams{batch, max_len, row_slots, seq_lens, w.err},
                                       w, dev, stream, cand_ids != nullptr));
  return SV_OK;
}

sv_status_t spec_verify_rejection_chain(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t m,
                                        int32_t vocab, const int32_t* verify_ids, const float* q, int64_t ldq,
                                        const float* temperature, const float* u_accept, const float* u_final,
                                        const int64_t* row_slots, const int64_t* seq_lens, const sv_out_t* out,
                                        void* ws, size_t ws_bytes, cudaStream_t stream) {
  return rejection_chain_entry(logits, dtype, ld, batch, m, vocab, verify_ids, q, ldq, temperature, u_accept,
                               u_final, row_slots, seq_lens, out, ws, ws_bytes, stream, false);
}

sv_status_t spec_verify_set_hand_off_limit_ns(uint64_t ns) {
  set_hand_off_limit_ns(ns);
  return SV_OK;
}

}  // extern "C"

namespace sv {
sv_status_t rejection_chain_entry(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t m,
                                  int32_t vocab, const int32_t* verify_ids, const float* q, int64_t ldq,
                                  const float* temperature, const float* u_accept, const float* u_final,
                                  const int64_t* row_slots, const int64_t* seq_lens, const sv_out_t* out, void* ws,
                                  size_t ws_bytes, cudaStream_t stream, bool clear_counters) {
  if (batch < 0 || m < 0 || m >= (1 << 20)) return SV_ERR_BAD_SHAPE;
  const int64_t rows = static_cast<int64_t>(batch) * (m + 1);
  return rejection_common(logits, dtype, ld, batch, rows, m + 1, m + 1, vocab, nullptr, verify_ids, q, ldq,
                          temperature, u_accept, u_final, row_slots, seq_lens, out, ws, ws_bytes, stream, nullptr,
                          nullptr, 0, 0, clear_counters);
}
}  // namespace sv

extern "C" {

sv_status_t spec_verify_sample_match_chain(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                           int32_t m, int32_t vocab, const int32_t* verify_ids,
                                           const float* temperature, const float* u_sample, const int64_t* row_slots,
                                           const int64_t* seq_lens, const sv_out_t* out, void* ws, size_t ws_bytes,
                                           cudaStream_t stream) {
  if (batch < 0 || m < 0 || m >= (1 << 20) || batch > 65535) return SV_ERR_BAD_SHAPE;
  if (batch == 0) return empty_batch(out, stream);
  const int64_t rows = static_cast<int64_t>(batch) * (m + 1);
  SV_TRY(check_logits(logits, dtype, ld, rows, vocab));
  if (!verify_ids || !temperature || !u_sample) return SV_ERR_NULL_ARG;
  SV_TRY(check_out(out, row_slots, seq_lens));
  Ws w{};
  SV_TRY(carve(ws, ws_bytes, rows, batch, vocab, m + 1, &w));
  DeviceInfo dev{};
  SV_TRY_CUDA(device_info(&dev));
  const LogitsView lg{logits, dtype, ld, rows, vocab};
  const OutView ov = out_view(out);
  // probe[row] = verify_ids[row + 1]: the draft each row tests (the last row of a request tests none)
  SV_TRY_CUDA(row_stats_timed(lg, RowMap{kMapFixed, m + 1, batch, nullptr, temperature}, w, stats_grid(dev, lg),
                              stream, verify_ids + 1, m + 1));
  ChainParams p{lg,       batch,    m + 1,   m + 1,   nullptr, verify_ids, nullptr, 0,
                temperature, u_sample, u_sample, nullptr, nullptr, 0,        0,       1};
  SV_TRY_CUDA(launch_accept_chain(p, ov, w, stream));
  SV_TRY_CUDA(launch_sample_and_commit(lg, nullptr, 0, w.ureq, ov,
                                       CommitParams{batch, m + 1, row_slots, seq_lens, w.err}, w, dev, stream));
  return SV_OK;
}

size_t spec_verify_sparse_workspace_bytes(int64_t rows, int32_t batch, int32_t vocab, int32_t max_len,
                                          int32_t /*num_cands*/) {
  return ws_layout(rows, batch, vocab, max_len).total;  // the candidate lists are read in place
}

sv_status_t spec_verify_rejection_chain_sparse(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                               int32_t m, int32_t vocab, const int32_t* verify_ids,
                                               const int32_t* cand_ids, const float* cand_probs, int32_t num_cands,
                                               int64_t ldc, const float* temperature, const float* u_accept,
                                               const float* u_final, const int64_t* row_slots,
                                               const int64_t* seq_lens, const sv_out_t* out, void* ws,
                                               size_t ws_bytes, cudaStream_t stream) {
  if (batch < 0 || m < 0 || m >= (1 << 20)) return SV_ERR_BAD_SHAPE;
  if (batch > 0 && !cand_ids) return SV_ERR_NULL_ARG;
  const int64_t rows = static_cast<int64_t>(batch) * (m + 1);
  return rejection_common(logits, dtype, ld, batch, rows, m + 1, m + 1, vocab, nullptr, verify_ids, nullptr, 0,
                          temperature, u_accept, u_final, row_slots, seq_lens, out, ws, ws_bytes, stream, cand_ids,
                          cand_probs, num_cands, ldc);
}

sv_status_t spec_verify_rejection_ragged(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                         int64_t total_rows, int32_t max_len, int32_t vocab,
                                         const int32_t* cu_seqlens, const int32_t* verify_ids, const float* q,
                                         int64_t ldq, const float* temperature, const float* u_accept,
                                         const float* u_final, const int64_t* row_slots, const int64_t* seq_lens,
                                         const sv_out_t* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (batch < 0 || total_rows < 0 || max_len < 1 || max_len >= (1 << 20)) return SV_ERR_BAD_SHAPE;
  if (!cu_seqlens) return SV_ERR_NULL_ARG;
  return rejection_common(logits, dtype, ld, batch, total_rows, max_len, 0, vocab, cu_seqlens, verify_ids, q, ldq,
                          temperature, u_accept, u_final, row_slots, seq_lens, out, ws, ws_bytes, stream);
}

static sv_status_t tree_common(int mode, const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                               int32_t nodes, int32_t vocab, const int32_t* tokens, const int32_t* parents,
                               const int32_t* first_child, const int32_t* next_sibling, const float* temperature,
                               float threshold_single, float threshold_acc, const float* u_accept,
                               const float* u_final, const int64_t* row_slots, const int64_t* seq_lens,
                               const sv_out_t* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (batch < 0 || nodes < 1 || nodes > kMaxNodes || (mode == 1 && batch > 65535)) return SV_ERR_BAD_SHAPE;
  if (batch == 0) return empty_batch(out, stream);
  const int64_t rows = static_cast<int64_t>(batch) * nodes;
  SV_TRY(check_logits(logits, dtype, ld, rows, vocab));
  if (!tokens || !parents) return SV_ERR_NULL_ARG;
  if ((first_child == nullptr) != (next_sibling == nullptr)) return SV_ERR_NULL_ARG;
  if (mode == 1) {
    if (!temperature || !u_accept || !u_final) return SV_ERR_NULL_ARG;
    if (!(threshold_acc > 0.0f) || !std::isfinite(threshold_acc) || std::isnan(threshold_single))
      return SV_ERR_BAD_SHAPE;
  }
  SV_TRY(check_out(out, row_slots, seq_lens));
  Ws w{};
  SV_TRY(carve(ws, ws_bytes, rows, batch, vocab, nodes, &w));
  DeviceInfo dev{};
  SV_TRY_CUDA(device_info(&dev));
  const LogitsView lg{logits, dtype, ld, rows, vocab};
  const OutView ov = out_view(out);
  const RowMap map = mode == 1 ? RowMap{kMapFixed, nodes, batch, nullptr, temperature}
                               : RowMap{kMapGreedy, nodes, batch, nullptr, nullptr};
  SV_TRY_CUDA(row_stats_timed(lg, map, w, stats_grid(dev, lg), stream));
  TreeParams p{lg,          batch,
               nodes,       tokens,
               parents,     first_child,
               next_sibling, mode == 1 ? temperature : nullptr,
               threshold_single, threshold_acc,
               u_accept,    u_final};
  const CommitParams cp{batch, nodes, row_slots, seq_lens, w.err};
  if (mode == 0 && accept_commit_fits(batch, nodes)) {  // one CTA walks and commits a small greedy batch
    SV_TRY_CUDA(launch_accept_commit_tree(p, ov, cp, w, stream));
    return SV_OK;
  }
  SV_TRY_CUDA(launch_accept_tree(p, ov, w, stream));
  if (mode == 1) {
    SV_TRY_CUDA(launch_sample_and_commit(lg, nullptr, 0, u_final, ov, cp, w, dev, stream));
  } else {
    SV_TRY_CUDA(launch_commit(ov, cp, stream));
  }
  return SV_OK;
}

sv_status_t spec_verify_greedy_tree(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t nodes,
                                    int32_t vocab, const int32_t* tokens, const int32_t* parents,
                                    const int32_t* first_child, const int32_t* next_sibling,
                                    const int64_t* row_slots, const int64_t* seq_lens, const sv_out_t* out,
                                    void* ws, size_t ws_bytes, cudaStream_t stream) {
  return tree_common(0, logits, dtype, ld, batch, nodes, vocab, tokens, parents, first_child, next_sibling, nullptr,
                     1.0f, 1.0f, nullptr, nullptr, row_slots, seq_lens, out, ws, ws_bytes, stream);
}

sv_status_t spec_verify_target_only_tree(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                         int32_t nodes, int32_t vocab, const int32_t* tokens,
                                         const int32_t* parents, const int32_t* first_child,
                                         const int32_t* next_sibling, const float* temperature,
                                         float threshold_single, float threshold_acc, const float* u_accept,
                                         const float* u_final, const int64_t* row_slots, const int64_t* seq_lens,
                                         const sv_out_t* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return tree_common(1, logits, dtype, ld, batch, nodes, vocab, tokens, parents, first_child, next_sibling,
                     temperature, threshold_single, threshold_acc, u_accept, u_final, row_slots, seq_lens, out, ws,
                     ws_bytes, stream);
}

sv_status_t spec_verify_row_stats(const void* logits, sv_dtype_t dtype, int64_t ld, int64_t rows, int32_t vocab,
                                  const float* row_temp, const int32_t* probe, float* out_max,
                                  int32_t* out_argmax, double* out_z, float* out_p, uint32_t* row_flags,
                                  void* ws, size_t ws_bytes, cudaStream_t stream) {
  SV_TRY(check_logits(logits, dtype, ld, rows, vocab));
  if (!out_max || !out_argmax || !out_z) return SV_ERR_NULL_ARG;
  if (rows == 0) return SV_OK;
  Ws w{};
  SV_TRY(carve(ws, ws_bytes, rows, 1, vocab, 1, &w));
  DeviceInfo dev{};
  SV_TRY_CUDA(device_info(&dev));
  const LogitsView lg{logits, dtype, ld, rows, vocab};
  const RowMap map = row_temp ? RowMap{kMapPerRow, 1, 0, nullptr, row_temp}
                              : RowMap{kMapGreedy, 1, 0, nullptr, nullptr};
  SV_TRY_CUDA(row_stats_timed(lg, map, w, stats_grid(dev, lg), stream));
  SV_TRY_CUDA(launch_export_stats(lg, w, probe, out_max, out_argmax, out_z, out_p, row_flags, stream));
  SV_TRY_CUDA(cudaMemsetAsync(w.err, 0, sizeof(uint32_t), stream));
  return SV_OK;
}

}  // extern "C"
