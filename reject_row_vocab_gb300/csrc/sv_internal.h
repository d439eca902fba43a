// Internal layout shared by the CUDA translation units of libspecverify.
//
// Not installed, not part of the C ABI: the public interface is
// include/specverify.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

// Per-request status bits (same values as SV_DEV_* in the public header).
constexpr uint32_t kStTokenRange = SV_DEV_TOKEN_RANGE;
constexpr uint32_t kStNonFinite = SV_DEV_NONFINITE;
constexpr uint32_t kStBadTree = SV_DEV_BAD_TREE;
constexpr uint32_t kStBadLayout = SV_DEV_BAD_LAYOUT;
constexpr uint32_t kStResidualEmpty = SV_DEV_RESIDUAL_EMPTY;
constexpr uint32_t kStDupSibling = SV_DEV_DUP_SIBLING;
constexpr uint32_t kStTimeout = SV_DEV_TIMEOUT;

// Final statistics of one logits row, written by the row-statistics kernel.
// M is the row maximum over usable entries (finite or -inf), argmax its lowest
// index (-1 for an all -inf row), k = log2(e)/T (0 for a greedy row),
// Z = sum_v 2^((l_v - M) * k) and inv_z = 1/Z (both 0 for a greedy row).
struct RowStat {
  float Z;
  float M;
  int32_t argmax;
  uint32_t flags;
  float k;
  float inv_z;
  float below;  // sum over ids below the row's probe token, in Z's units (probe-aware pass only)
  int32_t pad;
};
static_assert(sizeof(RowStat) == 32, "RowStat layout");

// A CTA's partial statistics for the part of one row it scanned.
struct RowPartial {
  float s;  // sum of 2^((l - m) * k) over the part
  float m;
  int32_t idx;
  uint32_t flags;
};
static_assert(sizeof(RowPartial) == 16, "RowPartial layout");

// Sampling weights are summed as exact 64-bit fixed-point integers with 44
// fractional bits (a lane's sum of eight weights is below 2^4, a row's total
// below 2^62), so prefix sums do not depend on the order of the additions.
constexpr int kFixedBits = 44;

// What the final-token step has to do for a request.
enum SampleMode : int32_t {
  kModeDone = 0,       // token already decided (greedy, unusable row)
  kModeResidual = 1,   // draw from [p - q]_+ of sample_row
  kModeP = 2,          // draw from p of sample_row (bonus)
  kModePExcl = 3,      // draw from p of sample_row with the excluded tokens zeroed
  kModeNoCommit = 4,   // bad layout: nothing to do
  kModeResidualSparse = 5  // draw from [p - q]_+ of sample_row, q given as the request's candidate list
};

struct ReqState {
  int32_t r;
  int32_t sample_row;
  int32_t mode;
  int32_t bonus;
  uint32_t status;
  int32_t n_excl;
  int32_t pad0;
  int32_t pad1;
};
static_assert(sizeof(ReqState) == 32, "ReqState layout");

// Elements per sampling tile (one warp, eight elements per lane).
constexpr int kTile = 256;
// Upper bound on tree nodes per request.
constexpr int kMaxNodes = 1024;

struct WsLayout {
  size_t done_cnt, counters_end;
  size_t rowstat, partial, psb, state, excl, ureq, tsum, total;
  int32_t ntiles;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int64_t rows, int32_t batch, int32_t vocab, int32_t max_len) {
  WsLayout L{};
  size_t off = 0;
  L.done_cnt = off;
  off += sizeof(uint32_t) * 4;
  L.counters_end = off = align_up(off, 256);
  L.rowstat = off;
  off = align_up(off + sizeof(RowStat) * static_cast<size_t>(rows > 0 ? rows : 1), 256);
  L.partial = off;  // one partial per chunk of a row (1024-vector chunks of fp32 rows bound every case)
  {
    const int64_t nfull = (vocab > 0 ? vocab : 1) / 4;
    int64_t cpr = (nfull + 1023) / 1024;
    if (cpr < 1) cpr = 1;
    off = align_up(off + sizeof(RowPartial) * static_cast<size_t>(rows > 0 ? rows : 1) * static_cast<size_t>(cpr), 256);
    L.psb = off;  // the probe chunk's partial sum below the probe token, one float per chunk
    off = align_up(off + sizeof(float) * static_cast<size_t>(rows > 0 ? rows : 1) * static_cast<size_t>(cpr), 256);
  }
  L.state = off;
  off = align_up(off + sizeof(ReqState) * static_cast<size_t>(batch > 0 ? batch : 1), 256);
  L.excl = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(batch > 0 ? batch : 1) *
                           static_cast<size_t>(max_len > 0 ? max_len : 1), 256);
  L.ureq = off;  // per request: the uniform of its final draw when it differs from u_final
  off = align_up(off + sizeof(float) * static_cast<size_t>(batch > 0 ? batch : 1), 256);
  L.ntiles = (vocab + kTile - 1) / kTile;
  L.tsum = off;
  off = align_up(off + sizeof(uint64_t) * static_cast<size_t>(batch > 0 ? batch : 1) *
                           static_cast<size_t>(L.ntiles > 0 ? L.ntiles : 1), 256);
  L.total = off;
  return L;
}

// Workspace pointers carved from the caller's buffer.
struct Ws {
  uint32_t* done_cnt;
  uint32_t* err;  // sticky error word: a bounded wait gave up (reported as SV_DEV_TIMEOUT)
  RowStat* rowstat;
  RowPartial* partial;
  float* psb;   // probe-aware pass: per chunk, the sum below the probe token
  float* ureq;  // per request: the uniform of the final draw (sample-then-match)
  ReqState* state;
  int32_t* excl;
  const int32_t* cand_id;  // sparse q: the caller's candidate lists [rows, cand_ld], read in place
  const float* cand_q;     // their probabilities
  int64_t cand_ld;
  uint64_t* tsum;  // fixed-point tile sums of the sampled rows
  int32_t ntiles;
};

// How the statistics kernel finds a row's temperature.
enum RowMapKind : int32_t {
  kMapGreedy = 0,     // every row greedy (no exponentials)
  kMapFixed = 1,      // request = row / rows_per_req, T = temperature[request]
  kMapCu = 2,         // request from cu_seqlens (upper bound search), T = temperature[request]
  kMapPerRow = 3      // T = temperature[row]
};

struct RowMap {
  int32_t kind;
  int32_t rows_per_req;
  int32_t batch;
  const int32_t* cu;
  const float* temperature;
};

struct LogitsView {
  const void* base;
  int32_t dtype;  // SV_F32 or SV_BF16
  int64_t ld;
  int64_t rows;
  int32_t vocab;
};

struct OutView {
  int32_t* accept_len;
  int32_t* num_out;
  int32_t* out_tokens;
  int32_t* bonus;
  int32_t* accept_rows;
  int32_t* commit_cu;
  int64_t* commit_src_slot;
  int64_t* commit_dst_pos;
  uint32_t* dev_status;
};

struct ChainParams {
  LogitsView lg;
  int32_t batch;
  int32_t max_len;
  int32_t fixed_len;          // > 0: request b owns rows [b*fixed_len, (b+1)*fixed_len)
  const int32_t* cu;          // otherwise cu_seqlens [B+1]
  const int32_t* ids;
  const float* q;
  int64_t ldq;
  const float* temperature;   // NULL: greedy for every request
  const float* u_accept;
  const float* u_final;
  const int32_t* cand_ids;    // sparse q: [rows, ldc] candidate ids (-1 pads), NULL for dense q
  const float* cand_probs;    // [rows, ldc] their probabilities
  int32_t num_cands;
  int64_t ldc;
  int32_t match;              // 1: verification by independent target sampling and prefix match
};

// Largest candidate list per row a sparse q may have.
constexpr int kMaxCands = 1024;

struct TreeParams {
  LogitsView lg;
  int32_t batch;
  int32_t nodes;
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* first_child;   // NULL or [B, nodes]
  const int32_t* next_sibling;  // NULL or [B, nodes]
  const float* temperature;     // NULL: greedy
  float th_single;
  float th_acc;
  const float* u_accept;
  const float* u_final;
};

struct CommitParams {
  int32_t batch;
  int32_t max_len;
  const int64_t* row_slots;
  const int64_t* seq_lens;
  uint32_t* err;  // workspace error word, cleared once the call's statuses carry it
};

// Launch with programmatic stream serialisation: the kernel may start while
// the previous work on the stream drains, and waits for it (griddepcontrol)
// before touching any memory that work produces.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Records e as the last CUDA error of this thread and returns SV_ERR_CUDA.
sv_status_t cuda_failure(cudaError_t e);

// Device properties cached per device.
struct DeviceInfo {
  int sms;
  int stats_blocks_per_sm[2];  // [dtype]
};
cudaError_t device_info(DeviceInfo* info);

// Launchers (each enqueues on `stream` and returns the launch error).
// probe: when non-NULL, probe[row] is row's probe token (every row but the last of each block of probe_rpr
// rows); the pass also leaves RowStat.below, the sum over ids below it.
// stats_done: when non-NULL, recorded on the stream between the streaming pass and the row merge
// (benchmark instrumentation of the streaming kernel alone).
cudaError_t launch_row_stats(const LogitsView& lg, const RowMap& map, const Ws& ws, int grid, cudaStream_t stream,
                             const int32_t* probe = nullptr, int32_t probe_rpr = 0,
                             cudaEvent_t stats_done = nullptr);

// Test hook: the limit (ns) of the statistics kernel's in-CTA hand-off waits, with a forced expiry (see
// k_row_stats); 0 restores normal operation.  Read at each launch.
void set_hand_off_limit_ns(uint64_t ns);

// The p/q rejection chain entry point.  clear_counters: after every host check has passed, zero the workspace's
// counter words on the stream before the first kernel (for a workspace shared between calls).
sv_status_t rejection_chain_entry(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t m,
                                  int32_t vocab, const int32_t* verify_ids, const float* q, int64_t ldq,
                                  const float* temperature, const float* u_accept, const float* u_final,
                                  const int64_t* row_slots, const int64_t* seq_lens, const sv_out_t* out, void* ws,
                                  size_t ws_bytes, cudaStream_t stream, bool clear_counters);

// Records ev on stream (as an event node while the stream is being captured).
cudaError_t record_event(cudaEvent_t ev, cudaStream_t stream);
int stats_grid(const DeviceInfo& dev, const LogitsView& lg);
cudaError_t stats_occupancy(int dtype, int* blocks_per_sm);

cudaError_t launch_accept_chain(const ChainParams& p, const OutView& out, const Ws& ws, cudaStream_t stream);
cudaError_t launch_accept_tree(const TreeParams& p, const OutView& out, const Ws& ws, cudaStream_t stream);

// Greedy calls of at most kSmallGreedyBatch requests (trees: node arrays within kAcceptCommitSmemBytes) are
// finished and committed by one CTA, one warp per request, instead of the acceptance and commit kernels.
constexpr int kSmallGreedyBatch = 32;
constexpr int64_t kAcceptCommitSmemBytes = 48 * 1024;
bool accept_commit_fits(int32_t batch, int32_t nodes);  // nodes <= 0: a chain
cudaError_t accept_smem_setup();
cudaError_t launch_accept_commit_chain(const ChainParams& p, const OutView& out, const CommitParams& cp, const Ws& ws,
                                       cudaStream_t stream);
cudaError_t launch_accept_commit_tree(const TreeParams& p, const OutView& out, const CommitParams& cp, const Ws& ws,
                                      cudaStream_t stream);

// Residual / bonus sampler (two passes) followed by the commit, or the commit alone.
cudaError_t launch_sample_and_commit(const LogitsView& lg, const float* q, int64_t ldq, const float* u_final,
                                     const OutView& out, const CommitParams& cp, const Ws& ws,
                                     const DeviceInfo& dev, cudaStream_t stream, bool sparse_q = false);
cudaError_t launch_commit(const OutView& out, const CommitParams& cp, cudaStream_t stream);
cudaError_t sample_smem_setup();

// Row statistics exported as plain arrays.
cudaError_t launch_export_stats(const LogitsView& lg, const Ws& ws, const int32_t* probe, float* out_max,
                                int32_t* out_argmax, double* out_z, float* out_p, uint32_t* row_flags,
                                cudaStream_t stream);

}  // namespace sv
