// Final token and commit.
//
// The correction / bonus token is an inverse-CDF draw over unnormalised
// weights w_v of one row ([E2D] §1.2 residual p' = [p - q]_+ / sum [p - q]_+;
// bonus from p, §1.1; inverse CDF as in §6.2 sample_path()):
//   w_v = max(0, p_v - q_v)          after a rejection,
//   w_v = p_v                        bonus after every draft passed,
//   w_v = p_v, children zeroed       target-only tree stop ([SGO]),
//   w_v = max(0, p_v - q_v), q sparse (a candidate list, [E2D] §6.5).
// Pass A (k_sample) splits each sampled row into tiles of 256 entries (one
// warp, eight entries per lane) spread over many CTAs and stores every tile's
// weight sum; one extra block performs the commit: exclusive scan of
// commit_lens and the KV slot / position lists ([E2D] §5.6.6, §8.1; [SGO]
// "两个容易误解的工程细节").  Pass B (k_draw, one CTA per request) scans the
// tile sums, picks the tile holding t = u_final * S, and one warp re-forms that
// tile's weights with exactly the same arithmetic to find the entry.
//
//   [E2D] "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理"
//   [SGO] SGLang speculative-decoding overview (zdszero.github.io)
#include <climits>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_commit.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;

__device__ __forceinline__ bool sampling_mode(int32_t mode) {
  return mode == kModeResidual || mode == kModeP || mode == kModePExcl || mode == kModeResidualSparse;
}

// Raw 16-byte loads of one lane's eight entries (logits, and q for a residual).
struct LaneRaw {
  uint4 l0, l1, q0, q1;
};

__device__ __forceinline__ void lane_load_full(const LogitsView& lg, const float* q, int64_t ldq, int64_t row,
                                               bool resid, int64_t col0, LaneRaw& r) {
  if (lg.dtype == SV_BF16) {
    r.l0 = ld_stream16(static_cast<const char*>(lg.base) + (row * lg.ld + col0) * 2);
  } else {
    const char* base = static_cast<const char*>(lg.base) + (row * lg.ld + col0) * 4;
    r.l0 = ld_stream16(base);
    r.l1 = ld_stream16(base + 16);
  }
  if (resid) {
    const char* qb = reinterpret_cast<const char*>(q + row * ldq + col0);
    r.q0 = ld_stream16(qb);
    r.q1 = ld_stream16(qb + 16);
  }
}

__device__ __forceinline__ void lane_unpack(const LaneRaw& r, int32_t dtype, bool resid, float (&x)[8],
                                            float (&qv)[8]) {
  if (dtype == SV_BF16) {
    x[0] = bf16_lo(r.l0.x);
    x[1] = bf16_hi(r.l0.x);
    x[2] = bf16_lo(r.l0.y);
    x[3] = bf16_hi(r.l0.y);
    x[4] = bf16_lo(r.l0.z);
    x[5] = bf16_hi(r.l0.z);
    x[6] = bf16_lo(r.l0.w);
    x[7] = bf16_hi(r.l0.w);
  } else {
    x[0] = __uint_as_float(r.l0.x);
    x[1] = __uint_as_float(r.l0.y);
    x[2] = __uint_as_float(r.l0.z);
    x[3] = __uint_as_float(r.l0.w);
    x[4] = __uint_as_float(r.l1.x);
    x[5] = __uint_as_float(r.l1.y);
    x[6] = __uint_as_float(r.l1.z);
    x[7] = __uint_as_float(r.l1.w);
  }
  if (resid) {
    qv[0] = __uint_as_float(r.q0.x);
    qv[1] = __uint_as_float(r.q0.y);
    qv[2] = __uint_as_float(r.q0.z);
    qv[3] = __uint_as_float(r.q0.w);
    qv[4] = __uint_as_float(r.q1.x);
    qv[5] = __uint_as_float(r.q1.y);
    qv[6] = __uint_as_float(r.q1.z);
    qv[7] = __uint_as_float(r.q1.w);
  }
}

// A sparse residual row's first 32 candidates held in registers, one per
// lane (loaded once per request; later entries are read from memory).  The
// list is the caller's, in candidate order; an id outside [0, V) (padding -1
// included) is held as -1 and never matches an entry.
struct CandRegs {
  int32_t id;
  float q;
};

__device__ __forceinline__ CandRegs load_cand_regs(const int32_t* cid, const float* cq, int32_t n, int32_t V) {
  const int lane = threadIdx.x & 31;
  const int32_t id = lane < n ? cid[lane] : -1;
  return CandRegs{id >= 0 && id < V ? id : -1, lane < n ? cq[lane] : 0.0f};
}

// Weights of eight entries from their values; the single definition both
// passes use, so a tile's weights are bit-identical in both.
// SP: the kernel serves sparse-q requests; a dense residual is compiled out of
// it.  For kModePExcl (excl, n_excl) lists the tokens to zero.  A sparse
// residual (kModeResidualSparse) takes p here (mode kModeP) and its
// candidates from apply_candidates_tile.
template <bool SP>
__device__ __forceinline__ void weights_from_values(const float (&x)[8], const float (&qv)[8], const RowStat& rs,
                                                    float inv_z, int32_t mode, const int32_t* excl, int32_t n_excl,
                                                    int64_t col0, float (&w)[8]) {
  // Packed pairs: each lane of a pair rounds exactly like the scalar
  // operation, so w_i = fl(fl(ex2(fl(fl(x_i - M) * k)) / Z) - q_i) either way.
  const float2 nM = make_float2(-rs.M, -rs.M), kk = make_float2(rs.k, rs.k), iz = make_float2(inv_z, inv_z);
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float2 t = __fmul2_rn(__fadd2_rn(make_float2(x[i], x[i + 1]), nM), kk);
    const float2 e = make_float2(usable_logit(x[i]) ? ex2_fast(t.x) : 0.0f, usable_logit(x[i + 1]) ? ex2_fast(t.y) : 0.0f);
    const float2 p = __fmul2_rn(e, iz);
    w[i] = p.x;
    w[i + 1] = p.y;
  }
  if (!SP && mode == kModeResidual) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const float2 d = __fadd2_rn(make_float2(w[i], w[i + 1]), make_float2(-qv[i], -qv[i + 1]));
      w[i] = fmaxf(d.x, 0.0f);
      w[i + 1] = fmaxf(d.y, 0.0f);
    }
  } else if (mode == kModePExcl) {
    for (int e = 0; e < n_excl; ++e) {
      const int64_t d = static_cast<int64_t>(excl[e]) - col0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (d == i) w[i] = 0.0f;
    }
  }
}

// The residual of a sparse q over a whole tile [t0, t0 + 256), the whole
// warp taking part: w = max(p - q, 0), where q at an entry is subtracted once
// per candidate carrying its id, in candidate order.  The warp finds the
// (rare) candidates inside the tile with a ballot and the owning lane
// subtracts them.  Ids outside [0, V) are ignored.  w holds p on entry.
__device__ __forceinline__ void apply_candidates_tile(float (&w)[8], int64_t t0, int lane, const int32_t* cid,
                                                      const float* cq, int32_t n, int32_t V, const CandRegs& cr) {
  for (int g = 0; g < n; g += 32) {
    const int c = g + lane;
    const int32_t id = g == 0 ? cr.id : (c < n ? cid[c] : -1);
    const float qq = g == 0 ? cr.q : (c < n ? cq[c] : 0.0f);
    const int64_t off = static_cast<int64_t>(id) - t0;
    unsigned hit = __ballot_sync(0xffffffffu, c < n && id < V && off >= 0 && off < kTile);
    while (hit) {
      const int src = __ffs(hit) - 1;
      hit &= hit - 1;
      const int o = static_cast<int>(__shfl_sync(0xffffffffu, off, src));
      const float hq = __shfl_sync(0xffffffffu, qq, src);
      if ((o >> 3) == lane) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if ((o & 7) == i) w[i] = __fsub_rn(w[i], hq);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = fmaxf(w[i], 0.0f);
}

// The eight weights of one lane of a tile: entries [col0, col0 + 8) of `row`.
// Entries past the vocabulary weigh 0.  A sparse residual (SP) needs the
// whole warp on one tile, lane l at col0 = tile start + 8 l.
template <bool SP>
__device__ __forceinline__ void lane_weights(const LogitsView& lg, const float* q, int64_t ldq, int64_t row,
                                             const RowStat& rs, float inv_z, int32_t mode, const int32_t* excl,
                                             const float* excl_q, int32_t n_excl, int64_t col0, float (&w)[8],
                                             const CandRegs& cr = CandRegs{-1, 0.0f}) {
  const bool resid = !SP && mode == kModeResidual;  // a sparse-q kernel never reads dense q
  float x[8], qv[8];
  if (col0 + 8 <= lg.vocab) {
    LaneRaw r;
    lane_load_full(lg, q, ldq, row, resid, col0, r);
    lane_unpack(r, lg.dtype, resid, x, qv);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool in = col0 + i < lg.vocab;
      x[i] = in ? load_logit(lg, row, col0 + i) : -kInfF;
      qv[i] = (resid && in) ? __ldg(q + row * ldq + col0 + i) : 0.0f;
    }
  }
  const bool sparse = SP && mode == kModeResidualSparse;
  weights_from_values<SP>(x, qv, rs, inv_z, sparse ? kModeP : mode, excl, n_excl, col0, w);
  if (sparse) {
    const int lane = threadIdx.x & 31;
    apply_candidates_tile(w, col0 - lane * 8, lane, excl, excl_q, n_excl, lg.vocab, cr);
  }
}

// A lane's weight sum: fp32, left to right.  Pass B walks the same additions.
__device__ __forceinline__ float lane_sum(const float (&w)[8]) {
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = __fadd_rn(s, w[i]);
  return s;
}

__device__ __forceinline__ float inverse_z(const RowStat& rs) { return rs.inv_z; }



// Weight sums of tiles [ta, tb) of one request's sampled row, U consecutive
// tiles in flight per warp; lane 0 stores each tile's sum.  Specialised on
// the logits type and on whether q is read, so no unused loads stay live.
template <int DT, bool RESID>
__device__ __forceinline__ void warp_tile_sums_t(const LogitsView& lg, const float* q, int64_t ldq, int64_t row,
                                                 const RowStat& rs, float inv_z, int32_t mode, const int32_t* excl,
                                                 int32_t n_excl, int ta, int tb, uint64_t* ts) {
  constexpr int U = 4;
  const int lane = threadIdx.x & 31;
  const int full_tiles = lg.vocab / kTile;
  for (int t0 = ta; t0 < tb; t0 += U) {
    float ls[U];
    if (t0 + U <= tb && t0 + U <= full_tiles) {  // all loads first, then the arithmetic
      uint4 l0[U], l1[U], q0[U], q1[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t col0 = static_cast<int64_t>(t0 + u) * kTile + lane * 8;
        if (DT == SV_BF16) {
          l0[u] = ld_stream16(static_cast<const char*>(lg.base) + (row * lg.ld + col0) * 2);
        } else {
          const char* base = static_cast<const char*>(lg.base) + (row * lg.ld + col0) * 4;
          l0[u] = ld_stream16(base);
          l1[u] = ld_stream16(base + 16);
        }
        if (RESID) {
          const char* qb = reinterpret_cast<const char*>(q + row * ldq + col0);
          q0[u] = ld_stream16(qb);
          q1[u] = ld_stream16(qb + 16);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        LaneRaw r;
        r.l0 = l0[u];
        if (DT != SV_BF16) r.l1 = l1[u];
        if (RESID) {
          r.q0 = q0[u];
          r.q1 = q1[u];
        }
        float x[8], qv[8], w[8];
        lane_unpack(r, DT, RESID, x, qv);
        weights_from_values<false>(x, qv, rs, inv_z, mode, excl, n_excl, static_cast<int64_t>(t0 + u) * kTile + lane * 8,
                                   w);
        ls[u] = lane_sum(w);
      }
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float w[8];
        if (t0 + u < tb) {
          lane_weights<false>(lg, q, ldq, row, rs, inv_z, mode, excl, nullptr, n_excl,
                       static_cast<int64_t>(t0 + u) * kTile + lane * 8, w);
          ls[u] = lane_sum(w);
        } else {
          ls[u] = 0.0f;
        }
      }
    }
    uint64_t fx[U];
#pragma unroll
    for (int u = 0; u < U; ++u) fx[u] = to_fixed(ls[u]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {  // U exact butterflies, interleaved
#pragma unroll
      for (int u = 0; u < U; ++u) fx[u] += __shfl_xor_sync(0xffffffffu, fx[u], off);
    }
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (t0 + u < tb) ts[t0 + u] = fx[u];
    }
  }
}

__device__ __forceinline__ void warp_tile_sums(const LogitsView& lg, const float* q, int64_t ldq, int64_t row,
                                               const RowStat& rs, float inv_z, int32_t mode, const int32_t* excl,
                                               int32_t n_excl, int ta, int tb, uint64_t* ts) {
  const bool resid = mode == kModeResidual;
  if (lg.dtype == SV_BF16) {
    if (resid) {
      warp_tile_sums_t<SV_BF16, true>(lg, q, ldq, row, rs, inv_z, mode, excl, n_excl, ta, tb, ts);
    } else {
      warp_tile_sums_t<SV_BF16, false>(lg, q, ldq, row, rs, inv_z, mode, excl, n_excl, ta, tb, ts);
    }
  } else {
    if (resid) {
      warp_tile_sums_t<SV_F32, true>(lg, q, ldq, row, rs, inv_z, mode, excl, n_excl, ta, tb, ts);
    } else {
      warp_tile_sums_t<SV_F32, false>(lg, q, ldq, row, rs, inv_z, mode, excl, n_excl, ta, tb, ts);
    }
  }
}

// The draw of one request by one CTA, once all its tile sums exist: scan the
// (exact, fixed-point) tile sums, pick the tile holding T = floor(u_final * S),
// then one warp re-forms that tile's weights (same arithmetic as the sums) and
// walks to the entry.  rs is the sampled row's statistics, u its uniform, cr
// the first candidates of a sparse residual row (load_cand_regs).
template <bool NAMED, bool SP>
__device__ __forceinline__ void block_draw(const LogitsView& lg, const float* q, int64_t ldq, float u,
                                           const OutView& out, const CommitParams& cp, const Ws& ws,
                                           int32_t excl_stride, int b, const ReqState& rq, const RowStat& rs,
                                           const CandRegs& cr) {
  __shared__ uint64_t s_scan[kSampleWarps + 1];
  __shared__ int s_tile;
  __shared__ int s_last_nz;
  __shared__ uint64_t s_pre;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = ws.ntiles;
  const int64_t row = rq.sample_row;
  const float inv_z = inverse_z(rs);
  const bool sparse = SP && rq.mode == kModeResidualSparse;
  const int32_t* excl = sparse ? ws.cand_id + row * ws.cand_ld : ws.excl + static_cast<int64_t>(b) * excl_stride;
  const float* excl_q = sparse ? ws.cand_q + row * ws.cand_ld : nullptr;
  uint64_t* ts = ws.tsum + static_cast<int64_t>(b) * T;
  int32_t mode = rq.mode;
  uint32_t st_add = 0u;
  const int per = (T + kSampleThreads - 1) / kSampleThreads;
  const int ta = min(T, tid * per), tb = min(T, ta + per);

  // Each thread's tile sums, loaded once (all loads issued before any use)
  // and kept in registers for both the scan and the search below.
  constexpr int kHeld = 8;
  const bool held = per <= kHeld;
  uint64_t tv[kHeld];
  uint64_t loc = 0;
  if (held) {
#pragma unroll
    for (int j = 0; j < kHeld; ++j)
      tv[j] = ta + j < tb ? __ldcg(reinterpret_cast<const unsigned long long*>(ts) + ta + j) : 0ull;
#pragma unroll
    for (int j = 0; j < kHeld; ++j) loc += tv[j];
  } else {
    for (int j = ta; j < tb; ++j) loc += __ldcg(reinterpret_cast<const unsigned long long*>(ts) + j);
  }
  uint64_t total;
  uint64_t pre = block_exclusive_scan<uint64_t, kSampleThreads, NAMED>(loc, s_scan, &total);
  if (total == 0) {  // residual (or what is left of p) is empty: draw from p instead
    mode = kModeP;
    st_add = kStResidualEmpty;
    warp_tile_sums(lg, q, ldq, row, rs, inv_z, mode, excl, 0, warp * ((T + kSampleWarps - 1) / kSampleWarps),
                   min(T, (warp + 1) * ((T + kSampleWarps - 1) / kSampleWarps)), ts);
    __threadfence_block();
    group_sync<kSampleThreads, NAMED>();
    loc = 0;
    if (held) {
#pragma unroll
      for (int j = 0; j < kHeld; ++j)
        tv[j] = ta + j < tb ? __ldcg(reinterpret_cast<const unsigned long long*>(ts) + ta + j) : 0ull;
#pragma unroll
      for (int j = 0; j < kHeld; ++j) loc += tv[j];
    } else {
      for (int j = ta; j < tb; ++j) loc += __ldcg(reinterpret_cast<const unsigned long long*>(ts) + j);
    }
    pre = block_exclusive_scan<uint64_t, kSampleThreads, NAMED>(loc, s_scan, &total);
  }
  const uint64_t t = scale_fixed(u, total);
  if (tid == 0) {
    s_tile = INT_MAX;
    s_last_nz = -1;
  }
  group_sync<kSampleThreads, NAMED>();
  int my_tile = INT_MAX, my_nz = -1;
  uint64_t my_pre = 0, run = pre;
  for (int j = ta; j < tb; ++j) {
    uint64_t wj = 0;
    if (held) {
#pragma unroll
      for (int i = 0; i < kHeld; ++i)
        if (i == j - ta) wj = tv[i];
    } else {
      wj = __ldcg(reinterpret_cast<const unsigned long long*>(ts) + j);
    }
    if (wj > 0) {
      my_nz = j;
      if (my_tile == INT_MAX && run <= t && t < run + wj) {
        my_tile = j;
        my_pre = run;
      }
    }
    run += wj;
  }
  if (my_tile != INT_MAX) atomicMin(&s_tile, my_tile);
  if (my_nz >= 0) atomicMax(&s_last_nz, my_nz);
  group_sync<kSampleThreads, NAMED>();
  if (my_tile != INT_MAX && my_tile == s_tile) s_pre = my_pre;
  group_sync<kSampleThreads, NAMED>();
  if (warp != 0) return;

  const bool located = s_tile != INT_MAX;
  int v = -1;
  if (located || s_last_nz >= 0) {
    const int tile = located ? s_tile : s_last_nz;
    const uint64_t tpre = located ? s_pre : 0;
    const int64_t col0 = static_cast<int64_t>(tile) * kTile + lane * 8;
    float w[8];
    lane_weights<SP>(lg, q, ldq, row, rs, inv_z, mode, excl, excl_q,
                     (mode == kModePExcl || mode == kModeResidualSparse) ? rq.n_excl : 0, col0, w, cr);
    const uint64_t W = to_fixed(lane_sum(w));
    const uint64_t li = warp_inclusive_scan_u64(W);
    const uint64_t lo = tpre + (li - W), hi = tpre + li;
    const unsigned hit = __ballot_sync(0xffffffffu, located && W > 0 && lo <= t && t < hi);
    if (hit) {
      const int f = __ffs(hit) - 1;
      int cand = -1;
      if (lane == f) {
        float cum = 0.0f;  // the same fp32 additions as lane_sum, so the last step reaches W
        for (int i = 0; i < 8; ++i) {
          cum = __fadd_rn(cum, w[i]);
          if (cand < 0 && lo + to_fixed(cum) > t) cand = i;
        }
        if (cand < 0)
          for (int i = 7; i >= 0; --i)
            if (cand < 0 && w[i] > 0.0f) cand = i;
      }
      cand = __shfl_sync(0xffffffffu, cand, f);
      v = static_cast<int>(static_cast<int64_t>(tile) * kTile + f * 8 + cand);
    } else {  // not reachable with exact sums; kept as a defined outcome: last positive entry of the tile
      const unsigned nz = __ballot_sync(0xffffffffu, W > 0);
      const int f = nz ? 31 - __clz(nz) : 0;
      int cand = -1;
      if (lane == f)
        for (int i = 7; i >= 0; --i)
          if (cand < 0 && w[i] > 0.0f) cand = i;
      cand = __shfl_sync(0xffffffffu, cand, f);
      v = cand < 0 ? -1 : static_cast<int>(static_cast<int64_t>(tile) * kTile + f * 8 + cand);
    }
  } else {
    st_add |= kStNonFinite;  // no positive weight at all (not reachable for a usable row)
  }
  if (lane == 0) {
    out.bonus[b] = v;
    out.out_tokens[static_cast<int64_t>(b) * cp.max_len + rq.r] = v;
    if (st_add) out.dev_status[b] = rq.status | st_add;
  }
}

// Tile sums and commit.  The batch's (request, tile) space is split into
// equal contiguous ranges, one per block (one resident wave).  In each block a
// producer warp streams the sampled rows' tiles (logits, and q for a dense
// residual) through a ring of shared-memory stages with bulk copies; eight
// consumer warps sum the weights of every tile.  The draws follow in k_draw,
// once every sum exists.  One extra block performs the commit (it needs only
// the acceptance results).  Every wait is bounded; no block waits on another.
constexpr int kSampleStages = 3;
constexpr int kSampleStageBytes = 32 * 1024;
constexpr int kSampleStageMaxTiles = 32;
constexpr int kSampleBlocksPerSM = 2;
constexpr uint64_t kSampleWaitNs = 1000000000ull;
constexpr int kSampleBlockThreads = kSampleThreads + 32;  // consumers + one producer warp
constexpr size_t kSampleSmemBytes = static_cast<size_t>(kSampleStages) * kSampleStageBytes + 256;

struct SampleRing {
  unsigned long long full[kSampleStages];
  unsigned long long empty[kSampleStages];
  int abort;
};

__device__ __forceinline__ int stage_tiles(int dtype, bool resid) {
  const int tb = kTile * ((dtype == SV_BF16 ? 2 : 4) + (resid ? 4 : 0));
  const int n = kSampleStageBytes / tb;
  return n < kSampleStageMaxTiles ? n : kSampleStageMaxTiles;
}

// Tile sums of one landed stage holding n tiles from tile c0 of the sampled row,
// by the eight consumer warps: logits at src and, for a residual draw, q at
// src + lb.  Specialised on the logits type and the draw, so no unused loads
// or branches stay live (excluded-token draws take the general path).
template <int DT, bool RESID>
__device__ __forceinline__ void stage_tile_sums(uint32_t src, uint32_t lb, int n, int c0, const RowStat& rs,
                                                float inv_z, uint64_t* ts) {
  constexpr int ES = DT == SV_BF16 ? 2 : 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < n; i += kSampleWarps) {
    const uint32_t off = static_cast<uint32_t>(i) * kTile + lane * 8;  // element offset in the stage
    LaneRaw raw;
    raw.l0 = lds16(src + off * ES);
    if (ES == 4) raw.l1 = lds16(src + off * ES + 16);
    if (RESID) {
      raw.q0 = lds16(src + lb + off * 4);
      raw.q1 = lds16(src + lb + off * 4 + 16);
    }
    float x[8], qv[8], w[8];
    lane_unpack(raw, DT, RESID, x, qv);
    weights_from_values<false>(x, qv, rs, inv_z, RESID ? kModeResidual : kModeP, nullptr, 0,
                               static_cast<int64_t>(c0 + i) * kTile + lane * 8, w);
    const uint64_t fa = warp_sum_u64(to_fixed(lane_sum(w)));
    if (lane == 0) ts[c0 + i] = fa;
  }
}

// The fixed-point weight sum of tile i of a stage holding a sparse residual
// row from tile c0 (logits only; p minus the candidate list cid / cq of nc
// entries, the first 32 in cr), summed over the lane's eight entries only.
template <int DT>
__device__ __forceinline__ uint64_t sparse_lane_fx(uint32_t src, int i, int c0, const RowStat& rs, float inv_z,
                                                   const int32_t* cid, const float* cq, int32_t nc, int32_t V,
                                                   const CandRegs& cr) {
  constexpr int ES = DT == SV_BF16 ? 2 : 4;
  const int lane = threadIdx.x & 31;
  const uint32_t off = static_cast<uint32_t>(i) * kTile + lane * 8;  // element offset in the stage
  LaneRaw raw;
  raw.l0 = lds16(src + off * ES);
  if (ES == 4) raw.l1 = lds16(src + off * ES + 16);
  float x[8], qv[8], w[8];
  lane_unpack(raw, DT, false, x, qv);
  weights_from_values<true>(x, qv, rs, inv_z, kModeP, nullptr, 0, static_cast<int64_t>(c0 + i) * kTile + lane * 8, w);
  apply_candidates_tile(w, static_cast<int64_t>(c0 + i) * kTile, lane, cid, cq, nc, V, cr);
  return to_fixed(lane_sum(w));
}

// Tile sums of one landed stage of a sparse residual row.  Two tiles per warp
// and iteration, so their dependency chains (weights, candidates, lane sum,
// fixed-point conversion, warp reduction) overlap.
template <int DT>
__device__ __forceinline__ void stage_tile_sums_sparse(uint32_t src, int n, int c0, const RowStat& rs, float inv_z,
                                                       const int32_t* cid, const float* cq, int32_t nc, int32_t V,
                                                       const CandRegs& cr, uint64_t* ts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < n; i += 2 * kSampleWarps) {
    const int i2 = i + kSampleWarps;
    const uint64_t a = sparse_lane_fx<DT>(src, i, c0, rs, inv_z, cid, cq, nc, V, cr);
    const uint64_t c = i2 < n ? sparse_lane_fx<DT>(src, i2, c0, rs, inv_z, cid, cq, nc, V, cr) : 0ull;
    const uint64_t fa = warp_sum_u64(a);  // i2 < n is the same in every lane
    const uint64_t fc = warp_sum_u64(c);
    if (lane == 0) {
      ts[c0 + i] = fa;
      if (i2 < n) ts[c0 + i2] = fc;
    }
  }
}

template <bool SP>
__global__ void __launch_bounds__(kSampleBlockThreads, kSampleBlocksPerSM) k_sample(LogitsView lg, const float* q, int64_t ldq,
                                                                   const float* u_final, OutView out,
                                                                   CommitParams cp, Ws ws, int32_t excl_stride,
                                                                   int32_t nblocks) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ SampleRing ring;
  if (blockIdx.x == 0) {  // the commit block (first, so it runs in the first wave)
    grid_dependency_wait();  // acceptance results from the previous kernel
    allow_dependents();
    if (threadIdx.x < kCommitThreads) commit_block_named(out, cp);
    return;
  }
  // The block's tile range and its ring depend on nothing the previous kernels write: set up before waiting.
  const int64_t blk = blockIdx.x - 1;
  unsigned char* stages = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                           ~uintptr_t(127));
  const int T = ws.ntiles;
  const int full_tiles = lg.vocab / kTile;
  const int es = lg.dtype == SV_BF16 ? 2 : 4;
  const int64_t total = static_cast<int64_t>(cp.batch) * T;
  const int64_t t_begin = blk * total / nblocks, t_end = (blk + 1) * total / nblocks;
  if (t_begin >= t_end) return;
  const int64_t b_first = t_begin / T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSampleStages; ++i) {
      mbar_init(smem_addr(&ring.full[i]), 1);
      mbar_init(smem_addr(&ring.empty[i]), kSampleWarps);
    }
    ring.abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  grid_dependency_wait();  // acceptance results from the previous kernel
  allow_dependents();

  if (warp == kSampleWarps) {  // ------------------------------------------ producer
    if (lane == 0) {
      uint32_t g = 0;
      for (int64_t b = b_first; b * T < t_end && !ring.abort; ++b) {
        const int ta = static_cast<int>((t_begin > b * T ? t_begin : b * T) - b * T);
        const int tb = static_cast<int>((t_end < (b + 1) * T ? t_end : (b + 1) * T) - b * T);
        const ReqState rq = ws.state[b];
        if (!sampling_mode(rq.mode)) continue;
        const bool resid = !SP && rq.mode == kModeResidual;
        const int per = stage_tiles(lg.dtype, resid);
        const int tc = min(tb, full_tiles);
        const int64_t row = rq.sample_row;
        for (int c0 = ta; c0 < tc; c0 += per, ++g) {
          const int n = min(per, tc - c0);
          const int st = g % kSampleStages;
          if (!mbar_wait_bounded(smem_addr(&ring.empty[st]), ((g / kSampleStages) & 1u) ^ 1u, &ring.abort,
                                 kSampleWaitNs)) {
            ring.abort = 1;
            atomicOr(ws.err, 1u);
            break;
          }
          const uint32_t lb = static_cast<uint32_t>(n) * kTile * es;
          const uint32_t qb = resid ? static_cast<uint32_t>(n) * kTile * 4 : 0u;
          unsigned char* dst = stages + static_cast<size_t>(st) * kSampleStageBytes;
          mbar_arrive_expect_tx(smem_addr(&ring.full[st]), lb + qb);
          bulk_copy_g2s(smem_addr(dst),
                        static_cast<const char*>(lg.base) + (row * lg.ld + static_cast<int64_t>(c0) * kTile) * es, lb,
                        smem_addr(&ring.full[st]));
          if (qb)
            bulk_copy_g2s(smem_addr(dst + lb), q + row * ldq + static_cast<int64_t>(c0) * kTile, qb,
                          smem_addr(&ring.full[st]));
        }
      }
      for (int i = 0; i < kSampleStages && g > 0; ++i) {  // drain before the block may exit
        --g;
        volatile int never = 0;
        mbar_wait_bounded(smem_addr(&ring.full[g % kSampleStages]), (g / kSampleStages) & 1u, &never,
                          kSampleWaitNs);
      }
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  uint32_t g = 0;
  for (int64_t b = b_first; b * T < t_end; ++b) {
    const int ta = static_cast<int>((t_begin > b * T ? t_begin : b * T) - b * T);
    const int tb = static_cast<int>((t_end < (b + 1) * T ? t_end : (b + 1) * T) - b * T);
    const ReqState rq = ws.state[b];
    if (!sampling_mode(rq.mode)) continue;
    const bool resid = !SP && rq.mode == kModeResidual;
    const int per = stage_tiles(lg.dtype, resid);
    const int tc = min(tb, full_tiles);
    const int64_t row = rq.sample_row;
    const RowStat rs = ws.rowstat[row];
    const float inv_z = inverse_z(rs);
    const bool sparse = SP && rq.mode == kModeResidualSparse;
    const int32_t* excl = sparse ? ws.cand_id + row * ws.cand_ld : ws.excl + static_cast<int64_t>(b) * excl_stride;
    const float* excl_q = sparse ? ws.cand_q + row * ws.cand_ld : nullptr;
    const CandRegs cr = sparse ? load_cand_regs(excl, excl_q, rq.n_excl, lg.vocab) : CandRegs{-1, 0.0f};
    uint64_t* ts = ws.tsum + static_cast<int64_t>(b) * T;
    for (int c0 = ta; c0 < tc; c0 += per, ++g) {
      const int n = min(per, tc - c0);
      const int st = g % kSampleStages;
      const unsigned char* src = stages + static_cast<size_t>(st) * kSampleStageBytes;
      const uint32_t lb = static_cast<uint32_t>(n) * kTile * es;
      if (!mbar_wait_bounded(smem_addr(&ring.full[st]), (g / kSampleStages) & 1u, &ring.abort, kSampleWaitNs)) {
        ring.abort = 1;
        atomicOr(ws.err, 1u);
      } else {
        if (SP && sparse) {
          if (lg.dtype == SV_BF16) {
            stage_tile_sums_sparse<SV_BF16>(smem_addr(src), n, c0, rs, inv_z, excl, excl_q, rq.n_excl, lg.vocab, cr,
                                            ts);
          } else {
            stage_tile_sums_sparse<SV_F32>(smem_addr(src), n, c0, rs, inv_z, excl, excl_q, rq.n_excl, lg.vocab, cr,
                                           ts);
          }
        } else if (!SP && rq.mode == kModePExcl) {  // excluded tokens: the general weights
          for (int i = warp; i < n; i += kSampleWarps) {
            const uint32_t off = static_cast<uint32_t>(i) * kTile + lane * 8;  // element offset in the stage
            LaneRaw r;
            r.l0 = lds16(smem_addr(src) + off * es);
            if (es == 4) r.l1 = lds16(smem_addr(src) + off * es + 16);
            float x[8], qv[8], w[8];
            lane_unpack(r, lg.dtype, false, x, qv);
            weights_from_values<SP>(x, qv, rs, inv_z, kModePExcl, excl, rq.n_excl,
                                    static_cast<int64_t>(c0 + i) * kTile + lane * 8, w);
            const uint64_t fa = warp_sum_u64(to_fixed(lane_sum(w)));
            if (lane == 0) ts[c0 + i] = fa;
          }
        } else if (lg.dtype == SV_BF16) {
          if (resid) {
            stage_tile_sums<SV_BF16, true>(smem_addr(src), lb, n, c0, rs, inv_z, ts);
          } else {
            stage_tile_sums<SV_BF16, false>(smem_addr(src), lb, n, c0, rs, inv_z, ts);
          }
        } else if (resid) {
          stage_tile_sums<SV_F32, true>(smem_addr(src), lb, n, c0, rs, inv_z, ts);
        } else {
          stage_tile_sums<SV_F32, false>(smem_addr(src), lb, n, c0, rs, inv_z, ts);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&ring.empty[st]));
    }
    for (int tile = max(tc, ta) + warp; tile < tb; tile += kSampleWarps) {  // the ragged last tile
      float w[8];
      lane_weights<SP>(lg, q, ldq, row, rs, inv_z, rq.mode, excl, excl_q, rq.n_excl,
                       static_cast<int64_t>(tile) * kTile + lane * 8, w, cr);
      const uint64_t fx = warp_sum_u64(to_fixed(lane_sum(w)));
      if (lane == 0) ts[tile] = fx;
    }
  }
}

// The draws, one CTA per request, once every tile sum exists (this grid
// starts after k_sample has completed): no streaming block ever stops to
// draw, and all requests draw at the same time.
template <bool SP>
__global__ void __launch_bounds__(kSampleThreads) k_draw(LogitsView lg, const float* q, int64_t ldq,
                                                         const float* u_final, OutView out, CommitParams cp, Ws ws,
                                                         int32_t excl_stride) {
  // The request's state, its row statistics and its uniform come from the kernels before k_sample, which had
  // completed before any k_sample block passed its own dependency wait and let this grid start, and a sparse
  // row's candidates are inputs: all are read before waiting for the tile sums.
  const int b = blockIdx.x;
  const ReqState rq = ws.state[b];
  const bool draws = sampling_mode(rq.mode);
  RowStat rs{};
  float u = 0.0f;
  CandRegs cr{-1, 0.0f};
  if (draws) {
    rs = ws.rowstat[rq.sample_row];
    u = u_final[b];
    if (SP && rq.mode == kModeResidualSparse && threadIdx.x < 32)
      cr = load_cand_regs(ws.cand_id + rq.sample_row * ws.cand_ld, ws.cand_q + rq.sample_row * ws.cand_ld,
                          rq.n_excl, lg.vocab);
  }
  grid_dependency_wait();  // the tile sums of k_sample
  allow_dependents();
  if (!draws) return;
  block_draw<false, SP>(lg, q, ldq, u, out, cp, ws, excl_stride, b, rq, rs, cr);
}

__global__ void __launch_bounds__(kCommitThreads) k_commit(OutView out, CommitParams cp) {
  grid_dependency_wait();  // acceptance results from the previous kernel
  allow_dependents();
  commit_block(out, cp);
}

}  // namespace

cudaError_t sample_smem_setup() {
  const cudaError_t e = cudaFuncSetAttribute(k_sample<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSampleSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_sample<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSampleSmemBytes));
}

cudaError_t launch_sample_and_commit(const LogitsView& lg, const float* q, int64_t ldq, const float* u_final,
                                     const OutView& out, const CommitParams& cp, const Ws& ws,
                                     const DeviceInfo& dev, cudaStream_t stream, bool sparse_q) {
  // one resident wave (kSampleBlocksPerSM blocks per SM, one slot for the commit block), at least ~16 tiles per
  // block
  const int64_t tiles = static_cast<int64_t>(cp.batch) * ws.ntiles;
  int64_t nblocks = static_cast<int64_t>(dev.sms) * kSampleBlocksPerSM - 1;
  if (nblocks > (tiles + 15) / 16) nblocks = (tiles + 15) / 16;
  if (nblocks < 1) nblocks = 1;
  const cudaError_t e =
      launch_pdl(sparse_q ? k_sample<true> : k_sample<false>, dim3(static_cast<unsigned>(nblocks + 1)),
                 dim3(kSampleBlockThreads), kSampleSmemBytes, stream, lg, q, ldq, u_final, out, cp, ws,
                 static_cast<int32_t>(cp.max_len), static_cast<int32_t>(nblocks));
  if (e != cudaSuccess) return e;
  return launch_pdl(sparse_q ? k_draw<true> : k_draw<false>, dim3(static_cast<unsigned>(cp.batch)),
                    dim3(kSampleThreads), 0, stream, lg, q, ldq, u_final, out, cp, ws,
                    static_cast<int32_t>(cp.max_len));
}

cudaError_t launch_commit(const OutView& out, const CommitParams& cp, cudaStream_t stream) {
  return launch_pdl(k_commit, dim3(1), dim3(kCommitThreads), 0, stream, out, cp);
}

}  // namespace sv
