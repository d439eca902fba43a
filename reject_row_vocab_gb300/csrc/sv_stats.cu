// Row statistics: one streaming pass over every logits row.
//
// For each verify row the pass produces the maximum M, its lowest index (the
// greedy argmax, [E2D] §1.2 first bullet) and, for sampling rows,
// Z = sum_v 2^((l_v - M) * log2(e)/T), the normaliser of softmax(l/T)
// ([E2D] §6.2).  [E2D] = "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理".
//
// Work split: the rows are viewed as one flat sequence of 16-byte vectors and
// the grid (one resident wave) takes equal contiguous ranges of it, so every
// CTA streams the same number of bytes whatever the row count.  A row cut by
// range boundaries is finished by the last CTA that touches it: each CTA
// publishes its partial (m, s, argmax) for the cut rows, takes a ticket on the
// row's counter, and the CTA drawing the final ticket merges the partials in
// CTA order (deterministic) and resets the counter.  No CTA waits on another.
//
// Data movement: one producer warp streams the CTA's range into a ring of
// shared-memory stages with bulk copies (the TMA engine, completion counted on
// an mbarrier per stage); eight consumer warps fold each stage and release it.
// Bytes in flight per SM are set by the ring, not by registers.  Every wait is
// bounded (one second); a timeout raises the workspace error word, which the
// acceptance kernels report as SV_DEV_TIMEOUT.
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kConsumers = 256;                      // eight consumer warps
constexpr int kProducerWarp = kConsumers / 32;       // warp 8 streams the stages
constexpr int kFinalizerWarp = kProducerWarp + 1;    // warp 9 finishes each row
constexpr int kStatsThreads = kConsumers + 64;
constexpr int kChunkVecs = 1024;                     // 16 KB per stage
constexpr int kStages = 4;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kRowsCached = 64;  // per-row log2(e)/T precomputed for the first rows of a range

// One consumer thread's statistics for one row segment, handed to the finalizer.
struct SegSlot {
  float m;
  float s;        // sum of 2^((l - m) k)
  int32_t vidx;   // vector holding the first occurrence of m (to resolve), or -1
  int32_t idx;    // resolved index when vidx < 0
  uint32_t flags;
};

struct StatsSmem {
  uint4 buf[kStages][kChunkVecs];
  SegSlot seg[2][kConsumers];
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
  unsigned long long seg_full[2];
  unsigned long long seg_empty[2];
  float kc[kRowsCached];
  int abort;
};
constexpr size_t kStatsSmemBytes = sizeof(StatsSmem) + 128;  // + alignment slack

template <int DT>
struct VecTraits;
template <>
struct VecTraits<SV_BF16> {
  static constexpr int E = 8;   // elements per 16-byte vector
  static constexpr int ES = 2;  // element bytes
};
template <>
struct VecTraits<SV_F32> {
  static constexpr int E = 4;
  static constexpr int ES = 4;
};

// Per-thread running statistics: maximum m, the vector where m was last
// raised (its element index is resolved once, at the end of the range), the
// resolved argmax, flags, and a packed fp32 accumulator of 2^((l - r) k)
// against a reference r that trails m: r only moves when m outgrows it by
// more than kRefSlack (in log2 units), so most vectors need no rescale.
struct ThreadAcc {
  float m;
  int32_t vidx;  // vector (within the row) holding the first occurrence of m, -1 if none yet
  int32_t idx;   // resolved argmax (tail handling and after resolution)
  uint32_t flags;
  float r;       // exponent reference, starts at -FLT_MAX (finite: no inf - inf)
  float2 s;
};

constexpr float kRefSlack = 16.0f;  // terms stay <= 2^16 between reference moves
constexpr float kMinFinite = -3.402823466e38f;

__device__ __forceinline__ ThreadAcc acc_init() {
  return ThreadAcc{-kInfF, -1, -1, 0u, kMinFinite, make_float2(0.0f, 0.0f)};
}

// The accumulated sum expressed against the maximum m (for merging).
__device__ __forceinline__ float acc_sum_at_max(const ThreadAcc& a, float k) {
  const float s = a.s.x + a.s.y;
  if (s == 0.0f || a.r == a.m) return s;
  return s * exp2f((a.r - a.m) * k);
}

template <int DT>
__device__ __forceinline__ void unpack(const uint4& raw, float (&x)[VecTraits<DT>::E]) {
  if constexpr (DT == SV_BF16) {
    x[0] = bf16_lo(raw.x);
    x[1] = bf16_hi(raw.x);
    x[2] = bf16_lo(raw.y);
    x[3] = bf16_hi(raw.y);
    x[4] = bf16_lo(raw.z);
    x[5] = bf16_hi(raw.z);
    x[6] = bf16_lo(raw.w);
    x[7] = bf16_hi(raw.w);
  } else {
    x[0] = __uint_as_float(raw.x);
    x[1] = __uint_as_float(raw.y);
    x[2] = __uint_as_float(raw.z);
    x[3] = __uint_as_float(raw.w);
  }
}

// NaN-propagating maximum of a raw vector: NaN or +inf here sends the
// vector down the (rare) sanitising path.
template <int DT>
__device__ __forceinline__ float raw_max_nan(const uint4& raw) {
  if constexpr (DT == SV_BF16) {
    const uint32_t w = bmax2_nan(bmax2_nan(raw.x, raw.y), bmax2_nan(raw.z, raw.w));
    return fmax_nan(bf16_lo(w), bf16_hi(w));
  } else {
    return fmax_nan(fmax_nan(__uint_as_float(raw.x), __uint_as_float(raw.y)),
                    fmax_nan(__uint_as_float(raw.z), __uint_as_float(raw.w)));
  }
}

// Sum of 2^((x - m) k) over E elements, as a packed pair (fixed order).
template <int E>
__device__ __forceinline__ float2 exp_sum(const float (&x)[E], float m, float k) {
  const float2 nm = make_float2(-m, -m), kk = make_float2(k, k);
  float2 e[E / 2];
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    const float2 t = __fmul2_rn(__fadd2_rn(make_float2(x[2 * i], x[2 * i + 1]), nm), kk);
    e[i] = make_float2(ex2_fast(t.x), ex2_fast(t.y));
  }
  if constexpr (E == 8) {
    return __fadd2_rn(__fadd2_rn(e[0], e[1]), __fadd2_rn(e[2], e[3]));
  } else {
    return __fadd2_rn(e[0], e[1]);
  }
}

// Fold E logits one at a time, NaN and +inf entries read as -inf (the caller
// flags them).  immediate: record the argmax index itself, else the vector.
template <int E, bool EXP>
__device__ __forceinline__ void consume_dirty(ThreadAcc& a, const float (&x)[E], int32_t vec, float k,
                                              bool immediate) {
  for (int i = 0; i < E; ++i) {
    const float v = usable_logit(x[i]) ? x[i] : -kInfF;
    if (v > a.m) {
      a.m = v;
      if (immediate) {
        a.idx = vec * E + i;
        a.vidx = -1;  // the pending vector no longer holds the maximum
      } else {
        a.vidx = vec;
      }
    }
    if (EXP) {
      if (v > a.r) {  // exact reference moves here (rare path)
        const float f = a.r > kMinFinite ? exp2f((a.r - v) * k) : 0.0f;
        a.s = __fmul2_rn(a.s, make_float2(f, f));
        a.r = v;
      }
      a.s.x += ex2_fast((v - a.r) * k);
    }
  }
}

// Fold one vector.  The common case (clean data, maximum within the slack of
// the reference) is branch-free.
template <int DT, bool EXP>
__device__ __forceinline__ void consume(ThreadAcc& a, const uint4& raw, int32_t vec, float k, float slack) {
  constexpr int E = VecTraits<DT>::E;
  float x[E];
  unpack<DT>(raw, x);
  const float vmax = raw_max_nan<DT>(raw);
  const float bound = EXP ? a.r + slack : kInfF;
  if (!(vmax < bound)) {  // NaN / +inf present, or the maximum outgrew the reference (rare)
    if (!(vmax < kInfF)) {
      a.flags |= kStNonFinite;
      consume_dirty<E, EXP>(a, x, vec, k, false);
      return;
    }
    if (EXP) {
      const float f = a.r > kMinFinite ? exp2f((a.r - vmax) * k) : 0.0f;
      a.s = __fmul2_rn(a.s, make_float2(f, f));
      a.r = vmax;
    }
  }
  const bool raised = vmax > a.m;
  a.vidx = raised ? vec : a.vidx;
  a.m = fmaxf(a.m, vmax);
  if (EXP) a.s = __fadd2_rn(a.s, exp_sum<E>(x, a.r, k));
}

// The index of the first entry equal to m in vector vidx of a row.
template <int DT>
__device__ __forceinline__ int32_t resolve_index(const char* rowp, int32_t vidx, float m) {
  constexpr int E = VecTraits<DT>::E;
  float x[E];
  unpack<DT>(ld_stream16(rowp + static_cast<int64_t>(vidx) * 16), x);
  int j = E - 1;
#pragma unroll
  for (int i = E - 1; i >= 0; --i)
    if (x[i] == m) j = i;
  return vidx * E + j;
}

// The row's ragged tail vector (vocab not a multiple of the vector width), by one thread.
template <int DT, bool EXP>
__device__ __forceinline__ void fold_tail(ThreadAcc& a, const LogitsView& lg, int64_t row, int64_t nfull, float k) {
  constexpr int E = VecTraits<DT>::E;
  float x[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int64_t col = nfull * E + i;
    x[i] = col < lg.vocab ? load_logit(lg, row, col) : -kInfF;
    if (!usable_logit(x[i])) a.flags |= kStNonFinite;
  }
  consume_dirty<E, EXP>(a, x, static_cast<int32_t>(nfull), k, true);
}

// Fold the first n vectors of a stage (chunk starting at vector c0 of the row).
template <int DT, bool EXP>
__device__ __forceinline__ void fold_stage(ThreadAcc& a, uint32_t stage_addr, int32_t c0, int n, float k,
                                           float slack) {
  constexpr int PER = kChunkVecs / kConsumers;  // vectors per consumer thread per full stage
  const int t = threadIdx.x;
  if (n == kChunkVecs) {
    uint4 raw[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) raw[j] = lds16(stage_addr + (t + j * kConsumers) * 16);
#pragma unroll
    for (int j = 0; j < PER; ++j) consume<DT, EXP>(a, raw[j], c0 + t + j * kConsumers, k, slack);
  } else {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int vi = t + j * kConsumers;
      if (vi < n) consume<DT, EXP>(a, lds16(stage_addr + vi * 16), c0 + vi, k, slack);
    }
  }
}

__device__ __forceinline__ float row_k(const RowMap& map, int64_t row) {
  float T = 0.0f;
  switch (map.kind) {
    case kMapFixed:
      T = map.temperature[row / map.rows_per_req];
      break;
    case kMapCu: {
      int lo = 0, hi = map.batch - 1;
      while (lo < hi) {  // last request whose start is <= row
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(map.cu[mid]) <= row) {
          lo = mid;
        } else {
          hi = mid - 1;
        }
      }
      T = map.temperature[lo];
      break;
    }
    case kMapPerRow:
      T = map.temperature[row];
      break;
    default:
      T = 0.0f;
  }
  return temperature_k(T);
}

__device__ __forceinline__ int64_t cta_of_vector(int64_t v, int64_t G, int64_t NV) {
  return ((v + 1) * G - 1) / NV;
}

// The row's final statistics from its merged partial.
__device__ __forceinline__ RowStat finish_row(const Part& p, float k) {
  RowStat st;
  const bool samp = k > 0.0f && p.m > -kInfF;
  st.Z = samp ? p.s : 0.0f;
  st.inv_z = samp ? __fdiv_rn(1.0f, p.s) : 0.0f;
  st.M = p.m;
  st.argmax = p.idx;
  st.flags = p.flags;
  st.k = k;
  return st;
}

// Segment geometry of one row within a CTA's range.
struct Seg {
  int64_t s0, s1, sf;  // vectors [s0, s1) of the row are ours; [s0, sf) are full vectors
};

__device__ __forceinline__ Seg segment_of(int64_t row, int64_t NVr, int64_t v_begin, int64_t v_end, int64_t nfull) {
  const int64_t row_v0 = row * NVr;
  Seg g;
  g.s0 = (v_begin > row_v0 ? v_begin : row_v0) - row_v0;
  g.s1 = (v_end < row_v0 + NVr ? v_end : row_v0 + NVr) - row_v0;
  g.sf = g.s1 < nfull ? g.s1 : nfull;
  return g;
}

template <int DT>
__global__ void __launch_bounds__(kStatsThreads, 3) k_row_stats(LogitsView lg, RowMap map, Ws ws, int64_t NVr,
                                                                int64_t NV) {
  using VT = VecTraits<DT>;
  constexpr int E = VT::E;
  extern __shared__ unsigned char smem_raw[];
  StatsSmem& sm = *reinterpret_cast<StatsSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int64_t G = gridDim.x, c = blockIdx.x;
  const int64_t v_begin = c * NV / G, v_end = (c + 1) * NV / G;
  if (v_begin >= v_end) return;
  const int64_t r_first = v_begin / NVr, r_last = (v_end - 1) / NVr;
  const int64_t nfull = lg.vocab / E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&sm.full[s]), 1);
      mbar_init(smem_addr(&sm.empty[s]), kConsumers / 32);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&sm.seg_full[s]), kConsumers);
      mbar_init(smem_addr(&sm.seg_empty[s]), 1);
    }
    sm.abort = 0;
    mbar_fence_init();
  }
  // the temperatures of the first rows, fetched once while the first stages load
  if (threadIdx.x < kRowsCached && r_first + threadIdx.x <= r_last) sm.kc[threadIdx.x] = row_k(map, r_first + threadIdx.x);
  __syncthreads();

  if (warp == kProducerWarp) {  // ------------------------------------------ producer
    if (lane == 0) {
      uint32_t g = 0;
      for (int64_t row = r_first; row <= r_last && !sm.abort; ++row) {
        const Seg sg = segment_of(row, NVr, v_begin, v_end, nfull);
        const char* rowp = static_cast<const char*>(lg.base) + row * lg.ld * VT::ES;
        for (int64_t c0 = sg.s0; c0 < sg.sf; c0 += kChunkVecs, ++g) {
          const int n = static_cast<int>(sg.sf - c0 < kChunkVecs ? sg.sf - c0 : kChunkVecs);
          const int st = g % kStages;
          if (!mbar_wait_bounded(smem_addr(&sm.empty[st]), ((g / kStages) & 1u) ^ 1u, &sm.abort, kWaitLimitNs)) {
            sm.abort = 1;
            atomicOr(ws.err, 1u);
            break;
          }
          mbar_arrive_expect_tx(smem_addr(&sm.full[st]), n * 16);
          bulk_copy_g2s(smem_addr(&sm.buf[st][0]), rowp + c0 * 16, n * 16, smem_addr(&sm.full[st]));
        }
      }
      for (int s = 0; s < kStages && g > 0; ++s) {  // drain before the CTA may exit
        --g;
        volatile int never = 0;
        mbar_wait_bounded(smem_addr(&sm.full[g % kStages]), (g / kStages) & 1u, &never, kWaitLimitNs);
      }
    }
    return;
  }

  if (warp == kFinalizerWarp) {  // ---------------------------------------- finalizer
    uint32_t i = 0;
    for (int64_t row = r_first; row <= r_last; ++row, ++i) {
      const Seg sg = segment_of(row, NVr, v_begin, v_end, nfull);
      const char* rowp = static_cast<const char*>(lg.base) + row * lg.ld * VT::ES;
      const float k = row - r_first < kRowsCached ? sm.kc[row - r_first] : row_k(map, row);
      const int slot = i & 1;
      if (!mbar_wait_bounded(smem_addr(&sm.seg_full[slot]), (i >> 1) & 1u, &sm.abort, kWaitLimitNs)) {
        sm.abort = 1;
        atomicOr(ws.err, 1u);
      }
      // each lane folds eight consumers' statistics, resolving argmax indices from the row
      constexpr int PER = kConsumers / 32;
      SegSlot sl[PER];
#pragma unroll
      for (int t = 0; t < PER; ++t) sl[t] = sm.seg[slot][lane * PER + t];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.seg_empty[slot]));  // the slot is free again
      // Only the consumers holding the segment maximum need their index resolved.
      float mseg = -kInfF;
#pragma unroll
      for (int t = 0; t < PER; ++t) mseg = fmaxf(mseg, sl[t].m);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mseg = fmaxf(mseg, __shfl_xor_sync(0xffffffffu, mseg, off));
      int32_t idx[PER];
#pragma unroll
      for (int t = 0; t < PER; ++t)
        idx[t] = (sl[t].vidx >= 0 && sl[t].m == mseg) ? resolve_index<DT>(rowp, sl[t].vidx, sl[t].m) : sl[t].idx;
      Part p = part_identity();
#pragma unroll
      for (int t = 0; t < PER; ++t) part_merge(p, Part{sl[t].m, sl[t].s, idx[t], sl[t].flags}, k);
      p = part_warp_reduce(p, k);

      const int64_t c_lo = cta_of_vector(row * NVr, G, NV);
      const int64_t c_hi = cta_of_vector(row * NVr + NVr - 1, G, NV);
      if (c_lo == c_hi) {  // the whole row is ours
        if (lane == 0) ws.rowstat[row] = finish_row(p, k);
        continue;
      }
      int last = 0;
      if (lane == 0) {
        RowPartial rp;
        rp.s = p.s;
        rp.m = p.m;
        rp.idx = p.idx;
        rp.flags = p.flags;
        ws.partial[2 * c + (row == r_first ? 0 : 1)] = rp;
        const unsigned ticket = ticket_add(&ws.row_cnt[row], 1u);
        last = (ticket == static_cast<unsigned>(c_hi - c_lo));
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {  // last arriver: merge the row's partials in CTA order
        __syncwarp();
        Part acc = part_identity();
        for (int64_t cc = c_lo + lane; cc <= c_hi; cc += 32) {
          const int64_t first_row_cc = (cc * NV / G) / NVr;
          part_merge(acc, load_partial_cg(&ws.partial[2 * cc + (row == first_row_cc ? 0 : 1)]), k);
        }
        acc = part_warp_reduce(acc, k);
        if (lane == 0) {
          ws.rowstat[row] = finish_row(acc, k);
          ws.row_cnt[row] = 0u;  // leave the counter clean for the next call
        }
      }
      (void)sg;
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  uint32_t g = 0, i = 0;
  for (int64_t row = r_first; row <= r_last; ++row, ++i) {
    const Seg sg = segment_of(row, NVr, v_begin, v_end, nfull);
    const float k = row - r_first < kRowsCached ? sm.kc[row - r_first] : row_k(map, row);
    ThreadAcc a = acc_init();
    const float slack = k > 0.0f ? kRefSlack / k : 0.0f;
    for (int64_t c0 = sg.s0; c0 < sg.sf; c0 += kChunkVecs, ++g) {
      const int n = static_cast<int>(sg.sf - c0 < kChunkVecs ? sg.sf - c0 : kChunkVecs);
      const int st = g % kStages;
      if (!mbar_wait_bounded(smem_addr(&sm.full[st]), (g / kStages) & 1u, &sm.abort, kWaitLimitNs)) {
        sm.abort = 1;
        atomicOr(ws.err, 1u);
      } else if (k > 0.0f) {
        fold_stage<DT, true>(a, smem_addr(&sm.buf[st][0]), static_cast<int32_t>(c0), n, k, slack);
      } else {
        fold_stage<DT, false>(a, smem_addr(&sm.buf[st][0]), static_cast<int32_t>(c0), n, k, slack);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.empty[st]));
    }
    if (threadIdx.x == 0 && sg.s1 > nfull && nfull >= sg.s0) {  // the row's ragged tail vector
      if (k > 0.0f) {
        fold_tail<DT, true>(a, lg, row, nfull, k);
      } else {
        fold_tail<DT, false>(a, lg, row, nfull, k);
      }
    }
    // hand the statistics to the finalizer and go on with the next row
    const int slot = i & 1;
    if (!mbar_wait_bounded(smem_addr(&sm.seg_empty[slot]), ((i >> 1) & 1u) ^ 1u, &sm.abort, kWaitLimitNs)) {
      sm.abort = 1;
      atomicOr(ws.err, 1u);
    }
    sm.seg[slot][threadIdx.x] = SegSlot{a.m, k > 0.0f ? acc_sum_at_max(a, k) : 0.0f, a.vidx, a.idx, a.flags};
    mbar_arrive(smem_addr(&sm.seg_full[slot]));
  }
}

// Copy the row statistics out as plain arrays (and p at a probe token).
__global__ void k_export_stats(LogitsView lg, Ws ws, const int32_t* probe, float* out_max, int32_t* out_argmax,
                               double* out_z, float* out_p, uint32_t* row_flags) {
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (row >= lg.rows) return;
  const RowStat st = ws.rowstat[row];
  out_max[row] = st.M;
  out_argmax[row] = st.argmax;
  out_z[row] = st.Z;
  if (row_flags) row_flags[row] = st.flags | (__ldcg(ws.err) ? kStTimeout : 0u);
  if (out_p) {
    float p = 0.0f;
    if (probe && st.k > 0.0f && st.argmax >= 0) {
      const int32_t t = probe[row];
      if (t >= 0 && t < lg.vocab) {
        const float l = load_logit(lg, row, t);
        if (usable_logit(l)) p = __fdiv_rn(exp2f((l - st.M) * st.k), st.Z);
      }
    }
    out_p[row] = p;
  }
}

}  // namespace

cudaError_t stats_occupancy(int dtype, int* blocks_per_sm) {
  cudaError_t e;
  if (dtype == SV_BF16) {
    e = cudaFuncSetAttribute(k_row_stats<SV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kStatsSmemBytes));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_row_stats<SV_BF16>, kStatsThreads,
                                                         kStatsSmemBytes);
  }
  e = cudaFuncSetAttribute(k_row_stats<SV_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kStatsSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_row_stats<SV_F32>, kStatsThreads,
                                                       kStatsSmemBytes);
}

int stats_grid(const DeviceInfo& dev, const LogitsView& lg) {
  const int E = lg.dtype == SV_BF16 ? 8 : 4;
  const int64_t NVr = (lg.vocab + E - 1) / E;
  const int64_t NV = NVr * lg.rows;
  // One resident wave; at least ~2 vectors per thread per CTA; never more CTAs than vectors.
  int64_t g = static_cast<int64_t>(dev.sms) * dev.stats_blocks_per_sm[lg.dtype == SV_BF16 ? 1 : 0];
  const int64_t by_work = (NV + 2 * kConsumers - 1) / (2 * kConsumers);
  if (g > by_work) g = by_work;
  if (g > kMaxStatsGrid) g = kMaxStatsGrid;
  if (g > NV) g = NV;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

cudaError_t launch_row_stats(const LogitsView& lg, const RowMap& map, const Ws& ws, int grid, cudaStream_t stream) {
  const int E = lg.dtype == SV_BF16 ? 8 : 4;
  const int64_t NVr = (lg.vocab + E - 1) / E;
  const int64_t NV = NVr * lg.rows;
  if (lg.dtype == SV_BF16) {
    k_row_stats<SV_BF16><<<grid, kStatsThreads, kStatsSmemBytes, stream>>>(lg, map, ws, NVr, NV);
  } else {
    k_row_stats<SV_F32><<<grid, kStatsThreads, kStatsSmemBytes, stream>>>(lg, map, ws, NVr, NV);
  }
  return cudaGetLastError();
}

cudaError_t launch_export_stats(const LogitsView& lg, const Ws& ws, const int32_t* probe, float* out_max,
                                int32_t* out_argmax, double* out_z, float* out_p, uint32_t* row_flags,
                                cudaStream_t stream) {
  const int threads = 256;
  const int64_t blocks = (lg.rows + threads - 1) / threads;
  k_export_stats<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(lg, ws, probe, out_max, out_argmax, out_z,
                                                                        out_p, row_flags);
  return cudaGetLastError();
}

}  // namespace sv
