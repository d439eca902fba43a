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
// CTA order (deterministic) and resets the counter.  No CTA ever waits.
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kStatsThreads = 256;

template <int DT>
struct VecTraits;
template <>
struct VecTraits<SV_BF16> {
  static constexpr int E = 8;   // elements per 16-byte vector
  static constexpr int ES = 2;  // element bytes
  static constexpr int U = 4;   // vectors in flight per thread
};
template <>
struct VecTraits<SV_F32> {
  static constexpr int E = 4;
  static constexpr int ES = 4;
  static constexpr int U = 4;
};

// Per-thread running statistics.  The scaled sum uses Kahan compensation so
// its error does not grow with the number of vectors a thread visits.
struct ThreadAcc {
  float m;
  float s;
  float c;
  int32_t idx;
  uint32_t flags;
};

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

// Fold E consecutive logits starting at column col0 into the accumulator.
template <int E, bool EXP>
__device__ __forceinline__ void consume(ThreadAcc& a, float (&x)[E], float vmax_nan, int64_t col0, float k) {
  float vmax = vmax_nan;
  if (!(vmax_nan < kInfF)) {  // NaN or +inf present: exclude those entries
    vmax = -kInfF;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if (!usable_logit(x[i])) {
        x[i] = -kInfF;
        a.flags |= kStNonFinite;
      }
      vmax = fmaxf(vmax, x[i]);
    }
  }
  if (vmax > a.m) {  // new running maximum (rare after the first vectors)
    if (EXP && a.m > -kInfF) {
      const float f = exp2f((a.m - vmax) * k);
      a.s *= f;
      a.c *= f;
    }
    a.m = vmax;
    int j = E - 1;
#pragma unroll
    for (int i = E - 1; i >= 0; --i)
      if (x[i] == vmax) j = i;
    a.idx = static_cast<int32_t>(col0 + j);
  }
  if (EXP && a.m > -kInfF) {
    float e[E];
#pragma unroll
    for (int i = 0; i < E; ++i) e[i] = ex2_fast((x[i] - a.m) * k);
    float vs;
    if constexpr (E == 8) {
      vs = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    } else {
      vs = (e[0] + e[1]) + (e[2] + e[3]);
    }
    const float y = vs - a.c;
    const float t = a.s + y;
    a.c = (t - a.s) - y;
    a.s = t;
  }
}

// Scan vectors [v0, v1) of one row (vector index within the row).
template <int DT, bool EXP>
__device__ __forceinline__ void scan_row_range(const LogitsView& lg, int64_t row, int64_t v0, int64_t v1, float k,
                                               ThreadAcc& a) {
  using VT = VecTraits<DT>;
  constexpr int E = VT::E, U = VT::U, BS = kStatsThreads;
  const char* rowp = static_cast<const char*>(lg.base) + row * lg.ld * VT::ES;
  const int64_t nfull = lg.vocab / E;  // vectors entirely inside the row
  const int64_t vend = v1 < nfull ? v1 : nfull;
  int64_t v = v0 + threadIdx.x;
  for (; v + (U - 1) * BS < vend; v += U * BS) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) raw[u] = ld_stream16(rowp + (v + u * BS) * 16);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float x[E];
      unpack<DT>(raw[u], x);
      consume<E, EXP>(a, x, raw_max_nan<DT>(raw[u]), (v + u * BS) * E, k);
    }
  }
  for (; v < v1; v += BS) {
    float x[E];
    float vmax;
    if (v < nfull) {
      const uint4 raw = ld_stream16(rowp + v * 16);
      unpack<DT>(raw, x);
      vmax = raw_max_nan<DT>(raw);
    } else {  // the row's ragged tail: element loads, padding is -inf
      vmax = -kInfF;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int64_t col = v * E + i;
        x[i] = col < lg.vocab ? load_logit(lg, row, col) : -kInfF;
        vmax = fmax_nan(vmax, x[i]);
      }
    }
    consume<E, EXP>(a, x, vmax, v * E, k);
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

template <int DT>
__global__ void __launch_bounds__(kStatsThreads) k_row_stats(LogitsView lg, RowMap map, Ws ws, int64_t NVr,
                                                             int64_t NV) {
  __shared__ Part s_red[kStatsThreads / 32];
  __shared__ float s_k;
  __shared__ int s_last;
  const int64_t G = gridDim.x, c = blockIdx.x;
  const int64_t v_begin = c * NV / G, v_end = (c + 1) * NV / G;
  if (v_begin >= v_end) return;
  const int64_t r_first = v_begin / NVr, r_last = (v_end - 1) / NVr;

  for (int64_t row = r_first; row <= r_last; ++row) {
    const int64_t row_v0 = row * NVr;
    const int64_t s0 = (v_begin > row_v0 ? v_begin : row_v0) - row_v0;
    const int64_t s1 = (v_end < row_v0 + NVr ? v_end : row_v0 + NVr) - row_v0;
    if (threadIdx.x == 0) s_k = row_k(map, row);
    __syncthreads();
    const float k = s_k;

    ThreadAcc a{-kInfF, 0.0f, 0.0f, -1, 0u};
    if (k > 0.0f) {
      scan_row_range<DT, true>(lg, row, s0, s1, k, a);
    } else {
      scan_row_range<DT, false>(lg, row, s0, s1, k, a);
    }
    Part p{a.m, static_cast<double>(a.s) - static_cast<double>(a.c), a.idx, a.flags};
    p = part_block_reduce<kStatsThreads>(p, k, s_red);

    const int64_t c_lo = cta_of_vector(row_v0, G, NV);
    const int64_t c_hi = cta_of_vector(row_v0 + NVr - 1, G, NV);
    if (c_lo == c_hi) {  // the whole row is ours
      if (threadIdx.x == 0) {
        RowStat st;
        st.Z = (k > 0.0f && p.m > -kInfF) ? p.s : 0.0;
        st.M = p.m;
        st.argmax = p.idx;
        st.flags = p.flags;
        st.k = k;
        ws.rowstat[row] = st;
      }
      continue;
    }
    if (threadIdx.x == 0) {
      RowPartial rp;
      rp.s = p.s;
      rp.m = p.m;
      rp.idx = p.idx;
      rp.flags = p.flags;
      rp.pad = 0u;
      ws.partial[2 * c + (row == r_first ? 0 : 1)] = rp;
      __threadfence();
      const unsigned ticket = atomicAdd(&ws.row_cnt[row], 1u);
      s_last = (ticket == static_cast<unsigned>(c_hi - c_lo));
    }
    __syncthreads();
    if (s_last && threadIdx.x < 32) {  // last arriver: merge the row's partials in CTA order
      __threadfence();
      const int lane = threadIdx.x;
      Part acc = part_identity();
      for (int64_t cc = c_lo + lane; cc <= c_hi; cc += 32) {
        const int64_t first_row_cc = (cc * NV / G) / NVr;
        const Part q = load_partial_cg(&ws.partial[2 * cc + (row == first_row_cc ? 0 : 1)]);
        part_merge(acc, q, k);
      }
      acc = part_warp_reduce(acc, k);
      if (lane == 0) {
        RowStat st;
        st.Z = (k > 0.0f && acc.m > -kInfF) ? acc.s : 0.0;
        st.M = acc.m;
        st.argmax = acc.idx;
        st.flags = acc.flags;
        st.k = k;
        ws.rowstat[row] = st;
        ws.row_cnt[row] = 0u;  // leave the counter clean for the next call
      }
    }
    __syncthreads();
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
  if (row_flags) row_flags[row] = st.flags;
  if (out_p) {
    float p = 0.0f;
    if (probe && st.k > 0.0f && st.argmax >= 0) {
      const int32_t t = probe[row];
      if (t >= 0 && t < lg.vocab) {
        const float l = load_logit(lg, row, t);
        if (usable_logit(l)) p = static_cast<float>(static_cast<double>(exp2f((l - st.M) * st.k)) / st.Z);
      }
    }
    out_p[row] = p;
  }
}

}  // namespace

cudaError_t stats_occupancy(int dtype, int* blocks_per_sm) {
  if (dtype == SV_BF16)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_row_stats<SV_BF16>, kStatsThreads, 0);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_row_stats<SV_F32>, kStatsThreads, 0);
}

int stats_grid(const DeviceInfo& dev, const LogitsView& lg) {
  const int E = lg.dtype == SV_BF16 ? 8 : 4;
  const int64_t NVr = (lg.vocab + E - 1) / E;
  const int64_t NV = NVr * lg.rows;
  // One resident wave; at least ~2 vectors per thread per CTA; never more CTAs than vectors.
  int64_t g = static_cast<int64_t>(dev.sms) * dev.stats_blocks_per_sm[lg.dtype == SV_BF16 ? 1 : 0];
  const int64_t by_work = (NV + 2 * kStatsThreads - 1) / (2 * kStatsThreads);
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
    k_row_stats<SV_BF16><<<grid, kStatsThreads, 0, stream>>>(lg, map, ws, NVr, NV);
  } else {
    k_row_stats<SV_F32><<<grid, kStatsThreads, 0, stream>>>(lg, map, ws, NVr, NV);
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
