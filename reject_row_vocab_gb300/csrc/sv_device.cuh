// Device helpers shared by the libspecverify kernels: vector loads, bf16
// unpacking, NaN-aware maxima, and the (max, scaled-sum, argmax) monoid used
// to merge partial row statistics.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "sv_internal.h"

namespace sv {

constexpr float kInfF = __builtin_huge_valf();
constexpr double kLog2eD = 1.4426950408889634074;

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------

// 16-byte streaming load through the non-coherent path, not kept in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One logit as float (exact widening for bf16).
__device__ __forceinline__ float load_logit(const LogitsView& lg, int64_t row, int64_t col) {
  const int64_t i = row * lg.ld + col;
  if (lg.dtype == SV_BF16) {
    const uint16_t b = __ldg(static_cast<const unsigned short*>(lg.base) + i);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  return __ldg(static_cast<const float*>(lg.base) + i);
}

// ---------------------------------------------------------------------------
// Arithmetic helpers
// ---------------------------------------------------------------------------

// max that propagates NaN (IEEE fmaxf would drop it).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 2^x on the special-function unit (flushes sub-normal results to zero).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool usable_logit(float x) { return !(x != x) && x != kInfF; }

// log2(e)/T rounded once to fp32, or 0 for a greedy temperature.
__device__ __forceinline__ float temperature_k(float T) {
  const bool sampling = (T >= 1e-30f) && (T < kInfF);
  return sampling ? static_cast<float>(kLog2eD / static_cast<double>(T)) : 0.0f;
}

__device__ __forceinline__ bool sampling_temperature(float T) { return (T >= 1e-30f) && (T < kInfF); }

// ---------------------------------------------------------------------------
// Partial row statistics: (m, s, idx, flags) with s = sum 2^((l - m) k)
// ---------------------------------------------------------------------------

struct Part {
  float m;
  double s;
  int32_t idx;
  uint32_t flags;
};

__device__ __forceinline__ Part part_identity() { return Part{-kInfF, 0.0, -1, 0u}; }

// Merge b into a.  The larger maximum wins its index; equal maxima keep the
// lower index; sums are rescaled to the common maximum (exactly 1 for the
// side that already holds it).
__device__ __forceinline__ void part_merge(Part& a, const Part& b, float k) {
  const float M = fmaxf(a.m, b.m);
  int32_t idx;
  if (a.m > b.m) {
    idx = a.idx;
  } else if (b.m > a.m) {
    idx = b.idx;
  } else {
    idx = min(a.idx, b.idx);
  }
  double s = 0.0;
  if (k > 0.0f && M > -kInfF) {
    if (a.m == M) {
      s += a.s;
    } else if (a.s != 0.0) {
      s += a.s * static_cast<double>(exp2f((a.m - M) * k));
    }
    if (b.m == M) {
      s += b.s;
    } else if (b.s != 0.0) {
      s += b.s * static_cast<double>(exp2f((b.m - M) * k));
    }
  }
  a.m = M;
  a.s = s;
  a.idx = idx;
  a.flags |= b.flags;
}

__device__ __forceinline__ Part part_shfl_xor(const Part& p, int lanemask) {
  Part o;
  o.m = __shfl_xor_sync(0xffffffffu, p.m, lanemask);
  o.s = __shfl_xor_sync(0xffffffffu, p.s, lanemask);
  o.idx = __shfl_xor_sync(0xffffffffu, p.idx, lanemask);
  o.flags = __shfl_xor_sync(0xffffffffu, p.flags, lanemask);
  return o;
}

// Butterfly reduction: every lane ends with the same, order-fixed result.
__device__ __forceinline__ Part part_warp_reduce(Part p, float k) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Part o = part_shfl_xor(p, off);
    part_merge(p, o, k);
  }
  return p;
}

// Reduce over the whole block; the result is valid in every thread of warp 0.
template <int BS>
__device__ __forceinline__ Part part_block_reduce(Part p, float k, Part* smem /* [BS/32] */) {
  constexpr int NW = BS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  p = part_warp_reduce(p, k);
  if (lane == 0) smem[warp] = p;
  __syncthreads();
  if (warp == 0) {
    p = lane < NW ? smem[lane] : part_identity();
    p = part_warp_reduce(p, k);
  }
  __syncthreads();
  return p;
}

// Coherent (L2) loads of a partial written by another CTA.
__device__ __forceinline__ Part load_partial_cg(const RowPartial* rp) {
  Part p;
  p.s = __ldcg(&rp->s);
  p.m = __ldcg(&rp->m);
  p.idx = __ldcg(&rp->idx);
  p.flags = __ldcg(&rp->flags);
  return p;
}

// Warp-wide inclusive scan of doubles in lane order.
__device__ __forceinline__ double warp_inclusive_scan(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += t;
  }
  return v;
}

__device__ __forceinline__ double warp_sum_xor(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

}  // namespace sv
