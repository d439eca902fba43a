// Device helpers shared by the libspecverify kernels: vector loads, bf16
// unpacking, NaN-aware maxima, and the (max, scaled-sum, argmax) monoid used
// to merge partial row statistics.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "sv_internal.h"

namespace sv {

constexpr float kInfF = __builtin_huge_valf();

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
// Bulk copies (TMA engine) and mbarriers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Announce `bytes` of incoming bulk-copy data without arriving (the arrival
// comes later, once the stage's description is written).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity, for at most about
// `limit_ns`; gives up early once *abort is set.  Returns false if it gave up.
// Between polls the warp sleeps about `sleep_ns` (0: poll back to back):
// warps that poll without pause take issue slots from the warps doing work.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  uint64_t limit_ns, uint32_t sleep_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (sleep_ns) __nanosleep(sleep_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// One bulk copy global -> shared, completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Start pulling `bytes` (a multiple of 16, 16-byte aligned) into L2 without waiting.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}

// Programmatic dependent launch: wait until the kernels this one depends on
// (earlier work on the stream) have completed and their writes are visible;
// and let the next kernel on the stream begin launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Ticket on a counter at GPU scope with release and acquire semantics: the
// caller's earlier writes (and, through a preceding barrier, its block's) are
// visible before the increment, and reads after it see the writes other
// arrivals made before theirs.
__device__ __forceinline__ unsigned ticket_add(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Barrier among the first `threads` threads of the block (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int threads) { asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory"); }

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

// log2(e)/T in fp32, or 0 for a greedy temperature.  log2(e) is split into
// a head and a tail float; the head's quotient is corrected with its exact
// remainder (one fused multiply-add), which brings the result within an ulp
// of the exact quotient without fp64 (whose dependent latency is long here).
__device__ __forceinline__ float temperature_k(float T) {
  const bool sampling = (T >= 1e-30f) && (T < kInfF);
  if (!sampling) return 0.0f;
  constexpr float kHi = 1.44269502162933349609375f;  // fp32 nearest to log2(e)
  constexpr float kLo = 1.925963033500011e-08f;      // log2(e) - kHi
  const float q = __fdiv_rn(kHi, T);
  const float r = fmaf(-q, T, kHi) + kLo;  // remainder of the head (exact) plus the tail
  return fmaf(r, __frcp_rn(T), q);
}

__device__ __forceinline__ bool sampling_temperature(float T) { return (T >= 1e-30f) && (T < kInfF); }

// ---------------------------------------------------------------------------
// Partial row statistics: (m, s, idx, flags) with s = sum 2^((l - m) k)
// ---------------------------------------------------------------------------

// In-CTA partial (fp32).  Merged in double only across CTAs.
struct Part {
  float m;
  float s;
  int32_t idx;
  uint32_t flags;
};

__device__ __forceinline__ Part part_identity() { return Part{-kInfF, 0.0f, -1, 0u}; }

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
  float s = 0.0f;
  if (k > 0.0f && M > -kInfF) {
    const float sa = (a.m == M) ? a.s : (a.s != 0.0f ? a.s * exp2f((a.m - M) * k) : 0.0f);
    const float sb = (b.m == M) ? b.s : (b.s != 0.0f ? b.s * exp2f((b.m - M) * k) : 0.0f);
    s = sa + sb;
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

// Reduce over the first NT threads (whole warps) with the named barrier; the
// result is valid in every thread of warp 0.
template <int NT>
__device__ __forceinline__ Part part_reduce_named(Part p, float k, Part* smem /* [NT/32] */) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  p = part_warp_reduce(p, k);
  if (lane == 0) smem[warp] = p;
  named_sync(NT);
  if (warp == 0) {
    p = lane < NW ? smem[lane] : part_identity();
    p = part_warp_reduce(p, k);
  }
  named_sync(NT);
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

// x >= 0 (a sum of sampling weights, below 2^18) as fixed point with
// kFixedBits fractional bits, rounded to nearest; monotone in x.
__device__ __forceinline__ uint64_t to_fixed(float x) {
  const uint32_t bits = __float_as_uint(x);
  const int e = static_cast<int>((bits >> 23) & 0xffu);
  if (e == 0) return 0ull;  // zero (and sub-normals, far below one unit)
  const uint64_t mant = static_cast<uint64_t>((bits & 0x7fffffu) | 0x800000u);
  const int sh = e - 127 - 23 + kFixedBits;  // value = mant * 2^sh
  if (sh >= 0) return mant << sh;
  if (sh <= -25) return 0ull;
  return (mant + (1ull << (-sh - 1))) >> (-sh);
}

// floor(u * S) for u in [0, 1) (any fp32) and a fixed-point total S < 2^62.
__device__ __forceinline__ uint64_t scale_fixed(float u, uint64_t S) {
  const uint32_t bits = __float_as_uint(u);
  const int e = static_cast<int>((bits >> 23) & 0xffu);
  if (e == 0 || (bits >> 31)) return 0ull;  // zero, sub-normal or negative
  const uint64_t mant = static_cast<uint64_t>((bits & 0x7fffffu) | 0x800000u);
  const int sh = 127 + 23 - e;  // u = mant * 2^-sh, sh >= 24 for u < 1
  const uint64_t lo = mant * S, hi = __umul64hi(mant, S);
  if (sh >= 128) return 0ull;
  if (sh >= 64) return hi >> (sh - 64);
  return (hi << (64 - sh)) | (lo >> sh);
}

// Exact warp sum of values below 2^59: the low 27 bits and the rest are summed
// as 32-bit words by the warp-reduce unit (neither part can overflow 32 lanes).
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
  const unsigned lo = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(v & ((1ull << 27) - 1)));
  const unsigned hi = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(v >> 27));
  return (static_cast<uint64_t>(hi) << 27) + lo;
}

__device__ __forceinline__ uint64_t warp_inclusive_scan_u64(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint64_t t = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += t;
  }
  return v;
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
