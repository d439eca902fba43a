// Row statistics: one streaming pass over every logits row.
//
// For each verify row the pass produces the maximum M, its lowest index (the
// greedy argmax, [E2D] §1.2 first bullet) and, for sampling rows,
// Z = sum_v 2^((l_v - M) * log2(e)/T), the normaliser of softmax(l/T)
// ([E2D] §6.2).  [E2D] = "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理".
//
// Work split: rows are cut into stages of 1024 16-byte vectors (16 KB) and
// stages into chunks, the unit of scheduling and of partial results.  Most
// rows use chunks of up to eight stages; the last rows, about three chunks'
// worth per CTA, use one-stage chunks, so CTAs that run out of work at
// different times are evened out by small pieces (the layout depends only on
// the shapes and the grid).  One resident wave of CTAs takes chunks from a
// queue: a CTA's first chunk is its own index, later ones come from an atomic
// counter, requested two chunks ahead.  Per CTA, a producer warp streams
// stages into a four-stage shared-memory ring with bulk copies (the TMA
// engine; completion counted on an mbarrier per stage), eight consumer warps
// fold each stage with packed fp32x2 arithmetic against an exponent reference
// that moves only when a logit grows 16 log2 units past it (then once, to the
// stage's maximum, so the stage stays on the packed path), and at the end of
// a chunk each warp combines its lanes and hands the result to a finalizer
// warp, which finds the chunk's argmax element in the one vector the warp
// results point to and writes the chunk's partial (maximum, its lowest index,
// the sum rescaled to the maximum, flags).  k_row_merge then merges each row's
// chunk partials in chunk order, so the result does not depend on which CTA
// streamed what.  No CTA waits on another.  Every mbarrier wait is bounded (one
// second); a timeout raises the workspace error word, reported by the next
// kernels as SV_DEV_TIMEOUT.
#include <atomic>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kConsumers = 256;                      // eight consumer warps
constexpr int kConsumerWarps = kConsumers / 32;
constexpr int kProducerWarp = kConsumerWarps;        // warp 8 streams the stages
constexpr int kFinalizerWarp = kProducerWarp + 1;    // warp 9 merges partials
constexpr int kStatsThreads = kConsumers + 64;
constexpr int kChunkVecs = 1024;                     // 16 KB per stage
constexpr int kStages = 4;
constexpr int kHeadChunkStages = 8;                  // chunks of the head rows span up to eight stages
constexpr int kTailRounds = 3;                       // tail rows hold about this many one-stage chunks per CTA
constexpr int kSlots = 4;                            // chunk partials in flight to the finalizer
constexpr int kTabCap = 512;                         // request tables staged in shared memory up to this size
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kProducerNap = 32;   // ns between polls: the producer's reaction time matters
constexpr uint32_t kConsumerNap = 128;  // consumers and finalizer mostly wait for memory

// What the producer tells the consumers about one stage.
struct StageMeta {
  int32_t item;  // chunk index in the queue, -1 marks the end
  int32_t row;
  int32_t c0;    // first vector of the stage within the row
  int32_t n;     // full vectors in the stage
  float k;       // log2(e)/T of the row (0: greedy row, no sums)
  float ik;      // 1/k (0 for greedy rows)
  int32_t nst;   // stages in this chunk
  int32_t tail;  // 1: the row's ragged tail vector follows this chunk
  int32_t probe; // probe-aware pass: the row's probe token when it lies in this chunk, else -1
};

// How rows are cut into chunks (queue items).  Head rows [0, rows_a) are cut
// into cpr_a nearly equal chunks of up to kHeadChunkStages stages (few queue
// and bookkeeping operations per byte); the remaining tail rows into one-stage
// chunks (fine-grained work for the end of the pass, when CTAs run out of
// queue at different times).  Items are numbered head rows first, so the
// queue hands out the coarse work first.  The layout depends only on the
// shapes and the grid, so the merge order of every row is fixed.
struct ChunkPlan {
  int32_t nst;     // stages (1024-vector pieces) per row, at least 1
  int32_t cpr_a;   // chunks per head row
  int32_t rows_a;  // head rows
  int32_t cpr_b;   // chunks per tail row (= nst)
  int64_t n_a;     // items in the head rows
  int64_t n_items;
};

// Row, stage range [s0, s1) and "last chunk of its row" of a queue item.
__host__ __device__ __forceinline__ void chunk_geometry(const ChunkPlan& P, int32_t item, int32_t& row, int32_t& s0,
                                                        int32_t& s1, bool& last) {
  if (item < P.n_a) {
    row = item / P.cpr_a;
    const int32_t ci = item - row * P.cpr_a;
    s0 = ci * P.nst / P.cpr_a;
    s1 = (ci + 1) * P.nst / P.cpr_a;
    last = ci == P.cpr_a - 1;
  } else {
    const int32_t j = item - static_cast<int32_t>(P.n_a);
    const int32_t r = j / P.cpr_b;
    const int32_t ci = j - r * P.cpr_b;
    row = P.rows_a + r;
    s0 = ci;
    s1 = ci + 1;
    last = ci == P.cpr_b - 1;
  }
}

// One chunk's per-warp partials, handed from the consumers to the finalizer.
struct ChunkSlot {
  Part wpart[kConsumerWarps];
  float wsb[kConsumerWarps];  // probe chunk: per-warp sums below the probe, at the warp maximum
  int32_t item;
  int32_t row;
  float k;
  int32_t pad;
};

struct StatsSmem {
  uint4 buf[kStages][kChunkVecs];
  StageMeta meta[kStages];
  ChunkSlot slot[kSlots];
  float tab_k[kTabCap];    // log2(e)/T by request (or by row)
  float tab_ik[kTabCap];   // T/log2(e), the reciprocal of tab_k (0 for greedy rows)
  int32_t tab_cu[kTabCap]; // request offsets of a ragged layout
  unsigned long long tab_ready;
  unsigned long long never;            // no thread ever arrives: the expiry test waits on it
  unsigned long long full[kStages];    // producer -> consumers (bulk-copy bytes)
  unsigned long long empty[kStages];   // consumers -> producer
  unsigned long long pfull[kSlots];    // consumers -> finalizer
  unsigned long long pempty[kSlots];   // finalizer -> consumers
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

// Per-thread running statistics of one chunk: the maximum m, the first vector
// (within the row) where it was reached (its element is found once per row,
// at the end), flags, and a packed fp32 accumulator of 2^(l k - R) against a
// reference R in log2 units.  R only moves when a logit reaches `bound`
// (about R + 16 log2 units), so most vectors need no rescale and every term is
// one fused multiply-add and one exponential.
struct ThreadAcc {
  float m;
  int32_t vidx;  // -1 while no usable entry has been seen
  uint32_t flags;
  float R;
  float bound;   // logits >= bound move the reference (+inf for greedy rows)
  float2 s;
  float sb;      // probe chunk only: the part of s over ids below the probe
};

constexpr float kRefSlack = 16.0f;  // terms stay <= 2^16 between reference moves
constexpr float kMinFinite = -3.402823466e38f;

template <bool EXP>
__device__ __forceinline__ ThreadAcc acc_init() {
  return ThreadAcc{-kInfF, -1, 0u, 0.0f, EXP ? kMinFinite : kInfF, make_float2(0.0f, 0.0f), 0.0f};
}

// Move the reference up to the finite logit v (rare path).
__device__ __forceinline__ void move_ref(ThreadAcc& a, float v, float k, float ik) {
  const float Rn = v * k;
  if (!(fabsf(Rn) < kInfF)) {  // l * log2(e)/T outside fp32: no meaningful sum
    a.flags |= kStNonFinite;
    a.bound = kInfF;
    return;
  }
  const bool have = a.s.x != 0.0f || a.s.y != 0.0f;
  const float f = have ? exp2f(a.R - Rn) : 0.0f;
  a.s = __fmul2_rn(a.s, make_float2(f, f));
  a.sb *= f;
  a.R = Rn;
  a.bound = (Rn + kRefSlack) * ik;
}

// Order-preserving map of a float (never NaN here) to an unsigned key.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}
__device__ __forceinline__ float warp_max(float m) {
  return key_float(__reduce_max_sync(0xffffffffu, order_key(m)));
}

// Combine one partial per lane into the warp's, given the warp maximum M and
// each lane's log2 factor e that rescales its sum s to M: the sum of the
// rescaled sums (the butterfly leaves the same value in every lane), the
// lowest vector holding M, and the union of the flags.
__device__ __forceinline__ Part warp_combine(float M, float m, float s, float e, int32_t vidx, uint32_t flags) {
  float sc = s != 0.0f ? (e == 0.0f ? s : s * exp2f(e)) : 0.0f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
  const int32_t V = __reduce_min_sync(0xffffffffu, (m == M && vidx >= 0) ? vidx : INT32_MAX);
  return Part{M, sc, V == INT32_MAX ? -1 : V, __reduce_or_sync(0xffffffffu, flags)};
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

// Sum of 2^(x k - R) over E elements, as a packed pair (fixed order).
template <int E>
__device__ __forceinline__ float2 exp_sum(const float (&x)[E], float k, float R) {
  const float2 kk = make_float2(k, k), nR = make_float2(-R, -R);
  float2 e[E / 2];
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    const float2 t = __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]), kk, nR);
    e[i] = make_float2(ex2_fast(t.x), ex2_fast(t.y));
  }
  if constexpr (E == 8) {
    return __fadd2_rn(__fadd2_rn(e[0], e[1]), __fadd2_rn(e[2], e[3]));
  } else {
    return __fadd2_rn(e[0], e[1]);
  }
}

// Fold E logits one at a time, NaN and +inf entries read as -inf (the caller
// flags them).
template <int E, bool EXP>
__device__ __forceinline__ void consume_dirty(ThreadAcc& a, const float (&x)[E], int32_t vec, float k, float ik) {
  for (int i = 0; i < E; ++i) {
    const float v = usable_logit(x[i]) ? x[i] : -kInfF;
    if (v > a.m) {
      a.m = v;
      a.vidx = vec;
    }
    if (EXP) {
      if (v >= a.bound) move_ref(a, v, k, ik);
      a.s.x += ex2_fast(fmaf(v, k, -a.R));
    }
  }
}

// Fold one vector.  The common case (clean data, maximum below the bound) is
// branch-free.
template <int DT, bool EXP>
__device__ __forceinline__ void consume(ThreadAcc& a, const uint4& raw, int32_t vec, float k, float ik) {
  constexpr int E = VecTraits<DT>::E;
  float x[E];
  unpack<DT>(raw, x);
  const float vmax = raw_max_nan<DT>(raw);
  if (!(vmax < a.bound)) {  // NaN / +inf present, or the reference must move (rare)
    if (!(vmax < kInfF)) {
      a.flags |= kStNonFinite;
      consume_dirty<E, EXP>(a, x, vec, k, ik);
      return;
    }
    if (EXP) move_ref(a, vmax, k, ik);
  }
  const bool raised = vmax > a.m;
  a.vidx = raised ? vec : a.vidx;
  a.m = fmaxf(a.m, vmax);
  if (EXP) {
    a.s = __fadd2_rn(a.s, exp_sum<E>(x, k, a.R));
  }
}

// Probe-aware folding (one chunk per row): as above, and the terms of ids
// below the probe token d are also added to a.sb.
template <int E>
__device__ __forceinline__ void consume_dirty_probe(ThreadAcc& a, const float (&x)[E], int32_t vec, float k, float ik,
                                                    int32_t d) {
  for (int i = 0; i < E; ++i) {
    const float v = usable_logit(x[i]) ? x[i] : -kInfF;
    if (v > a.m) {
      a.m = v;
      a.vidx = vec;
    }
    if (v >= a.bound) move_ref(a, v, k, ik);
    const float t = ex2_fast(fmaf(v, k, -a.R));
    a.s.x += t;
    if (vec * E + i < d) a.sb += t;
  }
}

// The terms of one clean vector (maximum below the bound), those of ids below d also to a.sb.
template <int E>
__device__ __forceinline__ void probe_vector_terms(ThreadAcc& a, const float (&x)[E], int32_t vec, float k,
                                                   int32_t d) {
  const float2 kk = make_float2(k, k), nR = make_float2(-a.R, -a.R);
  float t[E];
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float2 y = __ffma2_rn(make_float2(x[i], x[i + 1]), kk, nR);
    t[i] = ex2_fast(y.x);
    t[i + 1] = ex2_fast(y.y);
  }
  float tot = 0.0f, below = 0.0f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    tot += t[i];
    if (vec * E + i < d) below += t[i];
  }
  a.s.x += tot;
  a.sb += below;
}

template <int DT>
__device__ __forceinline__ void consume_probe(ThreadAcc& a, const uint4& raw, int32_t vec, float k, float ik,
                                              int32_t d) {
  constexpr int E = VecTraits<DT>::E;
  float x[E];
  unpack<DT>(raw, x);
  const float vmax = raw_max_nan<DT>(raw);
  if (!(vmax < a.bound)) {
    if (!(vmax < kInfF)) {
      a.flags |= kStNonFinite;
      consume_dirty_probe<E>(a, x, vec, k, ik, d);
      return;
    }
    move_ref(a, vmax, k, ik);
  }
  a.vidx = vmax > a.m ? vec : a.vidx;
  a.m = fmaxf(a.m, vmax);
  probe_vector_terms<E>(a, x, vec, k, d);
}

// The row's ragged tail (vocab not a multiple of the vector width) as vector nfull, by one thread.
template <int DT, bool EXP>
__device__ __forceinline__ void fold_tail(ThreadAcc& a, const LogitsView& lg, int64_t row, int64_t nfull, float k,
                                          float ik) {
  constexpr int E = VecTraits<DT>::E;
  float x[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int64_t col = nfull * E + i;
    x[i] = col < lg.vocab ? load_logit(lg, row, col) : -kInfF;
    if (col < lg.vocab && !usable_logit(x[i])) a.flags |= kStNonFinite;
  }
  consume_dirty<E, EXP>(a, x, static_cast<int32_t>(nfull), k, ik);
}

template <int DT>
__device__ __forceinline__ void fold_tail_probe(ThreadAcc& a, const LogitsView& lg, int64_t row, int64_t nfull, float k,
                                                float ik, int32_t d) {
  constexpr int E = VecTraits<DT>::E;
  float x[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int64_t col = nfull * E + i;
    x[i] = col < lg.vocab ? load_logit(lg, row, col) : -kInfF;
    if (col < lg.vocab && !usable_logit(x[i])) a.flags |= kStNonFinite;
  }
  consume_dirty_probe<E>(a, x, static_cast<int32_t>(nfull), k, ik, d);
}

// NaN-propagating maximum of PER raw vectors (packed bf16 pairs reduced as pairs until the last step).
template <int DT, int PER>
__device__ __forceinline__ float raw_max_nan_n(const uint4 (&raw)[PER]) {
  if constexpr (DT == SV_BF16) {
    uint32_t w = bmax2_nan(bmax2_nan(raw[0].x, raw[0].y), bmax2_nan(raw[0].z, raw[0].w));
#pragma unroll
    for (int j = 1; j < PER; ++j)
      w = bmax2_nan(w, bmax2_nan(bmax2_nan(raw[j].x, raw[j].y), bmax2_nan(raw[j].z, raw[j].w)));
    return fmax_nan(bf16_lo(w), bf16_hi(w));
  } else {
    float m = raw_max_nan<DT>(raw[0]);
#pragma unroll
    for (int j = 1; j < PER; ++j) m = fmax_nan(m, raw_max_nan<DT>(raw[j]));
    return m;
  }
}

// Fold the first n vectors of a stage (vectors c0.. of the row).  A full
// stage takes the thread's four vectors together: one maximum over all four
// (packed) is checked against the bound and against the running maximum;
// when it reaches the bound the reference moves once, to that maximum; only
// when the running maximum grows (rare after the first stages) is the first
// vector holding it looked for.  The sums run branch-free.
template <int DT, bool EXP>
__device__ __forceinline__ void fold_stage(ThreadAcc& a, uint32_t stage_addr, int32_t c0, int n, float k, float ik) {
  constexpr int E = VecTraits<DT>::E;
  constexpr int PER = kChunkVecs / kConsumers;  // vectors per consumer thread per full stage
  const int t = threadIdx.x;
  if (n == kChunkVecs) {
    uint4 raw[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) raw[j] = lds16(stage_addr + (t + j * kConsumers) * 16);
    const float smax = raw_max_nan_n<DT, PER>(raw);
    if (!(smax < a.bound)) {
      if (!EXP || !(smax < kInfF)) {  // NaN / +inf present: vector by vector (rare)
#pragma unroll
        for (int j = 0; j < PER; ++j) consume<DT, EXP>(a, raw[j], c0 + t + j * kConsumers, k, ik);
        return;
      }
      // The reference moves (a chunk's first stage, or a logit far above the running maximum, frequent at low
      // temperatures): once, to the stage maximum, so every term of the stage is at most 1.
      move_ref(a, smax, k, ik);
    }
    if (smax > a.m) {  // the first of the four vectors that reaches the new maximum
      int32_t v = c0 + t + (PER - 1) * kConsumers;
#pragma unroll
      for (int j = PER - 2; j >= 0; --j)
        if (raw_max_nan<DT>(raw[j]) == smax) v = c0 + t + j * kConsumers;
      a.vidx = v;
      a.m = smax;
    }
    if (EXP) {
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        float x[E];
        unpack<DT>(raw[j], x);
        a.s = __fadd2_rn(a.s, exp_sum<E>(x, k, a.R));
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int vi = t + j * kConsumers;
      if (vi < n) consume<DT, EXP>(a, lds16(stage_addr + vi * 16), c0 + vi, k, ik);
    }
  }
}

// The stage holding the probe's vector pv = d / E: folded like any full stage,
// and the terms of vectors below pv, and of the ids below d inside pv (one
// thread's vector), also go to a.sb.  A partial stage goes vector by vector.
template <int DT>
__device__ __forceinline__ void fold_stage_probe(ThreadAcc& a, uint32_t stage_addr, int32_t c0, int n, float k,
                                                 float ik, int32_t d) {
  constexpr int E = VecTraits<DT>::E;
  constexpr int PER = kChunkVecs / kConsumers;
  const int t = threadIdx.x;
  const int32_t pv = d / E;
  if (n == kChunkVecs) {
    uint4 raw[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) raw[j] = lds16(stage_addr + (t + j * kConsumers) * 16);
    const float smax = raw_max_nan_n<DT, PER>(raw);
    if (!(smax < a.bound)) {
      if (!(smax < kInfF)) {  // NaN / +inf present: vector by vector
#pragma unroll
        for (int j = 0; j < PER; ++j) consume_probe<DT>(a, raw[j], c0 + t + j * kConsumers, k, ik, d);
        return;
      }
      move_ref(a, smax, k, ik);
    }
    if (smax > a.m) {
      int32_t v = c0 + t + (PER - 1) * kConsumers;
#pragma unroll
      for (int j = PER - 2; j >= 0; --j)
        if (raw_max_nan<DT>(raw[j]) == smax) v = c0 + t + j * kConsumers;
      a.vidx = v;
      a.m = smax;
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int32_t vec = c0 + t + j * kConsumers;
      float x[E];
      unpack<DT>(raw[j], x);
      if (vec != pv) {
        const float2 es = exp_sum<E>(x, k, a.R);
        a.s = __fadd2_rn(a.s, es);
        if (vec < pv) a.sb += es.x + es.y;
      } else {
        probe_vector_terms<E>(a, x, vec, k, d);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int vi = t + j * kConsumers;
      if (vi < n) consume_probe<DT>(a, lds16(stage_addr + vi * 16), c0 + vi, k, ik, d);
    }
  }
}

// The index of the first entry equal to M in vector vidx of a row (the ragged
// tail when vidx == nfull), read back from global memory once per row.
template <int DT>
__device__ __forceinline__ int32_t resolve_index(const LogitsView& lg, int64_t row, int64_t nfull, int32_t vidx,
                                                 float M) {
  constexpr int E = VecTraits<DT>::E;
  if (vidx < 0) return -1;
  float x[E];
  if (vidx < nfull) {
    const uint4 raw = ld_stream16(reinterpret_cast<const uint4*>(static_cast<const char*>(lg.base) +
                                                                 row * lg.ld * VecTraits<DT>::ES) +
                                  vidx);
    unpack<DT>(raw, x);
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int64_t col = static_cast<int64_t>(vidx) * E + i;
      x[i] = col < lg.vocab ? load_logit(lg, row, col) : -kInfF;
    }
  }
  int j = E - 1;
#pragma unroll
  for (int i = E - 1; i >= 0; --i)
    if (x[i] == M) j = i;
  return vidx * E + j;
}

// Size of the request table a row map needs (temperatures, or offsets for a
// ragged layout), 0 for greedy rows.
__device__ __forceinline__ int32_t map_table_size(const RowMap& map, int64_t rows) {
  switch (map.kind) {
    case kMapFixed:
      return map.batch;
    case kMapCu:
      return map.batch + 1;
    case kMapPerRow:
      return rows > kTabCap ? kTabCap + 1 : static_cast<int32_t>(rows);
    default:
      return 0;
  }
}

// Index of a row's entry in the request tables (request, or the row itself
// for per-row temperatures), computed by a whole warp (same value in every
// lane).  Ragged layouts search the request offsets 32 at a time, so a lookup
// costs one round trip per factor of 32 in the batch size.
__device__ __forceinline__ int32_t row_entry(const RowMap& map, int32_t row, int lane, const int32_t* cu) {
  switch (map.kind) {
    case kMapFixed:
      return row / map.rows_per_req;
    case kMapPerRow:
      return row;
    case kMapCu: {
      // Invariant: cu[lo] <= row (cu[0] = 0); the answer, the last request
      // starting at or before row, is in [lo, hi].
      int32_t lo = 0, hi = map.batch - 1;
      while (hi > lo) {
        const int32_t step = (hi - lo + 31) / 32;
        const int32_t j = lo + (lane + 1) * step;
        const bool le = j <= hi && cu[j] <= row;
        const int32_t c = __popc(__ballot_sync(0xffffffffu, le));  // offsets are sorted: a prefix of lanes
        hi = min(hi, lo + (c + 1) * step - 1);
        lo += c * step;
      }
      return lo;
    }
    default:
      return -1;  // greedy rows
  }
}

// Temperature of a row read from global memory (whole warp).
__device__ __forceinline__ float row_temperature(const RowMap& map, int32_t row, int lane) {
  const int32_t e = row_entry(map, row, lane, map.cu);
  return e < 0 ? 0.0f : map.temperature[e];
}

// The sum part of warp_combine alone (same rescaling, same butterfly).
__device__ __forceinline__ float warp_sum_scaled(float s, float e) {
  float sc = s != 0.0f ? (e == 0.0f ? s : s * exp2f(e)) : 0.0f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
  return sc;
}

// Merge chunk partial b into a (sums relative to each side's own maximum).
__device__ __forceinline__ void chunk_merge(Part& a, const Part& b, float k) {
  const float M = fmaxf(a.m, b.m);
  if (M == -kInfF) {
    a.flags |= b.flags;
    return;
  }
  const float sa = a.s != 0.0f && a.m != M ? a.s * exp2f((a.m - M) * k) : a.s;
  const float sb = b.s != 0.0f && b.m != M ? b.s * exp2f((b.m - M) * k) : b.s;
  int32_t v = -1;
  if (a.m == M && a.idx >= 0) v = a.idx;
  if (b.m == M && b.idx >= 0 && (v < 0 || b.idx < v)) v = b.idx;
  a = Part{M, sa + sb, v, a.flags | b.flags};
}

// PFX: probe-aware pass (each row's probe token probe[row], for every row but
// the last of each block of probe_rpr rows): the chunk holding the probe also
// sums the terms of the ids below it.
// hand_off_ns: 0 in normal use.  Otherwise (a test of the expiry path) every
// in-CTA hand-off wait (stage full / empty, partial slots) gives up after
// hand_off_ns, and the finalizer first waits on a barrier that nothing
// completes, so at least one wait runs out; the waits that drain bulk copies
// still in flight keep the full limit.
template <int DT, bool PFX>
__global__ void __launch_bounds__(kStatsThreads, 3) k_row_stats(LogitsView lg, RowMap map, Ws ws, ChunkPlan plan,
                                                                const int32_t* probe, int32_t probe_rpr,
                                                                uint64_t hand_off_ns) {
  using VT = VecTraits<DT>;
  constexpr int E = VT::E;
  const int64_t n_items = plan.n_items;
  extern __shared__ unsigned char smem_raw[];
  StatsSmem& sm = *reinterpret_cast<StatsSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int64_t nfull = lg.vocab / E;
  const bool ragged = nfull * E < lg.vocab;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned* queue = ws.done_cnt + 2;
  volatile int* abort = &sm.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&sm.full[s]), 1);
      mbar_init(smem_addr(&sm.empty[s]), kConsumerWarps);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_addr(&sm.pfull[s]), kConsumerWarps);
      mbar_init(smem_addr(&sm.pempty[s]), 1);
    }
    mbar_init(smem_addr(&sm.tab_ready), 1);
    mbar_init(smem_addr(&sm.never), 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  grid_dependency_wait();  // the logits may come from the previous kernel on the stream
  allow_dependents();

  const uint64_t lim = hand_off_ns ? hand_off_ns : kWaitLimitNs;  // hand-off waits
  const int32_t tab_n = map_table_size(map, lg.rows);
  const bool tabbed = tab_n > 0 && tab_n <= kTabCap;
  if (warp == kProducerWarp) {  // ------------------------------------------ producer
    // The whole warp walks the queue; lane 0 drives the ring.  A CTA's first
    // chunk is its own index, later ones gridDim.x + a ticket.  Two tickets are kept in flight in two
    // different registers (a register is busy for the whole warp while any
    // atomic writes it), so each ticket is read two chunks after it was
    // requested.  A stage's
    // copy is issued before the row's temperature is first used: the full
    // barrier completes only after the stage description is written and
    // arrived on.
    uint32_t g = 0;  // stages issued
    unsigned tka = 0, tkb = 0;
    if (lane == 0) {
      tka = atomicAdd(queue, 1u);
      tkb = atomicAdd(queue, 1u);
    }
    int64_t pos = blockIdx.x;
    // k and 1/k of a row: from the staged tables, else computed from a global read.
    auto row_k_of = [&](int32_t row, float& k, float& ik) {
      if (tabbed) {
        const int32_t e = row_entry(map, row, lane, sm.tab_cu);
        k = e < 0 ? 0.0f : sm.tab_k[e];
        ik = e < 0 ? 0.0f : sm.tab_ik[e];
      } else {
        k = temperature_k(row_temperature(map, row, lane));
        ik = k > 0.0f ? __frcp_rn(k) : 0.0f;
      }
    };
    float nk = 0.0f, nik = 0.0f;  // k and 1/k of the next chunk's row
    int32_t nd = -1;              // probe token of the next chunk's row (probe-aware pass)
    auto probe_of = [&](int32_t row) -> int32_t {
      if (!PFX || probe_rpr <= 0 || row % probe_rpr == probe_rpr - 1) return -1;
      return probe[row];
    };
    bool have_k = false, ok = true;
    // Stream the chunk at queue position `pos`, then move to the position whose ticket is in `tk`.
    auto chunk_out = [&](unsigned& tk) {
      const int32_t item = static_cast<int32_t>(pos);
      int32_t row, s0, s1;
      bool last;
      chunk_geometry(plan, item, row, s0, s1, last);
      const int32_t cc0 = s0 * kChunkVecs;
      const int64_t left = nfull - cc0;
      const int32_t span = (s1 - s0) * kChunkVecs;
      const int32_t cn = left <= 0 ? 0 : static_cast<int32_t>(left < span ? left : span);
      const int32_t nst = s1 - s0;
      const int32_t tail = (ragged && last) ? 1 : 0;
      float k = 0.0f, ik = 0.0f;
      int32_t cprobe = -1;  // the probe token when it lies in this chunk
      for (int32_t s = 0; s < nst; ++s, ++g) {
        const int st = g % kStages;
        const int32_t c0 = cc0 + s * kChunkVecs;
        const int32_t rem = cn - s * kChunkVecs;
        const int32_t n = rem <= 0 ? 0 : (rem < kChunkVecs ? rem : kChunkVecs);
        if (lane == 0) {
          ok = mbar_wait_bounded(smem_addr(&sm.empty[st]), ((g / kStages) & 1u) ^ 1u, &sm.abort, lim, kProducerNap);
          if (ok && n > 0) {
            mbar_expect_tx(smem_addr(&sm.full[st]), n * 16);
            bulk_copy_g2s(smem_addr(&sm.buf[st][0]),
                          static_cast<const char*>(lg.base) + (row * lg.ld * VT::ES) + int64_t{c0} * 16, n * 16,
                          smem_addr(&sm.full[st]));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return;
        if (s == 0) {
          if (!have_k) {  // the first chunk: wait for the staged tables
            if (tabbed && lane == 0) {
              volatile int never = 0;
              ok = mbar_wait_bounded(smem_addr(&sm.tab_ready), 0u, &never, kWaitLimitNs);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) return;
            row_k_of(row, nk, nik);
            nd = probe_of(row);
            have_k = true;
          }
          k = nk;  // first use of the prefetched values: after the copy is on its way
          ik = nik;
          asm volatile("mov.b32 %0, %0;" : "+f"(k));
          if (PFX) {
            int32_t d = nd;
            asm volatile("mov.b32 %0, %0;" : "+r"(d));
            if (d >= 0 && d < lg.vocab) {
              const int64_t pv = d / E;  // the ragged tail is vector nfull and rides on the row's last chunk
              const bool here = pv >= nfull ? last : (pv / kChunkVecs >= s0 && pv / kChunkVecs < s1);
              if (here) cprobe = d;
            }
          }
        }
        if (lane == 0) {
          sm.meta[st] = StageMeta{item, row, c0, n, k, ik, nst, tail, cprobe};
          mbar_arrive(smem_addr(&sm.full[st]));
        }
      }
      pos = static_cast<int64_t>(gridDim.x) + __shfl_sync(0xffffffffu, tk, 0);
      if (lane == 0 && pos < n_items) tk = atomicAdd(queue, 1u);
      if (pos < n_items) {
        int32_t nrow, ns0, ns1;
        bool nlast;
        chunk_geometry(plan, static_cast<int32_t>(pos), nrow, ns0, ns1, nlast);
        row_k_of(nrow, nk, nik);
        nd = probe_of(nrow);
      }
    };
    while (pos < n_items) {
      chunk_out(tka);
      if (!ok || pos >= n_items) break;
      chunk_out(tkb);
      if (!ok) break;
    }
    if (lane == 0) {
      bool ended = false;
      if (!ok) {
        sm.abort = 1;
        atomicOr(ws.err, 1u);
      } else if (!*abort) {  // end marker
        const int st = g % kStages;
        if (mbar_wait_bounded(smem_addr(&sm.empty[st]), ((g / kStages) & 1u) ^ 1u, &sm.abort, lim)) {
          sm.meta[st] = StageMeta{-1, 0, 0, 0, 0.0f, 0.0f, 0, 0, -1};
          mbar_arrive(smem_addr(&sm.full[st]));
          ended = true;
        } else {
          sm.abort = 1;
          atomicOr(ws.err, 1u);
        }
      }
      if (*abort) {
        // The consumers may have left with copies still in flight: wait for the
        // last copy on each stage before the CTA exits.  Copies older than the
        // last kStages stages, and the stage the end marker reused, were
        // consumed before the producer could move on.
        const uint32_t first = g >= kStages ? g - kStages + (ended ? 1u : 0u) : 0u;
        for (uint32_t i = first; i < g; ++i) {
          volatile int never = 0;
          if (!mbar_wait_bounded(smem_addr(&sm.full[i % kStages]), (i / kStages) & 1u, &never, kWaitLimitNs))
            atomicOr(ws.err, 1u);
        }
      }
    }
    return;
  }

  if (warp == kFinalizerWarp) {  // ---------------------------------------- finalizer
    if (tabbed) {  // stage the request tables: k = log2(e)/T and its reciprocal, per request
      for (int32_t i0 = 0; i0 < tab_n; i0 += 32 * 8) {
        float tv[8];
        int32_t cv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // all loads first, then all stores: one round trip per 256 entries
          const int32_t i = i0 + u * 32 + lane;
          const bool in = i < tab_n;
          const bool has_t = in && (map.kind != kMapCu || i < map.batch);
          tv[u] = has_t ? map.temperature[i] : 0.0f;
          cv[u] = (in && map.kind == kMapCu) ? map.cu[i] : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int32_t i = i0 + u * 32 + lane;
          if (i < tab_n) {
            const float k = temperature_k(tv[u]);
            sm.tab_k[i] = k;
            sm.tab_ik[i] = k > 0.0f ? __frcp_rn(k) : 0.0f;
            sm.tab_cu[i] = cv[u];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.tab_ready));
    }
    if (hand_off_ns) {  // expiry test: a wait that nothing completes runs out like a stalled hand-off
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(smem_addr(&sm.never), 0u, &sm.abort, hand_off_ns, kConsumerNap);
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) {
          sm.abort = 1;
          atomicOr(ws.err, 1u);
        }
        return;
      }
    }
    // Each chunk's partial goes to the workspace; k_row_merge combines them
    // per row after this grid completes (no cross-CTA waiting here).
    for (uint32_t c = 0;; ++c) {
      const int sl = c % kSlots;
      if (!mbar_wait_bounded(smem_addr(&sm.pfull[sl]), (c / kSlots) & 1u, &sm.abort, lim, kConsumerNap)) {
        sm.abort = 1;
        atomicOr(ws.err, 1u);
        break;
      }
      const int32_t item = sm.slot[sl].item;
      const int32_t row = sm.slot[sl].row;
      const float k = sm.slot[sl].k;
      Part wp = lane < kConsumerWarps ? sm.slot[sl].wpart[lane] : part_identity();
      const float wsb = (PFX && lane < kConsumerWarps) ? sm.slot[sl].wsb[lane] : 0.0f;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.pempty[sl]));  // the slot is free again
      if (item < 0) break;
      const float M = warp_max(wp.m);
      const float sbc = PFX ? warp_sum_scaled(wsb, (wp.m - M) * k) : 0.0f;
      wp = warp_combine(M, wp.m, wp.s, (wp.m - M) * k, wp.idx, wp.flags);
      if (PFX && lane == 0) ws.psb[item] = sbc;
      if (lane == 0) {
        // The chunk's argmax element, from the vector it lies in (just streamed, usually still in L2).
        const int32_t idx = resolve_index<DT>(lg, row, nfull, wp.idx, M);
        ws.partial[item] = RowPartial{wp.s, M, idx, wp.flags};
        ws.rowstat[row].k = k;  // every chunk of the row writes the same value
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  // Hand a chunk's warp partial (or the end mark, item < 0) to the finalizer.
  auto hand_over = [&](uint32_t c, const Part& p, int32_t item, int32_t row, float k, float sbw) -> bool {
    const int sl = c % kSlots;
    if (!mbar_wait_bounded(smem_addr(&sm.pempty[sl]), ((c / kSlots) & 1u) ^ 1u, &sm.abort, lim, kConsumerNap)) {
      sm.abort = 1;
      atomicOr(ws.err, 1u);
      return false;
    }
    if (lane == 0) {
      sm.slot[sl].wpart[warp] = p;
      if (PFX) sm.slot[sl].wsb[warp] = sbw;
      if (warp == 0) {
        sm.slot[sl].item = item;
        sm.slot[sl].row = row;
        sm.slot[sl].k = k;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&sm.pfull[sl]));
    return true;
  };
  uint32_t g = 0;  // stages consumed
  for (uint32_t c = 0;; ++c) {
    int st = g % kStages;
    if (!mbar_wait_bounded(smem_addr(&sm.full[st]), (g / kStages) & 1u, &sm.abort, lim, kConsumerNap)) {
      sm.abort = 1;
      atomicOr(ws.err, 1u);
      break;
    }
    StageMeta md = sm.meta[st];
    if (md.item < 0) {
      hand_over(c, part_identity(), -1, 0, 0.0f, 0.0f);
      break;
    }
    const int32_t item = md.item, row = md.row, nst = md.nst, tail = md.tail;
    const int32_t pd = PFX ? md.probe : -1;
    const float k = md.k, ik = md.ik;
    Part p;
    float sbw = 0.0f;
    bool ok = true;
    if (k > 0.0f) {
      ThreadAcc a = acc_init<true>();  // one partial per chunk: independent of the schedule
      for (int32_t s = 0;; ++s) {
        // In the probe chunk, every term folded before the stage holding the
        // probe's vector lies below the probe: sb starts there as the running
        // sum, and that stage adds its own terms below the probe.
        const int64_t pv = PFX && pd >= 0 ? pd / E : -1;
        if (PFX && pd >= 0 && md.c0 <= pv && pv < md.c0 + md.n) {
          a.sb = a.s.x + a.s.y;
          fold_stage_probe<DT>(a, smem_addr(&sm.buf[st][0]), md.c0, md.n, k, ik, pd);
        } else {
          fold_stage<DT, true>(a, smem_addr(&sm.buf[st][0]), md.c0, md.n, k, ik);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[st]));  // the stage goes back to the producer
        ++g;
        if (s + 1 == nst) break;
        st = g % kStages;
        if (!mbar_wait_bounded(smem_addr(&sm.full[st]), (g / kStages) & 1u, &sm.abort, lim, kConsumerNap)) {
          ok = false;
          break;
        }
        md = sm.meta[st];
      }
      if (PFX && pd >= 0 && pd / E >= nfull) a.sb = a.s.x + a.s.y;  // the probe is in the ragged tail
      if (tail && threadIdx.x == 0) {
        if (PFX && pd >= 0) {
          fold_tail_probe<DT>(a, lg, row, nfull, k, ik, pd);
        } else {
          fold_tail<DT, true>(a, lg, row, nfull, k, ik);
        }
      }
      const float M = warp_max(a.m);
      // 2^(R - M k) rescales the lane's sum to the warp maximum (one rounding).
      const float e = -fmaf(M, k, -a.R);
      if (PFX && pd >= 0) sbw = warp_sum_scaled(a.sb, e);
      p = warp_combine(M, a.m, a.s.x + a.s.y, e, a.vidx, a.flags);
    } else {
      ThreadAcc a = acc_init<false>();
      for (int32_t s = 0;; ++s) {
        fold_stage<DT, false>(a, smem_addr(&sm.buf[st][0]), md.c0, md.n, 0.0f, 0.0f);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[st]));
        ++g;
        if (s + 1 == nst) break;
        st = g % kStages;
        if (!mbar_wait_bounded(smem_addr(&sm.full[st]), (g / kStages) & 1u, &sm.abort, lim, kConsumerNap)) {
          ok = false;
          break;
        }
        md = sm.meta[st];
      }
      if (tail && threadIdx.x == 0) fold_tail<DT, false>(a, lg, row, nfull, 0.0f, 0.0f);
      const float M = warp_max(a.m);
      p = warp_combine(M, a.m, 0.0f, 0.0f, a.vidx, a.flags);
    }
    if (!ok) {
      sm.abort = 1;
      atomicOr(ws.err, 1u);
      break;
    }
    if (!hand_over(c, p, item, row, k, sbw)) break;
  }
}

// Row statistics from the chunk partials, one warp per row: merge the row's
// chunks in chunk order (lane l takes chunks l, l+32, ...; the result does not
// depend on which CTA streamed which chunk; equal maxima keep the lowest
// index), and rewind the chunk queue for the next call.  PFX: also the sum
// below the row's probe token: every chunk wholly below it plus the probe
// chunk's own partial, each rescaled to the row maximum.
template <int DT, bool PFX>
__global__ void __launch_bounds__(256) k_row_merge(LogitsView lg, Ws ws, ChunkPlan plan, const int32_t* probe,
                                                   int32_t probe_rpr) {
  grid_dependency_wait();  // the partials come from k_row_stats
  allow_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) ws.done_cnt[2] = 0u;
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x * int64_t{8} + (threadIdx.x >> 5);
  if (row >= lg.rows) return;  // whole warps leave together
  const float k = __ldcg(&ws.rowstat[row].k);  // written by the streaming pass
  Part acc = part_identity();
  const bool head = row < plan.rows_a;
  const int32_t cnt = head ? plan.cpr_a : plan.cpr_b;
  const int64_t base = head ? row * plan.cpr_a : plan.n_a + (row - plan.rows_a) * plan.cpr_b;
  for (int j = lane; j < cnt; j += 32) chunk_merge(acc, load_partial_cg(&ws.partial[base + j]), k);
  const float M = warp_max(acc.m);
  const Part p = warp_combine(M, acc.m, acc.s, (acc.m - M) * k, acc.idx, acc.flags);
  float below = 0.0f;
  if (PFX && probe_rpr > 0 && row % probe_rpr != probe_rpr - 1 && k > 0.0f && M > -kInfF) {
    const int32_t d = probe[row];
    if (d >= 0 && d < lg.vocab) {
      const int64_t nfull = lg.vocab / VecTraits<DT>::E;
      const int64_t pv = d / VecTraits<DT>::E;
      float part = 0.0f;  // this lane's chunks, in chunk order
      for (int j = lane; j < cnt; j += 32) {
        int32_t r, s0, s1;
        bool last;
        chunk_geometry(plan, static_cast<int32_t>(base + j), r, s0, s1, last);
        const bool holds = pv >= nfull ? last : (pv / kChunkVecs >= s0 && pv / kChunkVecs < s1);
        const bool wholly_below = !holds && static_cast<int64_t>(s1) * kChunkVecs <= pv;
        if (holds || wholly_below) {
          const Part c = load_partial_cg(&ws.partial[base + j]);
          const float v = holds ? __ldcg(&ws.psb[base + j]) : c.s;
          if (v != 0.0f) part += c.m == M ? v : v * exp2f((c.m - M) * k);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      below = part;
    }
  }
  if (lane == 0) {
    RowStat st;
    st.below = below;
    st.pad = 0;
    const bool samp = k > 0.0f && M > -kInfF;
    st.Z = samp ? p.s : 0.0f;
    st.inv_z = samp ? __fdiv_rn(1.0f, p.s) : 0.0f;
    st.M = M;
    st.argmax = p.idx;
    st.flags = p.flags;
    st.k = k;
    ws.rowstat[row] = st;
  }
}

// Copy the row statistics out as plain arrays (and p at a probe token).
__global__ void k_export_stats(LogitsView lg, Ws ws, const int32_t* probe, float* out_max, int32_t* out_argmax,
                               double* out_z, float* out_p, uint32_t* row_flags) {
  grid_dependency_wait();
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

namespace {
std::atomic<uint64_t> g_hand_off_ns{0};  // 0: hand-off waits use the normal limit
}  // namespace

void set_hand_off_limit_ns(uint64_t ns) { g_hand_off_ns.store(ns, std::memory_order_relaxed); }

template <int DT>
cudaError_t stats_occupancy_t(int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(k_row_stats<DT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kStatsSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_row_stats<DT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kStatsSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_row_stats<DT, false>, kStatsThreads,
                                                       kStatsSmemBytes);
}

cudaError_t stats_occupancy(int dtype, int* blocks_per_sm) {
  return dtype == SV_BF16 ? stats_occupancy_t<SV_BF16>(blocks_per_sm) : stats_occupancy_t<SV_F32>(blocks_per_sm);
}

// Stages per row: 1024-vector pieces, at least one (the ragged tail rides on the last).
int32_t stages_per_row(const LogitsView& lg) {
  const int E = lg.dtype == SV_BF16 ? 8 : 4;
  const int64_t nfull = lg.vocab / E;
  const int64_t c = (nfull + kChunkVecs - 1) / kChunkVecs;
  return static_cast<int32_t>(c < 1 ? 1 : c);
}

ChunkPlan chunk_plan(const LogitsView& lg, int grid) {
  ChunkPlan P{};
  P.nst = stages_per_row(lg);
  P.cpr_a = (P.nst + kHeadChunkStages - 1) / kHeadChunkStages;
  P.cpr_b = P.nst;
  const int64_t tail_stages = static_cast<int64_t>(grid) * kTailRounds;
  int64_t rows_b = (tail_stages + P.nst - 1) / P.nst;
  if (rows_b > lg.rows) rows_b = lg.rows;
  P.rows_a = static_cast<int32_t>(lg.rows - rows_b);
  P.n_a = static_cast<int64_t>(P.rows_a) * P.cpr_a;
  P.n_items = P.n_a + rows_b * P.cpr_b;
  return P;
}

// One resident wave, never more CTAs than one-stage chunks (the plan then has at least as many items).
int stats_grid(const DeviceInfo& dev, const LogitsView& lg) {
  const int64_t cap = static_cast<int64_t>(stages_per_row(lg)) * lg.rows;
  int64_t g = static_cast<int64_t>(dev.sms) * dev.stats_blocks_per_sm[lg.dtype == SV_BF16 ? 1 : 0];
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

template <int DT, bool PFX>
cudaError_t launch_row_stats_t(const LogitsView& lg, const RowMap& map, const Ws& ws, int grid, cudaStream_t stream,
                               const ChunkPlan& plan, const int32_t* probe, int32_t probe_rpr,
                               cudaEvent_t stats_done) {
  const dim3 mgrid(static_cast<unsigned>((lg.rows + 7) / 8));
  cudaError_t e = launch_pdl(k_row_stats<DT, PFX>, dim3(grid), dim3(kStatsThreads), kStatsSmemBytes, stream, lg, map,
                             ws, plan, probe, probe_rpr, g_hand_off_ns.load(std::memory_order_relaxed));
  if (e != cudaSuccess) return e;
  if (stats_done && (e = record_event(stats_done, stream)) != cudaSuccess) return e;
  return launch_pdl(k_row_merge<DT, PFX>, mgrid, dim3(256), 0, stream, lg, ws, plan, probe, probe_rpr);
}

cudaError_t launch_row_stats(const LogitsView& lg, const RowMap& map, const Ws& ws, int grid, cudaStream_t stream,
                             const int32_t* probe, int32_t probe_rpr, cudaEvent_t stats_done) {
  const ChunkPlan plan = chunk_plan(lg, grid);
  if (plan.n_items > (int64_t{1} << 30)) return cudaErrorInvalidValue;  // chunk indices and the queue are 32-bit
  if (lg.dtype == SV_BF16) {
    return probe ? launch_row_stats_t<SV_BF16, true>(lg, map, ws, grid, stream, plan, probe, probe_rpr, stats_done)
                 : launch_row_stats_t<SV_BF16, false>(lg, map, ws, grid, stream, plan, nullptr, 0, stats_done);
  }
  return probe ? launch_row_stats_t<SV_F32, true>(lg, map, ws, grid, stream, plan, probe, probe_rpr, stats_done)
               : launch_row_stats_t<SV_F32, false>(lg, map, ws, grid, stream, plan, nullptr, 0, stats_done);
}

cudaError_t launch_export_stats(const LogitsView& lg, const Ws& ws, const int32_t* probe, float* out_max,
                                int32_t* out_argmax, double* out_z, float* out_p, uint32_t* row_flags,
                                cudaStream_t stream) {
  const int threads = 256;
  const int64_t blocks = (lg.rows + threads - 1) / threads;
  return launch_pdl(k_export_stats, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, lg, ws, probe,
                    out_max, out_argmax, out_z, out_p, row_flags);
}

}  // namespace sv
