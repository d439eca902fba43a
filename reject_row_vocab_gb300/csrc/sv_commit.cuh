// Commit bookkeeping ([E2D] §5.6.6 commit_lens = r + 1 and §8.1; [SGO] "两个容易误解的工程细节": the KV of
// the committed rows moves to the positions after the committed prefix): the exclusive scan of num_out and the
// per-entry KV slot and destination position, by one group of threads.  Used by the commit kernel, by the
// sampler's first block and by the acceptance-and-commit kernel of small greedy batches.
//
//   [E2D] "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理"
//   [SGO] SGLang speculative-decoding overview (zdszero.github.io)
#pragma once

#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kCommitThreads = 256;

// Barrier over the first BS threads: the named barrier when a producer warp
// beyond them must not take part, else the whole block.
template <int BS, bool NAMED>
__device__ __forceinline__ void group_sync() {
  if (NAMED) {
    named_sync(BS);
  } else {
    __syncthreads();
  }
}

// Exclusive scan over the first BS threads (lane order, then warp order).  smem: NW + 1.
template <typename Tv, int BS, bool NAMED = false>
__device__ __forceinline__ Tv block_exclusive_scan(Tv v, Tv* smem, Tv* total) {
  constexpr int NW = BS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Tv incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const Tv t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) smem[warp] = incl;
  group_sync<BS, NAMED>();
  if (warp == 0) {
    const Tv w = lane < NW ? smem[lane] : Tv(0);
    Tv wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const Tv t = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += t;
    }
    if (lane < NW) smem[lane] = wi - w;
    if (lane == NW - 1) smem[NW] = wi;
  }
  group_sync<BS, NAMED>();
  const Tv res = smem[warp] + (incl - v);
  *total = smem[NW];
  group_sync<BS, NAMED>();
  return res;
}

// Commit bookkeeping for the whole batch by the first kCommitThreads threads
// of a block: commit_cu = exclusive
// scan of num_out; for committed row k of request b, its KV slot and its
// destination position seq_lens[b] + k.  Needs only the acceptance results.
// s_slots / s_seq: copies of row_slots / seq_lens staged in shared memory by
// the caller, or NULL to read them from global memory.
template <bool NAMED>
__device__ __forceinline__ void commit_block_t(const OutView& out, const CommitParams& cp,
                                               const int64_t* s_slots = nullptr, const int64_t* s_seq = nullptr) {
  __shared__ int64_t s_scan[kCommitThreads / 32 + 1];
  const int B = cp.batch, ML = cp.max_len;
  const int per = (B + kCommitThreads - 1) / kCommitThreads;
  const int ba = min(B, static_cast<int>(threadIdx.x) * per), bb = min(B, ba + per);
  int64_t local = 0;
  for (int b = ba; b < bb; ++b) local += out.num_out[b];
  int64_t total;
  int64_t run = block_exclusive_scan<int64_t, kCommitThreads, NAMED>(local, s_scan, &total);
  for (int b = ba; b < bb; ++b) {
    out.commit_cu[b] = static_cast<int32_t>(run);
    run += out.num_out[b];
  }
  if (threadIdx.x == kCommitThreads - 1) {
    out.commit_cu[B] = static_cast<int32_t>(total);
    if (cp.err) *cp.err = 0u;
  }
  group_sync<kCommitThreads, NAMED>();  // commit_cu visible to the whole group
  if (!out.commit_src_slot && !out.commit_dst_pos) return;
  // one (request, k) entry per thread and step; all loads of a step are independent
  for (int64_t e = threadIdx.x; e < static_cast<int64_t>(B) * ML; e += kCommitThreads) {
    const int b = static_cast<int>(e / ML), k = static_cast<int>(e % ML);
    const int n = out.num_out[b];
    const int32_t row = out.accept_rows[e];
    const int64_t base = out.commit_cu[b];
    if (k >= n) continue;
    if (out.commit_src_slot && cp.row_slots) out.commit_src_slot[base + k] = s_slots ? s_slots[row] : cp.row_slots[row];
    if (out.commit_dst_pos && cp.seq_lens) out.commit_dst_pos[base + k] = (s_seq ? s_seq[b] : cp.seq_lens[b]) + k;
  }
}

__device__ __forceinline__ void commit_block(const OutView& out, const CommitParams& cp) { commit_block_t<false>(out, cp); }
__device__ __forceinline__ void commit_block_named(const OutView& out, const CommitParams& cp,
                                                   const int64_t* s_slots = nullptr, const int64_t* s_seq = nullptr) {
  commit_block_t<true>(out, cp, s_slots, s_seq);
}
}  // namespace sv
