// Final token and commit.
//
// The correction / bonus token is an inverse-CDF draw over unnormalised
// weights w_v of one row ([E2D] §1.2 residual p' = [p - q]_+ / sum [p - q]_+;
// bonus from p, §1.1; inverse CDF as in §6.2 sample_path()):
//   w_v = max(0, p_v - q_v)          after a rejection,
//   w_v = p_v                        bonus after every draft passed,
//   w_v = p_v, children zeroed       target-only tree stop ([SGO]).
// Pass A splits each sampled row into tiles of 256 entries (one warp, eight
// entries per lane) spread over many CTAs and stores every tile's weight sum.
// Pass B (one CTA per request) scans the tile sums, picks the tile holding
// t = u_final * S, and one warp re-forms that tile's weights with exactly the
// same arithmetic to find the entry.  The last CTA to finish then performs
// the commit: exclusive scan of commit_lens and the KV slot / position lists
// ([E2D] §5.6.6, §8.1; [SGO] "两个容易误解的工程细节").
//
//   [E2D] "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理"
//   [SGO] SGLang speculative-decoding overview (zdszero.github.io)
#include <climits>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kCommitThreads = 256;

__device__ __forceinline__ bool sampling_mode(int32_t mode) {
  return mode == kModeResidual || mode == kModeP || mode == kModePExcl;
}

// The eight weights of one lane of a tile: entries [col0, col0 + 8) of `row`.
// Entries past the vocabulary weigh 0.  Both passes call this with the same
// arguments, so a tile's weights are bit-identical in both.
__device__ __forceinline__ void lane_weights(const LogitsView& lg, const float* q, int64_t ldq, int64_t row,
                                             const RowStat& rs, float inv_z, int32_t mode, const int32_t* excl,
                                             int32_t n_excl, int64_t col0, float (&w)[8]) {
  const int V = lg.vocab;
  float x[8];
  if (col0 + 8 <= V) {
    if (lg.dtype == SV_BF16) {
      const uint4 r = ld_stream16(static_cast<const char*>(lg.base) + (row * lg.ld + col0) * 2);
      x[0] = bf16_lo(r.x);
      x[1] = bf16_hi(r.x);
      x[2] = bf16_lo(r.y);
      x[3] = bf16_hi(r.y);
      x[4] = bf16_lo(r.z);
      x[5] = bf16_hi(r.z);
      x[6] = bf16_lo(r.w);
      x[7] = bf16_hi(r.w);
    } else {
      const char* base = static_cast<const char*>(lg.base) + (row * lg.ld + col0) * 4;
      const uint4 r0 = ld_stream16(base), r1 = ld_stream16(base + 16);
      x[0] = __uint_as_float(r0.x);
      x[1] = __uint_as_float(r0.y);
      x[2] = __uint_as_float(r0.z);
      x[3] = __uint_as_float(r0.w);
      x[4] = __uint_as_float(r1.x);
      x[5] = __uint_as_float(r1.y);
      x[6] = __uint_as_float(r1.z);
      x[7] = __uint_as_float(r1.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (col0 + i < V) ? load_logit(lg, row, col0 + i) : -kInfF;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float e = usable_logit(x[i]) ? ex2_fast(__fmul_rn(__fsub_rn(x[i], rs.M), rs.k)) : 0.0f;
    w[i] = __fmul_rn(e, inv_z);
  }
  if (mode == kModeResidual) {
    float qv[8];
    if (col0 + 8 <= V) {
      const char* qb = reinterpret_cast<const char*>(q + row * ldq + col0);
      const uint4 r0 = ld_stream16(qb), r1 = ld_stream16(qb + 16);
      qv[0] = __uint_as_float(r0.x);
      qv[1] = __uint_as_float(r0.y);
      qv[2] = __uint_as_float(r0.z);
      qv[3] = __uint_as_float(r0.w);
      qv[4] = __uint_as_float(r1.x);
      qv[5] = __uint_as_float(r1.y);
      qv[6] = __uint_as_float(r1.z);
      qv[7] = __uint_as_float(r1.w);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] = (col0 + i < V) ? __ldg(q + row * ldq + col0 + i) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = fmaxf(__fsub_rn(w[i], qv[i]), 0.0f);
  } else if (mode == kModePExcl) {
    for (int e = 0; e < n_excl; ++e) {
      const int64_t d = static_cast<int64_t>(excl[e]) - col0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (d == i) w[i] = 0.0f;
    }
  }
}

__device__ __forceinline__ double lane_sum(const float (&w)[8]) {
  double s = 0.0;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += static_cast<double>(w[i]);
  return s;
}

__device__ __forceinline__ float inverse_z(const RowStat& rs) { return static_cast<float>(1.0 / rs.Z); }

// Block-wide exclusive scan (lane order, then warp order).  smem: NW + 1.
template <typename Tv, int BS>
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
  __syncthreads();
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
  __syncthreads();
  const Tv res = smem[warp] + (incl - v);
  *total = smem[NW];
  __syncthreads();
  return res;
}

// Commit bookkeeping for the whole batch by one CTA: commit_cu = exclusive
// scan of num_out; for committed row k of request b, its KV slot and its
// destination position seq_lens[b] + k.
__device__ void commit_block(const OutView& out, const CommitParams& cp) {
  __shared__ int64_t s_scan[kCommitThreads / 32 + 1];
  const int B = cp.batch, ML = cp.max_len;
  const int per = (B + kCommitThreads - 1) / kCommitThreads;
  const int ba = min(B, static_cast<int>(threadIdx.x) * per), bb = min(B, ba + per);
  int64_t local = 0;
  for (int b = ba; b < bb; ++b) local += out.num_out[b];
  int64_t total;
  int64_t run = block_exclusive_scan<int64_t, kCommitThreads>(local, s_scan, &total);
  for (int b = ba; b < bb; ++b) {
    out.commit_cu[b] = static_cast<int32_t>(run);
    const int n = out.num_out[b];
    for (int k = 0; k < n; ++k) {
      const int64_t idx = run + k;
      if (out.commit_src_slot && cp.row_slots) {
        const int32_t row = out.accept_rows[static_cast<int64_t>(b) * ML + k];
        out.commit_src_slot[idx] = cp.row_slots[row];
      }
      if (out.commit_dst_pos && cp.seq_lens) out.commit_dst_pos[idx] = cp.seq_lens[b] + k;
    }
    run += n;
  }
  if (threadIdx.x == kCommitThreads - 1) out.commit_cu[B] = static_cast<int32_t>(total);
}

// Pass A: weight sums of every tile of the sampled rows.  grid = (chunks, batch).
__global__ void __launch_bounds__(kSampleThreads) k_sample_tiles(LogitsView lg, const float* q, int64_t ldq, Ws ws,
                                                                 int32_t excl_stride) {
  const int b = blockIdx.y;
  const ReqState rq = ws.state[b];
  if (!sampling_mode(rq.mode)) return;
  const int64_t row = rq.sample_row;
  const RowStat rs = ws.rowstat[row];
  const float inv_z = inverse_z(rs);
  const int32_t* excl = ws.excl + static_cast<int64_t>(b) * excl_stride;
  const int T = ws.ntiles;
  const int nchunk = gridDim.x;
  const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * T / nchunk);
  const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * T / nchunk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int tile = t0 + warp; tile < t1; tile += kSampleWarps) {
    float w[8];
    lane_weights(lg, q, ldq, row, rs, inv_z, rq.mode, excl, rq.n_excl, static_cast<int64_t>(tile) * kTile + lane * 8,
                 w);
    const double s = warp_sum_xor(lane_sum(w));
    if (lane == 0) ws.tsum[static_cast<int64_t>(b) * T + tile] = s;
  }
}

// Pass B + commit.  grid = batch.
__global__ void __launch_bounds__(kSampleThreads) k_sample_finish(LogitsView lg, const float* q, int64_t ldq,
                                                                  const float* u_final, OutView out,
                                                                  CommitParams cp, Ws ws, int32_t excl_stride) {
  __shared__ double s_scan[kSampleWarps + 1];
  __shared__ int s_tile;
  __shared__ int s_last_nz;
  __shared__ double s_pre;
  __shared__ int s_last;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const ReqState rq = ws.state[b];
  if (sampling_mode(rq.mode)) {
    const int64_t row = rq.sample_row;
    const RowStat rs = ws.rowstat[row];
    const float inv_z = inverse_z(rs);
    const int32_t* excl = ws.excl + static_cast<int64_t>(b) * excl_stride;
    const int T = ws.ntiles;
    double* ts = ws.tsum + static_cast<int64_t>(b) * T;
    int32_t mode = rq.mode;
    uint32_t st_add = 0u;
    const int per = (T + kSampleThreads - 1) / kSampleThreads;
    const int ta = min(T, tid * per), tb = min(T, ta + per);

    double loc = 0.0;
    for (int j = ta; j < tb; ++j) loc += ts[j];
    double total;
    double pre = block_exclusive_scan<double, kSampleThreads>(loc, s_scan, &total);
    if (!(total > 0.0)) {  // residual (or what is left of p) is empty: draw from p instead
      mode = kModeP;
      st_add = kStResidualEmpty;
      for (int tile = warp; tile < T; tile += kSampleWarps) {
        float w[8];
        lane_weights(lg, q, ldq, row, rs, inv_z, mode, excl, 0, static_cast<int64_t>(tile) * kTile + lane * 8, w);
        const double s = warp_sum_xor(lane_sum(w));
        if (lane == 0) ts[tile] = s;
      }
      __syncthreads();
      loc = 0.0;
      for (int j = ta; j < tb; ++j) loc += ts[j];
      pre = block_exclusive_scan<double, kSampleThreads>(loc, s_scan, &total);
    }
    const double t = static_cast<double>(u_final[b]) * total;
    if (tid == 0) {
      s_tile = INT_MAX;
      s_last_nz = -1;
    }
    __syncthreads();
    int my_tile = INT_MAX, my_nz = -1;
    double my_pre = 0.0, run = pre;
    for (int j = ta; j < tb; ++j) {
      const double wj = ts[j];
      if (wj > 0.0) {
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
    __syncthreads();
    if (my_tile != INT_MAX && my_tile == s_tile) s_pre = my_pre;
    __syncthreads();

    if (warp == 0 && (s_tile != INT_MAX || s_last_nz >= 0)) {
      const bool located = s_tile != INT_MAX;
      const int tile = located ? s_tile : s_last_nz;
      const double tpre = located ? s_pre : 0.0;
      const int64_t col0 = static_cast<int64_t>(tile) * kTile + lane * 8;
      float w[8];
      lane_weights(lg, q, ldq, row, rs, inv_z, mode, excl, mode == kModePExcl ? rq.n_excl : 0, col0, w);
      const double ls = lane_sum(w);
      const double incl = warp_inclusive_scan(ls);
      const double lo = tpre + (incl - ls), hi = tpre + incl;
      int v = -1;
      const unsigned hit = __ballot_sync(0xffffffffu, located && ls > 0.0 && lo <= t && t < hi);
      if (hit) {
        const int f = __ffs(hit) - 1;
        int cand = -1;
        if (lane == f) {
          double cum = lo;
          for (int i = 0; i < 8; ++i) {
            cum += static_cast<double>(w[i]);
            if (cand < 0 && cum > t) cand = i;
          }
          if (cand < 0)
            for (int i = 7; i >= 0; --i)
              if (cand < 0 && w[i] > 0.0f) cand = i;
        }
        cand = __shfl_sync(0xffffffffu, cand, f);
        v = static_cast<int>(static_cast<int64_t>(tile) * kTile + f * 8 + cand);
      } else {  // rounding left t outside every lane: last positive entry of the tile
        const unsigned nz = __ballot_sync(0xffffffffu, ls > 0.0);
        const int f = nz ? 31 - __clz(nz) : 0;
        int cand = -1;
        if (lane == f)
          for (int i = 7; i >= 0; --i)
            if (cand < 0 && w[i] > 0.0f) cand = i;
        cand = __shfl_sync(0xffffffffu, cand, f);
        v = cand < 0 ? -1 : static_cast<int>(static_cast<int64_t>(tile) * kTile + f * 8 + cand);
      }
      if (lane == 0) {
        out.bonus[b] = v;
        out.out_tokens[static_cast<int64_t>(b) * cp.max_len + rq.r] = v;
        if (st_add) out.dev_status[b] = rq.status | st_add;
      }
    } else if (warp == 0 && lane == 0) {  // no positive weight at all (not reachable for a usable row)
      out.bonus[b] = -1;
      out.dev_status[b] = rq.status | st_add | kStNonFinite;
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned ticket = atomicAdd(ws.done_cnt, 1u);
    s_last = (ticket == gridDim.x - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    commit_block(out, cp);
    if (tid == 0) *ws.done_cnt = 0u;
  }
}

__global__ void __launch_bounds__(kCommitThreads) k_commit(OutView out, CommitParams cp) { commit_block(out, cp); }

}  // namespace

cudaError_t launch_sample_and_commit(const LogitsView& lg, const float* q, int64_t ldq, const float* u_final,
                                     const OutView& out, const CommitParams& cp, const Ws& ws,
                                     const DeviceInfo& dev, cudaStream_t stream) {
  const int T = ws.ntiles;
  int nchunk = (4 * dev.sms + cp.batch - 1) / cp.batch;
  if (nchunk > T) nchunk = T;
  if (nchunk < 1) nchunk = 1;
  k_sample_tiles<<<dim3(nchunk, cp.batch), kSampleThreads, 0, stream>>>(lg, q, ldq, ws, cp.max_len);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_sample_finish<<<cp.batch, kSampleThreads, 0, stream>>>(lg, q, ldq, u_final, out, cp, ws, cp.max_len);
  return cudaGetLastError();
}

cudaError_t launch_commit(const OutView& out, const CommitParams& cp, cudaStream_t stream) {
  k_commit<<<1, kCommitThreads, 0, stream>>>(out, cp);
  return cudaGetLastError();
}

}  // namespace sv
