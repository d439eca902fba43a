// Acceptance: one warp per request decides how many drafts are accepted.
//
// Chains and ragged blocks ([E2D] §1.1, §1.2, §5.6.5): every lane takes one
// verify row, evaluates its test (greedy: argmax == draft; sampling:
// u * q(d) < p(d) with p = 2^((l_d - M) k) / Z, [E2D] §1.2 equation for
// alpha), and a warp ballot finds the first failure.  Trees ([SGO]
// "为什么结果不受 draft 影响": verify_tree_greedy and
// tree_speculative_sampling_target_only): the walk goes from the root, the
// children of the current node are found with a ballot over the parent
// array, and the accepted child is the first (ballot) match.
//
//   [E2D] "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理"
//   [SGO] SGLang speculative-decoding overview (zdszero.github.io)
//
// Each request leaves in the workspace what the final-token step must do
// (nothing, residual draw, bonus draw, or bonus draw with excluded tokens),
// and writes its accepted prefix straight into the outputs.
#include <cstdint>

#include "sv_commit.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kChainWarps = 4;

__device__ __forceinline__ uint32_t warp_or(uint32_t v) { return __reduce_or_sync(kFull, v); }

// p_row(token) from the row statistics; 0 for an excluded (NaN / +inf) entry.
__device__ __forceinline__ float target_prob(float l, const RowStat& rs) {
  if (!usable_logit(l)) return 0.0f;
  return __fdiv_rn(exp2f((l - rs.M) * rs.k), rs.Z);
}

// q(d) of a sparse row: the sum of the candidate probabilities whose id is d
// (in candidate order); *bad is set when an id other than the padding -1
// falls outside [0, V).
__device__ __forceinline__ float sparse_q_at(const ChainParams& p, int64_t row, int32_t d, bool* bad) {
  const int32_t* ids = p.cand_ids + row * p.ldc;
  const float* pr = p.cand_probs + row * p.ldc;
  constexpr int U = 8;  // loads issued together, one round trip per U candidates
  float q = 0.0f;
  for (int c0 = 0; c0 < p.num_cands; c0 += U) {
    int32_t id[U];
    float pv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      id[u] = c0 + u < p.num_cands ? ids[c0 + u] : -1;
      pv[u] = c0 + u < p.num_cands ? pr[c0 + u] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (id[u] == d) q = __fadd_rn(q, pv[u]);
      if (id[u] != -1 && (id[u] < 0 || id[u] >= p.lg.vocab)) *bad = true;
    }
  }
  return q;
}

// One chain request (b < p.batch) by one warp.  The inputs (ids, logits, q,
// uniforms) were complete before the statistics pass started, and the calling
// grid starts only after that pass: the gathers below are issued before
// waiting for the row statistics, overlapping that wait.
__device__ __forceinline__ void accept_chain_request(const ChainParams& p, const OutView& out, const Ws& ws, int b) {
  const int lane = threadIdx.x & 31;
  const int ML = p.max_len;
  int32_t* otok = out.out_tokens + static_cast<int64_t>(b) * ML;
  int32_t* orow = out.accept_rows + static_cast<int64_t>(b) * ML;

  int64_t start, end;
  if (p.fixed_len > 0) {
    start = static_cast<int64_t>(b) * p.fixed_len;
    end = start + p.fixed_len;
  } else {
    start = p.cu[b];
    end = p.cu[b + 1];
  }
  const int64_t L = end - start;
  const bool bad_layout = start < 0 || end > p.lg.rows || L < 1 || L > ML;
  const float T = p.temperature ? p.temperature[b] : 0.0f;
  const bool greedy = !sampling_temperature(T);
  // Gathers of the first 32 rows' tests (id, and for sampling l[d], q[d], u).
  const bool sparse = p.cand_ids != nullptr;
  int32_t pre_d = -1;
  float pre_l = 0.0f, pre_q = 0.0f, pre_u = 0.0f;
  bool cand_bad = false;  // a tested row lists a candidate id outside [0, V)
  for (int64_t j = lane; !bad_layout && j < L - 1; j += 32) {
    const int64_t row = start + j;
    const int32_t d = p.ids[row + 1];
    if (sparse) {  // every tested row's list is checked, visited or not
      const float qd = sparse_q_at(p, row, d, &cand_bad);
      if (j == lane) pre_q = qd;
    }
    if (j == lane) {
      pre_d = d;
      if (!greedy && d >= 0 && d < p.lg.vocab) {
        pre_l = load_logit(p.lg, row, d);
        if (!sparse && !p.match) pre_q = p.q[row * p.ldq + d];
        pre_u = p.u_accept[row];
      }
    }
  }
  grid_dependency_wait();  // row statistics from the previous kernel
  allow_dependents();
  if (bad_layout) {  // invalid layout: commit nothing
    for (int k = lane; k < ML; k += 32) {
      otok[k] = -1;
      orow[k] = -1;
    }
    if (lane == 0) {
      out.accept_len[b] = 0;
      out.num_out[b] = 0;
      out.bonus[b] = -1;
      out.dev_status[b] = kStBadLayout;
      ws.state[b] = ReqState{0, -1, kModeNoCommit, -1, kStBadLayout, 0, 0, 0};
    }
    return;
  }

  uint32_t st = (__ldcg(ws.err) ? kStTimeout : 0u) | (warp_or(cand_bad ? 1u : 0u) ? kStTokenRange : 0u);
  int64_t s = L - 1;  // row (within the request) that yields the final token
  int how = 0;        // 0 all accepted, 1 rejected, 2 unusable row
  RowStat fs{};
  // Each lane takes one row (the last row too, for its statistics): the
  // statistics and the tested id load together, then the two gathers.
  for (int64_t j0 = 0; j0 < L; j0 += 32) {
    const int64_t j = j0 + lane;
    const bool has_row = j < L;
    const bool tested = j < L - 1;
    const int64_t row = start + j;
    RowStat rs{};
    int32_t d = -1;
    if (has_row) rs = ws.rowstat[row];
    if (tested) d = j0 == 0 ? pre_d : p.ids[row + 1];
    int stop = 0;
    uint32_t fl = rs.flags;
    if (tested) {
      if (rs.argmax < 0) {
        stop = 2;
        fl |= kStNonFinite;
      } else if (d < 0 || d >= p.lg.vocab) {
        stop = 1;
        fl |= kStTokenRange;
      } else if (greedy) {
        stop = (rs.argmax != d) ? 1 : 0;
      } else {
        bool unused = false;
        const float l = j0 == 0 ? pre_l : load_logit(p.lg, row, d);
        const float u = j0 == 0 ? pre_u : p.u_accept[row];
        if (p.match) {
          // The target's own inverse-CDF draw with u equals d iff u * Z falls in
          // [sum below d, sum below d + term of d) (all in Z's units).
          const float uz = __fmul_rn(u, rs.Z);
          const float ed = usable_logit(l) ? exp2f((l - rs.M) * rs.k) : 0.0f;
          stop = (uz >= rs.below && uz < __fadd_rn(rs.below, ed)) ? 0 : 1;
        } else {
          const float qd =
              j0 == 0 ? pre_q : (sparse ? sparse_q_at(p, row, d, &unused) : p.q[row * p.ldq + d]);
          stop = (__fmul_rn(u, qd) < target_prob(l, rs)) ? 0 : 1;
        }
      }
    }
    const unsigned bal = __ballot_sync(kFull, tested && stop != 0);
    const int first = bal ? __ffs(bal) - 1 : 32;
    st |= warp_or((tested && lane <= first) ? fl : 0u);  // rows past the stop are not visited
    int src = -1;
    if (bal) {
      s = j0 + first;
      how = __shfl_sync(kFull, stop, first);
      src = first;
    } else if (L - 1 - j0 < 32) {
      src = static_cast<int>(L - 1 - j0);  // every draft passed: the last row gives the bonus
    }
    if (src >= 0) {
      fs.Z = __shfl_sync(kFull, rs.Z, src);
      fs.M = __shfl_sync(kFull, rs.M, src);
      fs.argmax = __shfl_sync(kFull, rs.argmax, src);
      fs.flags = __shfl_sync(kFull, rs.flags, src);
      fs.k = __shfl_sync(kFull, rs.k, src);
      break;
    }
  }

  const int64_t fr = start + s;
  st |= fs.flags;
  int32_t bonus = -1;
  int32_t mode = kModeDone;
  if (how == 2 || fs.argmax < 0) {
    st |= kStNonFinite;
  } else if (greedy) {
    bonus = fs.argmax;
  } else {
    // sample-then-match: the final row is drawn from its own p with its own uniform
    mode = (how == 1 && !p.match) ? (sparse ? kModeResidualSparse : kModeResidual) : kModeP;
  }
  // a sparse residual draw reads row fr's candidate list in place, all num_cands entries
  const int32_t n_list = mode == kModeResidualSparse ? p.num_cands : 0;
  for (int64_t k = lane; k < ML; k += 32) {
    int32_t t = -1, r = -1;
    if (k < s) {
      t = p.ids[start + 1 + k];
      r = static_cast<int32_t>(start + k);
    } else if (k == s) {
      t = bonus;
      r = static_cast<int32_t>(start + k);
    }
    otok[k] = t;
    orow[k] = r;
  }
  if (lane == 0) {
    out.accept_len[b] = static_cast<int32_t>(s);
    out.num_out[b] = static_cast<int32_t>(s + 1);
    out.bonus[b] = bonus;
    out.dev_status[b] = st;
    ws.state[b] = ReqState{static_cast<int32_t>(s), static_cast<int32_t>(fr), mode, bonus, st, n_list, 0, 0};
    if (p.match) ws.ureq[b] = p.u_accept[fr];
  }
}

// One tree request (b < p.batch) by one warp, its node data staged in the
// shared-memory arrays given (p.nodes entries each).  Node data and the tree's
// validation come from inputs that were complete before the statistics pass
// started (the calling grid starts after that pass), so they are staged before
// waiting for the row statistics.
// Sampling walks also stage, for every node, its token's logit under its
// parent's row and the node's uniform (s_lg, s_u; NULL for greedy-only calls),
// so a visited level waits only for its row statistics.
__device__ __forceinline__ void accept_tree_request(const TreeParams& p, const OutView& out, const Ws& ws, int b,
                                                    int32_t* s_tok, int32_t* s_par, int32_t* s_kid, float* s_pk,
                                                    float* s_lg, float* s_u) {
  const int lane = threadIdx.x & 31;
  const int N = p.nodes;
  const int V = p.lg.vocab;
  const int64_t row0 = static_cast<int64_t>(b) * N;
  int32_t* otok = out.out_tokens + row0;
  int32_t* orow = out.accept_rows + row0;
  const bool lists = p.first_child != nullptr;
  const int32_t* fc = lists ? p.first_child + row0 : nullptr;
  const int32_t* ns = lists ? p.next_sibling + row0 : nullptr;

  for (int i = lane; i < N; i += 32) {
    s_tok[i] = p.tokens[row0 + i];
    s_par[i] = p.parents[row0 + i];
  }
  __syncwarp();

  // Validation: parents point strictly backwards, sibling lists (when given)
  // only list children of their node and end within N steps.
  bool bad = false;
  for (int i = lane; i < N; i += 32) {
    const int32_t pi = s_par[i];
    if (i == 0 ? pi != -1 : (pi < 0 || pi >= i)) bad = true;
  }
  if (lists) {
    for (int i = lane; i < N; i += 32) {
      int32_t c = fc[i];
      for (int steps = 0; c != -1 && !bad; ++steps) {
        if (steps >= N || c < 1 || c >= N || s_par[c] != i) {
          bad = true;
        } else {
          c = ns[c];
        }
      }
    }
  }
  bad = __any_sync(kFull, bad);

  const float T = p.temperature ? p.temperature[b] : 0.0f;
  const bool greedy = !sampling_temperature(T);
  if (!greedy && s_lg) {
    for (int i = lane; i < N; i += 32) {
      const int32_t pi = s_par[i], t = s_tok[i];
      s_lg[i] = (!bad && i > 0 && t >= 0 && t < V) ? load_logit(p.lg, row0 + pi, t) : 0.0f;
      s_u[i] = p.u_accept[row0 + i];
    }
    __syncwarp();
  }
  grid_dependency_wait();  // row statistics from the previous kernel
  allow_dependents();
  uint32_t st = (bad ? kStBadTree : 0u) | (__ldcg(ws.err) ? kStTimeout : 0u);
  int cur = 0, depth = 0;
  int32_t bonus = -1;
  int32_t mode = kModeDone;
  int32_t n_excl = 0;
  int64_t sample_row = -1;
  if (lane == 0) orow[0] = static_cast<int32_t>(row0);

  for (;;) {
    const int64_t row = row0 + cur;
    const RowStat rs = ws.rowstat[row];
    st |= rs.flags;
    if (rs.argmax < 0) {
      st |= kStNonFinite;
      break;
    }
    // Children of cur, in verification order, into s_kid[0, nk).
    int nk = 0;
    if (!bad) {
      if (!lists) {
        for (int i0 = cur + 1; i0 < N; i0 += 32) {
          const int i = i0 + lane;
          const bool is_child = i < N && s_par[i] == cur;
          const unsigned bal = __ballot_sync(kFull, is_child);
          if (is_child) s_kid[nk + __popc(bal & ((1u << lane) - 1u))] = i;
          nk += __popc(bal);
        }
      } else {
        if (lane == 0) {
          for (int32_t c = fc[cur]; c != -1; c = ns[c]) s_kid[nk++] = c;
        }
        nk = __shfl_sync(kFull, nk, 0);
      }
    }
    __syncwarp();

    int next = -1;
    if (greedy) {
      for (int k0 = 0; k0 < nk; k0 += 32) {
        const int kk = k0 + lane;
        const bool valid = kk < nk;
        const int32_t t = valid ? s_tok[s_kid[kk]] : -1;
        const bool oor = valid && (t < 0 || t >= V);
        const bool match = valid && !oor && t == rs.argmax;
        const unsigned bal = __ballot_sync(kFull, match);
        const int first = bal ? __ffs(bal) - 1 : 32;
        if (__any_sync(kFull, oor && lane <= first)) st |= kStTokenRange;
        if (bal) {
          next = s_kid[k0 + first];
          break;
        }
      }
      if (next < 0) {
        bonus = rs.argmax;
        break;
      }
    } else {
      for (int kk = lane; kk < nk; kk += 32) {
        const int32_t t = s_tok[s_kid[kk]];
        s_pk[kk] = (t >= 0 && t < V) ? target_prob(s_lg ? s_lg[s_kid[kk]] : load_logit(p.lg, row, t), rs) : 0.0f;
      }
      __syncwarp();
      if (lane == 0) {
        const float u = s_u ? s_u[cur] : p.u_accept[row];
        float c = 0.0f;
        int32_t* excl = ws.excl + static_cast<int64_t>(b) * N;
        for (int kk = 0; kk < nk; ++kk) {
          const int32_t t = s_tok[s_kid[kk]];
          if (t < 0 || t >= V) {
            st |= kStTokenRange;
            continue;
          }
          bool dup = false;
          for (int e = 0; e < n_excl; ++e) dup |= (excl[e] == t);
          if (dup) {
            st |= kStDupSibling;
            continue;
          }
          excl[n_excl++] = t;
          const float pk = s_pk[kk];
          c = __fadd_rn(c, pk);
          if (u < __fdiv_rn(c, p.th_acc) || pk >= p.th_single) {
            next = s_kid[kk];
            break;
          }
        }
      }
      next = __shfl_sync(kFull, next, 0);
      n_excl = __shfl_sync(kFull, n_excl, 0);
      st = __shfl_sync(kFull, st, 0);
      if (next < 0) {
        mode = kModePExcl;
        sample_row = row;
        break;
      }
      n_excl = 0;
    }
    ++depth;
    if (lane == 0) {
      orow[depth] = static_cast<int32_t>(row0 + next);
      otok[depth - 1] = s_tok[next];
    }
    cur = next;
  }
  __syncwarp();
  for (int k = depth + lane; k < N; k += 32) {
    otok[k] = (k == depth) ? bonus : -1;
    if (k > depth) orow[k] = -1;
  }
  if (lane == 0) {
    out.accept_len[b] = depth;
    out.num_out[b] = depth + 1;
    out.bonus[b] = bonus;
    out.dev_status[b] = st;
    ws.state[b] = ReqState{depth, static_cast<int32_t>(sample_row), mode, bonus, st, n_excl, 0, 0};
  }
}

__global__ void __launch_bounds__(32 * kChainWarps) k_accept_chain(ChainParams p, OutView out, Ws ws) {
  const int b = blockIdx.x * kChainWarps + (threadIdx.x >> 5);
  if (b >= p.batch) {
    grid_dependency_wait();
    allow_dependents();
    return;
  }
  accept_chain_request(p, out, ws, b);
}

// One warp per request.  Node data is staged in shared memory.
__global__ void __launch_bounds__(32) k_accept_tree(TreeParams p, OutView out, Ws ws) {
  __shared__ int32_t s_tok[kMaxNodes];
  __shared__ int32_t s_par[kMaxNodes];
  __shared__ int32_t s_kid[kMaxNodes];
  __shared__ float s_pk[kMaxNodes];
  __shared__ float s_lg[kMaxNodes];
  __shared__ float s_u[kMaxNodes];
  accept_tree_request(p, out, ws, blockIdx.x, s_tok, s_par, s_kid, s_pk, s_lg, s_u);
}

// Greedy calls of a small batch: one CTA finishes every request (warp b takes
// request b) and, once all are finished (a block barrier), writes the commit
// lists with its first kCommitThreads threads, so the step needs no separate
// commit launch.  Trees stage their node data in dynamic shared memory, four
// arrays of p.nodes entries per warp.  The KV slots of up to kStagedSlots rows
// and the sequence lengths (inputs) are staged in shared memory before the
// dependency wait, so the commit gathers them without a memory round trip.
constexpr int kStagedSlots = 1024;

template <bool TREE>
__global__ void __launch_bounds__(1024) k_accept_commit(ChainParams pc, TreeParams pt, OutView out, Ws ws,
                                                       CommitParams cp) {
  extern __shared__ int32_t s_nodes[];
  __shared__ int64_t s_slots[kStagedSlots];
  __shared__ int64_t s_seq[kSmallGreedyBatch];
  const int warp = threadIdx.x >> 5;
  const int B = TREE ? pt.batch : pc.batch;
  const int64_t rows = TREE ? pt.lg.rows : pc.lg.rows;
  const bool stage_slots = cp.row_slots && out.commit_src_slot && rows <= kStagedSlots;
  const bool stage_seq = cp.seq_lens && out.commit_dst_pos;
  for (int64_t i = threadIdx.x; stage_slots && i < rows; i += blockDim.x) s_slots[i] = cp.row_slots[i];
  if (stage_seq && threadIdx.x < B) s_seq[threadIdx.x] = cp.seq_lens[threadIdx.x];
  if (warp < B) {
    if constexpr (TREE) {
      const int N = pt.nodes;
      int32_t* base = s_nodes + static_cast<size_t>(warp) * 4 * N;
      accept_tree_request(pt, out, ws, warp, base, base + N, base + 2 * N, reinterpret_cast<float*>(base + 3 * N),
                          nullptr, nullptr);  // greedy calls only
    } else {
      accept_chain_request(pc, out, ws, warp);
    }
  }
  __syncthreads();  // every request's outputs are written (and the staged slots)
  if (threadIdx.x < kCommitThreads)
    commit_block_named(out, cp, stage_slots ? s_slots : nullptr, stage_seq ? s_seq : nullptr);
}

}  // namespace

cudaError_t accept_smem_setup() {
  // node arrays up to kAcceptCommitSmemBytes beside the staged slots
  return cudaFuncSetAttribute(k_accept_commit<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kAcceptCommitSmemBytes));
}

bool accept_commit_fits(int32_t batch, int32_t nodes) {
  return batch >= 1 && batch <= kSmallGreedyBatch &&
         (nodes <= 0 || int64_t{16} * nodes * batch <= kAcceptCommitSmemBytes);
}

cudaError_t launch_accept_commit_chain(const ChainParams& p, const OutView& out, const CommitParams& cp, const Ws& ws,
                                       cudaStream_t stream) {
  const int threads = 32 * p.batch > kCommitThreads ? 32 * p.batch : kCommitThreads;
  return launch_pdl(k_accept_commit<false>, dim3(1), dim3(threads), 0, stream, p, TreeParams{}, out, ws, cp);
}

cudaError_t launch_accept_commit_tree(const TreeParams& p, const OutView& out, const CommitParams& cp, const Ws& ws,
                                      cudaStream_t stream) {
  const int threads = 32 * p.batch > kCommitThreads ? 32 * p.batch : kCommitThreads;
  const size_t smem = size_t{16} * p.nodes * p.batch;
  return launch_pdl(k_accept_commit<true>, dim3(1), dim3(threads), smem, stream, ChainParams{}, p, out, ws, cp);
}

cudaError_t launch_accept_chain(const ChainParams& p, const OutView& out, const Ws& ws, cudaStream_t stream) {
  const int blocks = (p.batch + kChainWarps - 1) / kChainWarps;
  return launch_pdl(k_accept_chain, dim3(blocks), dim3(32 * kChainWarps), 0, stream, p, out, ws);
}

cudaError_t launch_accept_tree(const TreeParams& p, const OutView& out, const Ws& ws, cudaStream_t stream) {
  return launch_pdl(k_accept_tree, dim3(p.batch), dim3(32), 0, stream, p, out, ws);
}

}  // namespace sv
