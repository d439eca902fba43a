// Speculative-decoding verification: plain fp64 CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
// its Python binding) may call, link or load this file; only the tests, the
// package smoke check and the benchmark's CPU-baseline leg do.  It shares no
// code, header or table with the CUDA path.
//
// Every quantity is computed the slow, obvious way: one row at a time, one
// vocabulary entry at a time, in double precision.  bf16 logits are widened
// exactly (bits << 16) and then to double; fp32 logits and q are widened to
// double; temperatures are the caller's fp32 values widened to double.
//
// Sources (page title, then section / equation):
//   [E2D]  "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理"
//          (tom-jerr.github.io/sglang/eagle2-in-sglang)
//   [SGO]  SGLang speculative-decoding overview (zdszero.github.io/speculative_decoding.html)
//
//   verify layout, m+1 outputs when all pass ......... [E2D] §1.1, notation table
//   greedy acceptance, same tie-breaking ............. [E2D] §1.2 first bullet; [SGO] "为什么结果不受 draft 影响"
//   alpha = min(1, p/q) .............................. [E2D] §1.2, equation for alpha_j
//   residual p' = [p-q]_+ / sum [p-q]_+ .............. [E2D] §1.2, equation for p'_j
//   softmax with temperature (l/T) ................... [E2D] §6.2, equation for q_j(b|d)
//   inverse CDF (count of cdf <= u, clamped) ......... [E2D] §6.2, sample_path() paragraph
//   ragged verify_lens incl. anchor, offsets ......... [E2D] §5.6.5
//   commit_lens = correct_len + 1, rows [anchor..] ... [E2D] §5.6.6 and §8.1 table
//   KV moved to the slots after seq_lens ............. [SGO] "两个容易误解的工程细节"
//   greedy tree walk (chain is a special case) ....... [SGO] "为什么结果不受 draft 影响" (verify_tree_greedy)
//   target-only tree sampling, thresholds 1.0 ........ [SGO] same section (tree_speculative_sampling_target_only)
//
// Readings where the pages leave a step open (each also listed in the design notes):
//   * acceptance is the strict test u*q(d) < p(d) (equals u < alpha for q>0, u in [0,1)).
//   * inverse CDF: smallest v with cumsum_v > u*S; if none (rounding), the last v with w_v > 0.
//   * residual mass S <= 0: sample from p instead and set status bit 16.
//   * argmax ties: lowest index.  NaN and +inf elements are excluded (status bit 2); a row
//     with no finite-or-(-inf) maximum (all -inf) is unusable: stop there, bonus -1.
//   * a request samples iff 1e-30 <= T < inf ([E2D] §6.2: T > 0 rows sample, greedy rows take
//     the argmax); any other temperature (0, negative, NaN, inf, tiny) is verified greedily.
//   * target-only tree: at node cur with uniform u, walk the children in order, c += p(tok);
//     accept the first child with u < c/theta_acc or p(tok) >= theta_single.  A child whose
//     token repeats an earlier sibling's is skipped (status bit 32).  If none is accepted,
//     sample from p with the children's tokens zeroed; at a leaf, sample from p.
//     Thresholds other than 1 make the rule lossy and no page fixes them; the reading is pinned
//     by its special cases (theta_single = 0 takes the first child at every level and is
//     inclusive at p = 0; no child passing stops at the root with the children excluded; a huge
//     theta_acc leaves the first child at or above theta_single) and by the acceptance law
//     min(1, c_i/theta_acc) - min(1, c_(i-1)/theta_acc) of child i.
//   * a tree that fails validation is verified as its root alone (status bit 4).
//   * a request whose row range is invalid commits nothing (status bit 8).
//
// Decision gaps.  For each request the oracle reports how far each decision on
// its path was from going the other way, in the units of the caller's uniform:
//   test_gap[b, k]  the acceptance test(s) made at step k of the path (chain row
//                   start + k, or the tree node at depth k): |u - p/q| for a p/q
//                   test; min(|u - c/theta_acc|, |p - theta_single|) over the
//                   children tried for a target-only node; +inf where no test
//                   was made (greedy steps, steps past the end of the path);
//   draw_gap[b]     the final inverse-CDF draw: the distance of u to the nearer
//                   CDF edge of the drawn index that some u in [0, 1) can cross
//                   (the lower edge when a positive weight lies before the
//                   index, the upper edge when one lies after it); +inf when
//                   no draw was made or the weights have a single positive entry;
//   min_gap[b]      the minimum of the above.
// A decision whose gap is below 1e-6 is one a finite-precision implementation
// may legitimately take the other way; every decision before the first such
// one is certain.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr uint32_t kTokenRange = 1u;
constexpr uint32_t kNonFinite = 2u;
constexpr uint32_t kBadTree = 4u;
constexpr uint32_t kBadLayout = 8u;
constexpr uint32_t kResidualEmpty = 16u;
constexpr uint32_t kDupSibling = 32u;

constexpr double kInf = std::numeric_limits<double>::infinity();

struct Logits {
  const void* base;
  int dtype;   // 0 = fp32, 1 = bf16 bits
  int64_t ld;  // row stride in elements
  int32_t vocab;

  double at(int64_t row, int64_t v) const {
    if (dtype == 1) {
      uint16_t bits = static_cast<const uint16_t*>(base)[row * ld + v];
      uint32_t w = static_cast<uint32_t>(bits) << 16;
      float f;
      std::memcpy(&f, &w, sizeof f);
      return static_cast<double>(f);
    }
    return static_cast<double>(static_cast<const float*>(base)[row * ld + v]);
  }
};

// One row's target distribution.  p_v = exp((l_v - M)/T) / Z over the usable
// entries (finite or -inf); M is the maximum, argmax its lowest index.
struct RowDist {
  double M = -kInf;
  int64_t argmax = -1;
  double T = 0.0;  // > 0: sampling row; otherwise greedy (Z not formed)
  double Z = 0.0;
  bool nonfinite = false;
};

bool usable(double l) { return !std::isnan(l) && l != kInf; }

bool sampling_temperature(double T) { return T >= 1e-30 && T < kInf; }

RowDist row_dist(const Logits& lg, int64_t row, double T) {
  RowDist r;
  r.T = T;
  for (int64_t v = 0; v < lg.vocab; ++v) {
    double l = lg.at(row, v);
    if (!usable(l)) {
      r.nonfinite = true;
      continue;
    }
    if (l > r.M) {  // strict: the first (lowest) index of the maximum wins
      r.M = l;
      r.argmax = v;
    }
  }
  if (T > 0.0 && r.argmax >= 0) {  // callers pass T = 0 for greedy rows
    double Z = 0.0;
    for (int64_t v = 0; v < lg.vocab; ++v) {
      double l = lg.at(row, v);
      if (usable(l)) Z += std::exp((l - r.M) / T);
    }
    r.Z = Z;
  }
  return r;
}

double prob(const RowDist& r, double l) {
  if (!usable(l)) return 0.0;
  return std::exp((l - r.M) / r.T) / r.Z;
}

void row_probs(const Logits& lg, int64_t row, const RowDist& r, std::vector<double>& p) {
  p.assign(lg.vocab, 0.0);
  for (int64_t v = 0; v < lg.vocab; ++v) p[v] = prob(r, lg.at(row, v));
}

// Classic rejection test: accept d iff u * q(d) < p(d), i.e. u < min(1, p/q).
bool accept_pq(double p, double q, double u) { return u * q < p; }

// Residual weights w_v = max(0, p_v - q_v).
void residual(const std::vector<double>& p, const float* q, std::vector<double>& w) {
  w.resize(p.size());
  for (size_t v = 0; v < p.size(); ++v) w[v] = std::max(0.0, p[v] - static_cast<double>(q[v]));
}

// Inverse CDF over unnormalised weights: the smallest v whose running sum
// exceeds u * S.  Returns -1 when S <= 0.  *gap: distance of u to the nearer
// normalised CDF edge of the chosen index that a uniform in [0, 1) can cross.
// The lower edge counts only when positive weight lies before the index (with
// none, t = u*S >= 0 never falls below it); the upper edge only when positive
// weight lies after it (with none, it is S itself, and t < S for u < 1).
// +inf when neither edge counts; 0 when the rounding fallback fired.
int64_t sample_index(const double* w, int64_t n, double u, double* gap) {
  double S = 0.0;
  for (int64_t v = 0; v < n; ++v) S += w[v];
  if (!(S > 0.0)) {
    *gap = 0.0;
    return -1;
  }
  double t = u * S;
  double cum = 0.0;
  for (int64_t v = 0; v < n; ++v) {
    double prev = cum;
    cum += w[v];
    if (cum > t) {
      const double lower = prev > 0.0 ? (t - prev) / S : kInf;
      const double upper = cum < S ? (cum - t) / S : kInf;
      *gap = std::min(lower, upper);
      return v;
    }
  }
  *gap = 0.0;
  for (int64_t v = n - 1; v >= 0; --v)
    if (w[v] > 0.0) return v;
  return -1;
}

struct Out {
  int32_t* accept_len;
  int32_t* num_out;
  int32_t* out_tokens;  // [B, max_len]
  int32_t* bonus;
  int32_t* accept_rows;  // [B, max_len]
  int32_t* commit_cu;    // [B+1]
  int64_t* commit_src_slot;
  int64_t* commit_dst_pos;
  uint32_t* status;
  double* min_gap;
  double* test_gap;  // [B, max_len] or NULL
  double* draw_gap;  // [B] or NULL
};

struct ReqResult {
  int32_t r = 0;
  int32_t bonus = -1;
  bool committed = true;
  std::vector<int32_t> tokens;  // accepted draft tokens
  std::vector<int32_t> rows;    // rows committed: anchor row then accepted rows
  uint32_t status = 0;
  double gap = kInf;                // minimum over every decision below
  std::vector<double> test_gap;     // per step of the path: the acceptance test(s) made there
  double draw_gap = kInf;           // the final draw

  void test_at(size_t step, double g) {
    if (test_gap.size() <= step) test_gap.resize(step + 1, kInf);
    test_gap[step] = std::min(test_gap[step], g);
    gap = std::min(gap, g);
  }
  void draw(double g) {
    draw_gap = std::min(draw_gap, g);
    gap = std::min(gap, g);
  }
};

void write_request(const Out& o, int32_t b, int32_t max_len, const ReqResult& rr) {
  o.accept_len[b] = rr.r;
  o.num_out[b] = rr.committed ? rr.r + 1 : 0;
  o.bonus[b] = rr.bonus;
  o.status[b] = rr.status;
  if (o.min_gap) o.min_gap[b] = rr.gap;
  if (o.draw_gap) o.draw_gap[b] = rr.draw_gap;
  for (int32_t k = 0; k < max_len; ++k) {
    if (o.test_gap)
      o.test_gap[static_cast<int64_t>(b) * max_len + k] =
          static_cast<size_t>(k) < rr.test_gap.size() ? rr.test_gap[k] : kInf;
    int32_t tok = -1, row = -1;
    if (rr.committed && k < rr.r) tok = rr.tokens[k];
    if (rr.committed && k == rr.r) tok = rr.bonus;
    if (rr.committed && k <= rr.r) row = rr.rows[k];
    o.out_tokens[static_cast<int64_t>(b) * max_len + k] = tok;
    o.accept_rows[static_cast<int64_t>(b) * max_len + k] = row;
  }
}

// Commit bookkeeping: exclusive scan of commit_lens, then for each committed
// row its KV slot and its destination position seq_len + k.
void commit(const Out& o, int32_t B, int32_t max_len, const int64_t* row_slots, const int64_t* seq_lens) {
  o.commit_cu[0] = 0;
  for (int32_t b = 0; b < B; ++b) o.commit_cu[b + 1] = o.commit_cu[b] + o.num_out[b];
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t k = 0; k < o.num_out[b]; ++k) {
      int64_t dst = o.commit_cu[b] + k;
      int32_t row = o.accept_rows[static_cast<int64_t>(b) * max_len + k];
      if (o.commit_src_slot && row_slots) o.commit_src_slot[dst] = row_slots[row];
      if (o.commit_dst_pos && seq_lens) o.commit_dst_pos[dst] = seq_lens[b] + k;
    }
  }
}

template <typename F>
void for_requests(int32_t B, int32_t threads, F fn) {
  if (threads <= 1 || B <= 1) {
    for (int32_t b = 0; b < B; ++b) fn(b);
    return;
  }
  threads = std::min(threads, B);
  std::vector<std::thread> pool;
  for (int32_t t = 0; t < threads; ++t)
    pool.emplace_back([&, t] {
      for (int32_t b = t; b < B; b += threads) fn(b);
    });
  for (auto& th : pool) th.join();
}

// --------------------------------------------------------------------------
// Chains and ragged blocks
// --------------------------------------------------------------------------

struct ChainArgs {
  Logits lg;
  bool greedy_all;
  int32_t B;
  int64_t total_rows;
  int32_t max_len;
  const int32_t* cu;
  const int32_t* ids;
  const float* q;
  int64_t ldq;
  const float* temperature;
  const float* u_accept;
  const float* u_final;
};

ReqResult verify_chain_request(const ChainArgs& a, int32_t b) {
  ReqResult rr;
  int64_t start = a.cu[b], end = a.cu[b + 1];
  int64_t L = end - start;
  if (start < 0 || end > a.total_rows || L < 1 || L > a.max_len) {
    rr.status |= kBadLayout;
    rr.committed = false;
    rr.gap = kInf;
    return rr;
  }
  const double Tb = a.greedy_all ? 0.0 : static_cast<double>(a.temperature[b]);
  const bool greedy = !sampling_temperature(Tb);
  const double T = greedy ? 0.0 : Tb;
  rr.rows.push_back(static_cast<int32_t>(start));

  enum { kAllAccepted, kRejected, kUnusable } how = kAllAccepted;
  int64_t j = 0;
  for (; j < L - 1; ++j) {
    const int64_t row = start + j;
    RowDist st = row_dist(a.lg, row, T);
    if (st.nonfinite) rr.status |= kNonFinite;
    if (st.argmax < 0) {
      how = kUnusable;
      break;
    }
    const int64_t d = a.ids[row + 1];
    if (d < 0 || d >= a.lg.vocab) {
      rr.status |= kTokenRange;
      how = kRejected;
      break;
    }
    bool ok;
    if (greedy) {
      ok = (st.argmax == d);
    } else {
      const double p = prob(st, a.lg.at(row, d));
      const double qd = static_cast<double>(a.q[row * a.ldq + d]);
      const double u = static_cast<double>(a.u_accept[row]);
      ok = accept_pq(p, qd, u);
      if (qd > 0.0) rr.test_at(static_cast<size_t>(j), std::fabs(u - p / qd));
    }
    if (!ok) {
      how = kRejected;
      break;
    }
    rr.tokens.push_back(static_cast<int32_t>(d));
    rr.rows.push_back(static_cast<int32_t>(row + 1));
  }
  rr.r = static_cast<int32_t>(j);

  // The final token comes from row s = start + r: a correction after a
  // rejection, or the bonus when every draft passed.
  const int64_t s = start + j;
  RowDist st = row_dist(a.lg, s, T);
  if (st.nonfinite) rr.status |= kNonFinite;
  if (how == kUnusable || st.argmax < 0) {
    rr.status |= kNonFinite;
    rr.bonus = -1;
    return rr;
  }
  if (greedy) {
    rr.bonus = static_cast<int32_t>(st.argmax);
    return rr;
  }
  std::vector<double> p, w;
  row_probs(a.lg, s, st, p);
  if (how == kRejected) {
    residual(p, a.q + s * a.ldq, w);
  } else {
    w = p;
  }
  double gap = 0.0;
  int64_t v = sample_index(w.data(), static_cast<int64_t>(w.size()), a.u_final[b], &gap);
  if (v < 0) {
    rr.status |= kResidualEmpty;
    v = sample_index(p.data(), static_cast<int64_t>(p.size()), a.u_final[b], &gap);
  }
  rr.draw(gap);
  rr.bonus = static_cast<int32_t>(v);
  return rr;
}

// --------------------------------------------------------------------------
// Trees given by parent indices (optionally first-child / next-sibling lists)
// --------------------------------------------------------------------------

struct TreeArgs {
  Logits lg;
  int mode;  // 0 greedy, 1 target-only sampling
  int32_t B;
  int32_t N;
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* first_child;
  const int32_t* next_sibling;
  const float* temperature;
  double th_single;
  double th_acc;
  const float* u_accept;
  const float* u_final;
};

// Children of `cur` in verification order; false if the sibling lists are
// inconsistent with the parent array.
bool children_of(const TreeArgs& a, int32_t b, int32_t cur, std::vector<int32_t>& kids) {
  kids.clear();
  const int32_t* par = a.parents + static_cast<int64_t>(b) * a.N;
  if (!a.first_child) {
    for (int32_t i = cur + 1; i < a.N; ++i)
      if (par[i] == cur) kids.push_back(i);
    return true;
  }
  const int32_t* fc = a.first_child + static_cast<int64_t>(b) * a.N;
  const int32_t* ns = a.next_sibling + static_cast<int64_t>(b) * a.N;
  int32_t c = fc[cur];
  for (int32_t steps = 0; c != -1; ++steps) {
    if (steps >= a.N || c < 1 || c >= a.N || par[c] != cur) return false;
    kids.push_back(c);
    c = ns[c];
  }
  return true;
}

bool tree_valid(const TreeArgs& a, int32_t b) {
  const int32_t* par = a.parents + static_cast<int64_t>(b) * a.N;
  if (par[0] != -1) return false;
  for (int32_t i = 1; i < a.N; ++i)
    if (par[i] < 0 || par[i] >= i) return false;
  std::vector<int32_t> kids;
  for (int32_t i = 0; i < a.N; ++i)
    if (!children_of(a, b, i, kids)) return false;
  return true;
}

ReqResult verify_tree_request(const TreeArgs& a, int32_t b) {
  ReqResult rr;
  const int32_t N = a.N;
  const int64_t row0 = static_cast<int64_t>(b) * N;
  const int32_t* tok = a.tokens + row0;
  const bool ok_tree = tree_valid(a, b);
  if (!ok_tree) rr.status |= kBadTree;
  const double Tb = (a.mode == 1) ? static_cast<double>(a.temperature[b]) : 0.0;
  const bool greedy = !sampling_temperature(Tb);
  const double T = greedy ? 0.0 : Tb;

  int32_t cur = 0;
  rr.rows.push_back(static_cast<int32_t>(row0));
  std::vector<int32_t> kids;
  std::vector<double> p, w;
  for (;;) {
    const int64_t row = row0 + cur;
    RowDist st = row_dist(a.lg, row, T);
    if (st.nonfinite) rr.status |= kNonFinite;
    if (st.argmax < 0) {
      rr.status |= kNonFinite;
      rr.bonus = -1;
      break;
    }
    if (ok_tree) {
      children_of(a, b, cur, kids);
    } else {
      kids.clear();  // an invalid tree is verified as its root alone
    }
    int32_t next = -1;
    std::vector<int32_t> seen;
    if (greedy) {
      for (int32_t k : kids) {
        if (tok[k] < 0 || tok[k] >= a.lg.vocab) {
          rr.status |= kTokenRange;
          continue;
        }
        if (tok[k] == st.argmax) {
          next = k;
          break;
        }
      }
      if (next < 0) {
        rr.bonus = static_cast<int32_t>(st.argmax);
        break;
      }
    } else {
      const double u = static_cast<double>(a.u_accept[row]);
      double c = 0.0;
      for (int32_t k : kids) {
        if (tok[k] < 0 || tok[k] >= a.lg.vocab) {
          rr.status |= kTokenRange;
          continue;
        }
        if (std::find(seen.begin(), seen.end(), tok[k]) != seen.end()) {
          rr.status |= kDupSibling;
          continue;
        }
        seen.push_back(tok[k]);
        const double pk = prob(st, a.lg.at(row, tok[k]));
        c += pk;
        rr.test_at(rr.tokens.size(), std::min(std::fabs(u - c / a.th_acc), std::fabs(pk - a.th_single)));
        if (u < c / a.th_acc || pk >= a.th_single) {
          next = k;
          break;
        }
      }
      if (next < 0) {
        row_probs(a.lg, row, st, p);
        w = p;
        for (int32_t t : seen) w[t] = 0.0;
        double gap = 0.0;
        int64_t v = sample_index(w.data(), static_cast<int64_t>(w.size()), a.u_final[b], &gap);
        if (v < 0) {
          rr.status |= kResidualEmpty;
          v = sample_index(p.data(), static_cast<int64_t>(p.size()), a.u_final[b], &gap);
        }
        rr.draw(gap);
        rr.bonus = static_cast<int32_t>(v);
        break;
      }
    }
    rr.tokens.push_back(tok[next]);
    rr.rows.push_back(static_cast<int32_t>(row0 + next));
    cur = next;
  }
  rr.r = static_cast<int32_t>(rr.tokens.size());
  return rr;
}

}  // namespace

// ----------------------------------------------------------------------------
// C entry points (called from Python through ctypes by the tests)
// ----------------------------------------------------------------------------

extern "C" {

typedef struct {
  int32_t* accept_len;
  int32_t* num_out;
  int32_t* out_tokens;
  int32_t* bonus;
  int32_t* accept_rows;
  int32_t* commit_cu;
  int64_t* commit_src_slot;
  int64_t* commit_dst_pos;
  uint32_t* status;
  double* min_gap;
  double* test_gap;  // [B, max_len] per-step acceptance-test gaps, or NULL
  double* draw_gap;  // [B] final-draw gaps, or NULL
} oracle_out_t;

// Chain or ragged verification.  greedy_all != 0 verifies every request
// greedily (temperature, q and uniforms may be NULL); otherwise each request
// with temperature > 0 uses p/q rejection with residual resampling and the
// others are verified greedily.  cu_seqlens gives each request's rows
// [cu[b], cu[b+1]) including the anchor row.
int oracle_verify_chain(int greedy_all, const void* logits, int dtype, int64_t ld, int32_t batch,
                        int64_t total_rows, int32_t max_len, int32_t vocab, const int32_t* cu_seqlens,
                        const int32_t* verify_ids, const float* q, int64_t ldq, const float* temperature,
                        const float* u_accept, const float* u_final, const int64_t* row_slots,
                        const int64_t* seq_lens, const oracle_out_t* out, int32_t threads) {
  ChainArgs a{{logits, dtype, ld, vocab}, greedy_all != 0, batch, total_rows, max_len, cu_seqlens,
              verify_ids, q, ldq, temperature, u_accept, u_final};
  Out o{out->accept_len, out->num_out, out->out_tokens, out->bonus, out->accept_rows,
        out->commit_cu, out->commit_src_slot, out->commit_dst_pos, out->status, out->min_gap,
        out->test_gap, out->draw_gap};
  for_requests(batch, threads, [&](int32_t b) { write_request(o, b, max_len, verify_chain_request(a, b)); });
  commit(o, batch, max_len, row_slots, seq_lens);
  return 0;
}

// Tree verification: mode 0 greedy, mode 1 target-only sampling.  Node i of
// request b owns logits row b*nodes + i; node 0 is the root (anchor).
int oracle_verify_tree(int mode, const void* logits, int dtype, int64_t ld, int32_t batch, int32_t nodes,
                       int32_t vocab, const int32_t* tokens, const int32_t* parents,
                       const int32_t* first_child, const int32_t* next_sibling, const float* temperature,
                       double threshold_single, double threshold_acc, const float* u_accept,
                       const float* u_final, const int64_t* row_slots, const int64_t* seq_lens,
                       const oracle_out_t* out, int32_t threads) {
  TreeArgs a{{logits, dtype, ld, vocab}, mode, batch, nodes, tokens, parents,
             (first_child && next_sibling) ? first_child : nullptr,
             (first_child && next_sibling) ? next_sibling : nullptr,
             temperature, threshold_single, threshold_acc, u_accept, u_final};
  Out o{out->accept_len, out->num_out, out->out_tokens, out->bonus, out->accept_rows,
        out->commit_cu, out->commit_src_slot, out->commit_dst_pos, out->status, out->min_gap,
        out->test_gap, out->draw_gap};
  for_requests(batch, threads, [&](int32_t b) { write_request(o, b, nodes, verify_tree_request(a, b)); });
  commit(o, batch, nodes, row_slots, seq_lens);
  return 0;
}

// Per-row statistics: maximum, lowest argmax, Z = sum exp((l-M)/T) (0 when
// the row's temperature is <= 0 or row_temp is NULL), p at probe[row] (when
// given and T > 0), and flags (bit 2 non-finite entries).
int oracle_row_stats(const void* logits, int dtype, int64_t ld, int64_t rows, int32_t vocab,
                     const float* row_temp, const int32_t* probe, double* out_max, int32_t* out_argmax,
                     double* out_z, double* out_p, uint32_t* out_flags) {
  Logits lg{logits, dtype, ld, vocab};
  for (int64_t r = 0; r < rows; ++r) {
    double T = row_temp ? static_cast<double>(row_temp[r]) : 0.0;
    if (!sampling_temperature(T)) T = 0.0;
    RowDist st = row_dist(lg, r, T);
    out_max[r] = st.M;
    out_argmax[r] = static_cast<int32_t>(st.argmax);
    out_z[r] = st.Z;
    out_flags[r] = st.nonfinite ? kNonFinite : 0u;
    if (out_p) {
      double pv = 0.0;
      if (probe && T > 0.0 && st.argmax >= 0 && probe[r] >= 0 && probe[r] < vocab)
        pv = prob(st, lg.at(r, probe[r]));
      out_p[r] = pv;
    }
  }
  return 0;
}

// The full target distribution of one row (for identity checks).
int oracle_row_probs(const void* logits, int dtype, int64_t ld, int64_t row, int32_t vocab, double T,
                     double* p_out) {
  Logits lg{logits, dtype, ld, vocab};
  if (!sampling_temperature(T)) return -1;
  RowDist st = row_dist(lg, row, T);
  if (st.argmax < 0) return -1;
  std::vector<double> p;
  row_probs(lg, row, st, p);
  std::copy(p.begin(), p.end(), p_out);
  return 0;
}

// The residual weights max(0, p - q) the oracle resamples from.
void oracle_residual(const double* p, const float* q, int64_t n, double* w_out) {
  std::vector<double> pv(p, p + n), w;
  residual(pv, q, w);
  std::copy(w.begin(), w.end(), w_out);
}

// The acceptance test used on every sampled chain row.
int oracle_accept(double p, double q, double u) { return accept_pq(p, q, u) ? 1 : 0; }

// The inverse-CDF sampler used for every correction / bonus token.
int64_t oracle_sample_index(const double* w, int64_t n, double u, double* gap) {
  double g = 0.0;
  int64_t v = sample_index(w, n, u, &g);
  if (gap) *gap = g;
  return v;
}

}  // extern "C"
