// Host-side checks of the workspace layout and of the row-statistics chunk
// plan (no GPU needed).
//
// Layout: every region starts on a 256-byte boundary, in order, and holds what
// its users index for the given rows, batch, vocabulary, row bound and
// candidate count.
//
// For many shapes and grids: the queue items of every row, found the way the
// merge kernel finds them, map back to that row, cover its full vectors
// exactly once in increasing order with only the last one marked last, and
// every item belongs to exactly one row; the plan's item count fits the
// partial area the workspace layout reserves.  Built by tests/test_chunk_plan.py
// together with the library's other translation units.
#include <cstdio>
#include <vector>

#include "sv_stats.cu"

using namespace sv;

// Workspace layout: regions in order, 256-byte aligned, each as large as its users index.
static int check_ws_layout() {
  int bad = 0, cases = 0;
  const int64_t rowss[] = {0, 1, 5, 272, 1024, 1152, 65536};
  const int32_t batches[] = {0, 1, 8, 64, 256, 4096};
  const int32_t vocabs[] = {1, 3, 1000, 32000, 151936, 262144};
  const int32_t maxlens[] = {1, 5, 16, 1024};
  for (int64_t R : rowss)
    for (int32_t B : batches)
      for (int32_t V : vocabs)
        for (int32_t ML : maxlens) {
            const WsLayout L = ws_layout(R, B, V, ML);
            ++cases;
            const size_t r1 = R > 0 ? R : 1, b1 = B > 0 ? B : 1, m1 = ML > 0 ? ML : 1;
            const size_t nfull = (V > 0 ? V : 1) / 4;
            const size_t cpr = nfull >= 1 ? (nfull + 1023) / 1024 : 1;  // chunks per row, 1024-vector chunks
            const size_t starts[] = {L.done_cnt, L.counters_end, L.rowstat, L.partial, L.psb, L.state, L.excl,
                                     L.ureq, L.tsum, L.total};
            bool ok = L.done_cnt == 0 && L.counters_end >= 16 && L.rowstat >= L.counters_end;
            for (size_t i = 1; i < sizeof(starts) / sizeof(starts[0]); ++i)
              ok = ok && starts[i] % 256 == 0 && starts[i] >= starts[i - 1];
            ok = ok && L.partial - L.rowstat >= sizeof(RowStat) * r1;
            ok = ok && L.psb - L.partial >= sizeof(RowPartial) * r1 * cpr;
            ok = ok && L.state - L.psb >= sizeof(float) * r1 * cpr;
            ok = ok && L.excl - L.state >= sizeof(ReqState) * b1;
            ok = ok && L.ureq - L.excl >= sizeof(int32_t) * b1 * m1;
            ok = ok && L.tsum - L.ureq >= sizeof(float) * b1;
            ok = ok && L.ntiles == (V + kTile - 1) / kTile &&
                 L.total - L.tsum >= sizeof(uint64_t) * b1 * static_cast<size_t>(L.ntiles > 0 ? L.ntiles : 1);
            if (!ok) {
              if (bad < 10)
                std::printf("ws layout: R=%lld B=%d V=%d ML=%d\n", (long long)R, B, V, ML);
              ++bad;
            }
          }
  std::printf("workspace layout: %d cases, %d failures\n", cases, bad);
  return bad;
}

int main() {
  int bad = check_ws_layout(), cases = 0;
  const int vocabs[] = {1, 3, 7, 8, 9, 16, 255, 1000, 2048, 4099, 8191, 8192, 8200, 32000, 128256, 151936, 262144};
  const int64_t rowss[] = {1, 2, 5, 17, 64, 272, 1024, 1152, 5000};
  const int grids[] = {1, 3, 40, 152, 456};
  for (int dt = 0; dt < 2; ++dt)
    for (int V : vocabs)
      for (int64_t R : rowss)
        for (int G : grids) {
          const LogitsView lg{nullptr, dt == 0 ? SV_F32 : SV_BF16, V, R, V};
          const int64_t nfull = V / (dt == 0 ? 4 : 8);
          const ChunkPlan P = chunk_plan(lg, G);
          const WsLayout L = ws_layout(R, 1, V, 1);
          const int64_t cap = static_cast<int64_t>((L.psb - L.partial) / sizeof(RowPartial));
          ++cases;
          if (P.n_items > cap) {
            std::printf("capacity: V=%d R=%lld G=%d dt=%d items=%lld cap=%lld\n", V, (long long)R, G, dt,
                        (long long)P.n_items, (long long)cap);
            ++bad;
          }
          std::vector<int> seen(static_cast<size_t>(P.n_items), 0);
          for (int64_t row = 0; row < R; ++row) {
            const bool head = row < P.rows_a;  // as k_row_merge finds a row's items
            const int32_t cnt = head ? P.cpr_a : P.cpr_b;
            const int64_t base = head ? row * P.cpr_a : P.n_a + (row - P.rows_a) * P.cpr_b;
            int32_t expect = 0;  // next stage the row's chunks must start at
            for (int32_t j = 0; j < cnt; ++j) {
              const int64_t it = base + j;
              if (it < 0 || it >= P.n_items) {
                std::printf("item out of range: V=%d R=%lld G=%d row=%lld\n", V, (long long)R, G, (long long)row);
                ++bad;
                break;
              }
              ++seen[static_cast<size_t>(it)];
              int32_t r, s0, s1;
              bool last;
              chunk_geometry(P, static_cast<int32_t>(it), r, s0, s1, last);
              const bool ok = r == row && s0 == expect && s1 > s0 && last == (j == cnt - 1);
              if (!ok) {
                if (bad < 20)
                  std::printf("geometry: V=%d R=%lld G=%d dt=%d row=%lld j=%d: r=%d s0=%d s1=%d last=%d\n", V,
                              (long long)R, G, dt, (long long)row, j, r, s0, s1, (int)last);
                ++bad;
              }
              expect = s1;
            }
            // Stages of 1024 vectors cover the row's full vectors (at least one stage: the ragged tail rides on it).
            const int32_t want = static_cast<int32_t>(nfull == 0 ? 1 : (nfull + kChunkVecs - 1) / kChunkVecs);
            if (expect != want || P.nst != want) {
              if (bad < 20)
                std::printf("coverage: V=%d R=%lld G=%d row=%lld ends at stage %d of %d (plan %d)\n", V,
                            (long long)R, G, (long long)row, expect, want, P.nst);
              ++bad;
            }
          }
          for (int64_t i = 0; i < P.n_items; ++i)
            if (seen[static_cast<size_t>(i)] != 1) {
              std::printf("item %lld owned %d times: V=%d R=%lld G=%d\n", (long long)i, seen[static_cast<size_t>(i)],
                          V, (long long)R, G);
              ++bad;
              break;
            }
        }
  std::printf("chunk plan: %d cases, %d failures (with the layout's)\n", cases, bad);
  return bad != 0;
}
