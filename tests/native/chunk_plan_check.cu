// Host-side check of the row-statistics chunk plan (no GPU needed).
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

int main() {
  int bad = 0, cases = 0;
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
  std::printf("chunk plan: %d cases, %d failures\n", cases, bad);
  return bad != 0;
}
