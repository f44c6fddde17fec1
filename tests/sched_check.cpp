// Host check of the tensor-core sweeps' work-unit schedule (tc_schedule.h):
// enumerates every unit the way the producer does, applies the epilogue's skip
// rules, and verifies that each tile pair a sweep must evaluate is evaluated
// exactly once and no other pair is.  Prints "ok" or the first failure.
#include <cstdio>
#include <vector>

#include "../all_pairs_distance_gb300/csrc/tc_schedule.h"

using namespace dbscan;

enum { COUNT, UNION, BORDER, UNION_ONE_BAND };

static bool run(int mode, int n_rows, int n_cols, int rt) {
    const int nrt = (n_rows + TC_TILE - 1) / TC_TILE, nct = (n_cols + TC_TILE - 1) / TC_TILE;
    std::vector<unsigned char> seen((size_t)nrt * nct, 0);
    const int tri = mode != BORDER;
    const bool uni = mode == UNION || mode == UNION_ONE_BAND;
    // the union's bands, or the single band [1, end) of small problems
    const int nb = mode == UNION ? UNION_BANDS : 1;
    for (int bd = 0; bd < nb; ++bd) {
        const int lo = mode == UNION ? kUnionBandEdges[bd] : (uni ? 1 : 0);
        const int hi = mode == UNION ? kUnionBandEdges[bd + 1] : -1;
        const TcSched s = tc_sched(n_rows, n_cols, tri, lo, hi, rt, tc_chunk(uni, hi, n_cols));
        for (unsigned u = 0; u < s.units; ++u) {
            int rb, nrow, t0, t1;
            if (!tc_unit(s, u, tri, lo, hi, rb, nrow, t0, t1)) continue;
            if (rb < 0 || rb % rt || nrow < 1 || rb + nrow > nrt || t0 < 0 || t1 > nct) {
                printf("bad unit mode %d rows %d cols %d rt %d: u %u rb %d nrow %d t [%d, %d)\n", mode,
                       n_rows, n_cols, rt, u, rb, nrow, t0, t1);
                return false;
            }
            for (int r = rb; r < rb + nrow; ++r)
                for (int t = t0; t < t1; ++t) {
                    // the epilogue's skips: below the diagonal in the triangle, and
                    // for the union the diagonal too
                    if (tri && (uni ? t <= r : t < r)) continue;
                    ++seen[(size_t)r * nct + t];
                }
        }
    }
    for (int r = 0; r < nrt; ++r)
        for (int t = 0; t < nct; ++t) {
            const int want = mode == BORDER ? 1 : (uni ? (t > r) : (t >= r));
            if (seen[(size_t)r * nct + t] != want) {
                printf("mode %d rows %d cols %d rt %d: pair (%d, %d) evaluated %d times, want %d\n", mode,
                       n_rows, n_cols, rt, r, t, seen[(size_t)r * nct + t], want);
                return false;
            }
        }
    return true;
}

int main() {
    const int tiles[] = {1, 2, 3, 7, 33, 511, 512, 513, 1024, 1025, 1537, 2600};
    for (int rt = 1; rt <= 2; ++rt)
        for (int a : tiles)
            for (int ra : {0, 1, 77}) {
                const int n = a * TC_TILE - ra;
                if (n <= 0) continue;
                if (!run(COUNT, n, n, rt) || !run(UNION, n, n, rt) || !run(UNION_ONE_BAND, n, n, rt))
                    return 1;
                for (int b : {1, 5, 600}) {
                    if (!run(BORDER, n, b * TC_TILE - 3, rt)) return 1;
                }
            }
    printf("ok\n");
    return 0;
}
