/*
 * DBSCAN oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU DBSCAN written from the definitions in
 * "Design and optimization of DBSCAN Algorithm based on CUDA" (Wang et al.),
 * §II "Background":
 *   - eps-neighbourhood: all points within distance eps of a point;
 *   - core point: at least MinPts points within distance eps of it;
 *   - reachability: a chain of directly reachable points whose every step
 *     starts at a core point;
 *   - cluster: maximal (closed under reachability) and connected.
 * §IV-A fixes the comparison as squared distance against eps^2, and §IV-B
 * writes the neighbour test as "distance <= eps^2" (inclusive).
 *
 * Readings taken where the page is silent or inconsistent (each also listed
 * in the design notes of this repository):
 *   - the point itself belongs to its eps-neighbourhood (distance 0 <= eps^2),
 *     so it counts toward MinPts;
 *   - core means count >= MinPts ("at least" in §II, not the "greater than"
 *     of §IV-B);
 *   - eps^2 is the single-precision product eps*eps of the float eps;
 *   - clusters are the connected components of the core points under the
 *     eps relation; a cluster is named by its smallest core-point index;
 *   - a non-core point with a core neighbour (a border point) takes the
 *     smallest name among the clusters of its core neighbours; a point with
 *     no core neighbour is noise, labelled -1.
 *
 * The algorithm is the textbook one: an O(N^2 d) counting double loop, then a
 * breadth-first expansion started from each unlabelled core point in
 * ascending index order.  Because expansions start in ascending order, each
 * cluster's name is its smallest core index, and the first expansion that
 * reaches a border point is the one with the smallest name.  No N x N matrix
 * is stored.  Arithmetic is double precision: coordinates are converted by the
 * caller, and for integer coordinates every squared distance is exact.
 *
 * This file shares no code with the CUDA library and must not be linked into
 * it; only tests, the smoke check and the benchmark's CPU-baseline leg use it.
 */
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* eps^2 as the single-precision product of the single-precision eps. */
static double threshold_sq(float eps)
{
    volatile float e2 = eps * eps;  /* volatile: keep the float rounding step */
    return (double)e2;
}

/* Squared Euclidean distance between points i and j (row-major [n, d]). */
static double sq_dist(const double *pts, int32_t d, int64_t i, int64_t j)
{
    const double *a = pts + i * (int64_t)d;
    const double *b = pts + j * (int64_t)d;
    double s = 0.0;
    for (int32_t k = 0; k < d; ++k) {
        double t = a[k] - b[k];
        s += t * t;
    }
    return s;
}

/* Number of points within eps of point i, the point itself included. */
static int32_t neighbour_count(const double *pts, int64_t n, int32_t d,
                               double thr, int64_t i)
{
    int32_t c = 0;
    for (int64_t j = 0; j < n; ++j)
        if (sq_dist(pts, d, i, j) <= thr)
            ++c;
    return c;
}

/* cnt[i] = |eps-neighbourhood of i| for every i. */
void oracle_counts(const double *pts, int64_t n, int32_t d, float eps,
                   int32_t *cnt)
{
    double thr = threshold_sq(eps);
    for (int64_t i = 0; i < n; ++i)
        cnt[i] = neighbour_count(pts, n, d, thr, i);
}

/* Counts for the listed rows only (sampled checks at large n). */
void oracle_row_counts(const double *pts, int64_t n, int32_t d, float eps,
                       const int64_t *rows, int64_t nrows, int32_t *cnt)
{
    double thr = threshold_sq(eps);
    for (int64_t r = 0; r < nrows; ++r)
        cnt[r] = neighbour_count(pts, n, d, thr, rows[r]);
}

/* Indices j (ascending) with d^2(i, j) <= eps^2, i itself included.
 * Writes at most cap of them; returns the full count. */
int64_t oracle_row_neighbours(const double *pts, int64_t n, int32_t d,
                              float eps, int64_t i, int64_t *out, int64_t cap)
{
    double thr = threshold_sq(eps);
    int64_t c = 0;
    for (int64_t j = 0; j < n; ++j) {
        if (sq_dist(pts, d, i, j) <= thr) {
            if (c < cap)
                out[c] = j;
            ++c;
        }
    }
    return c;
}

/* Threads the count loop of oracle_dbscan uses: 1 unless this file was built
 * with OpenMP (a separately timed baseline; the loop's iterations are
 * independent, so the result does not depend on it). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Full DBSCAN.  Outputs: cnt[n], core[n] (0/1), label[n] (cluster name or -1).
 * Returns 0, or -1 if the work queue cannot be allocated. */
int oracle_dbscan(const double *pts, int64_t n, int32_t d, float eps,
                  int32_t min_pts, int32_t *cnt, uint8_t *core, int32_t *label)
{
    double thr = threshold_sq(eps);

#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < n; ++i) {
        cnt[i] = neighbour_count(pts, n, d, thr, i);
        core[i] = (uint8_t)(cnt[i] >= min_pts);
        label[i] = -1;
    }
    if (n == 0)
        return 0;

    int64_t *queue = (int64_t *)malloc((size_t)n * sizeof(int64_t));
    if (!queue)
        return -1;
#ifdef _OPENMP
    /* OpenMP build only: the scan of one expansion step tests every j in
     * parallel first (hit[j]), then applies the hits in ascending j.  Testing
     * j reads label[j] alone and applying a hit writes label[j] alone, so the
     * labels and the queue order are those of the plain loop below. */
    uint8_t *hit = (uint8_t *)malloc((size_t)n);
    if (!hit) {
        free(queue);
        return -1;
    }
#endif

    for (int64_t root = 0; root < n; ++root) {
        if (!core[root] || label[root] != -1)
            continue;
        int32_t name = (int32_t)root;
        int64_t head = 0, tail = 0;
        label[root] = name;
        queue[tail++] = root;
        while (head < tail) {
            int64_t q = queue[head++];          /* q is a core point */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
            for (int64_t j = 0; j < n; ++j)
                hit[j] = (uint8_t)(label[j] == -1 && sq_dist(pts, d, q, j) <= thr);
            for (int64_t j = 0; j < n; ++j) {
                if (!hit[j])
                    continue;
                label[j] = name;
                if (core[j])
                    queue[tail++] = j;
            }
#else
            for (int64_t j = 0; j < n; ++j) {
                if (label[j] != -1)
                    continue;
                if (sq_dist(pts, d, q, j) > thr)
                    continue;
                label[j] = name;                /* j is reachable from q */
                if (core[j])
                    queue[tail++] = j;          /* only core points expand */
            }
#endif
        }
    }
#ifdef _OPENMP
    free(hit);
#endif
    free(queue);
    return 0;
}
