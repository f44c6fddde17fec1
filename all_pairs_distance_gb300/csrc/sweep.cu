// The tiled all-pairs sweeps on CUDA cores: neighbour counting (pass 1),
// core-core union-find (pass 2) and border assignment (pass 3).
//
// "Design and optimization of DBSCAN Algorithm based on CUDA" stages tiles of
// points in shared memory (§IV-A3), unrolls the inner loop (§IV-A4), fuses
// the distance evaluation with the neighbour count so no distance matrix is
// stored (§IV-B1), and hoists the per-point terms of the squared distance out
// of the loop (§IV-B2).  The sweeps here keep those ideas and change the rest
// for sm_103a:
//
// * Work is a persistent grid pulling units (one 128-row block x a run of
//   128-column tiles) from an atomic counter.  Counting and union sweep only
//   the upper triangle of tiles (a pair is evaluated once and, in pass 1,
//   credited to both points); the border sweep is a rectangle (candidates x
//   cores).
// * Column tiles stream through a 3-stage cp.async ring in shared memory; the
//   tile layout (structure of arrays, 128 points per row) makes every load a
//   conflict-free 16-byte vector.  The union and border sweeps also stage one
//   int per column (the union-find parent, or the final cluster label), so a
//   neighbour pair is usually settled from shared memory alone.
// * A thread owns 8 rows x 8 columns per tile.  Per pair the fast path does d
//   fused multiply-adds (two pairs per packed f32x2 instruction for d <= 4)
//   into v_ij = nrm_j - 2 c_i . c_j, and half a three-input min; a row whose
//   minimum over its 8 columns is not below its threshold T_i has no neighbour
//   there.  Only rows with a neighbour take the slow path, which re-tests the
//   8 pairs one by one and acts on each neighbour pair.
#include "dbscan_internal.cuh"
#include "tc_schedule.h"

#include <map>
#include <mutex>
#include <utility>

namespace dbscan {

constexpr int THREADS = 256;
constexpr int R = 8;             // rows per thread
constexpr int C = 8;             // columns per thread per tile
constexpr int UF_CAP = 1 << 22;  // iteration cap of union-find loops

// Counters in Ctrl::unit_ctr.
constexpr int CTR_COUNT = 0, CTR_UNION0 = 1, CTR_BORDER = 5;
// Union bands (both paths): UNION_BANDS and kUnionBandEdges in tc_schedule.h.

struct SweepArgs {
    const float *rows;     // staged row points
    const float *rowT;     // row thresholds
    const int *n_rows;     // device-side row count
    const float *cols;     // staged column points
    const int *n_cols;     // device-side column count
    const int *aux;        // per-column int staged with the tile (parent or label), or null
    int tri;               // 1: rows and cols are one set, sweep the upper triangle
    int ulo, uhi;          // unit range [ulo * grid, uhi * grid), uhi = -1: to the end
    unsigned *ctr;         // work-unit counter (zeroed before the launch)
    Ctrl *ctrl;
    int *cnt;              // pass 1: neighbour counts
    int *parent;           // pass 2: union-find parents
    const int *candidx;    // pass 3: original index of each candidate position
    int32_t *labels;       // pass 3: labels (original order)
    int srank, sworld;     // sharding: this rank takes units ubegin + k * sworld + srank
    const float *rbox, *cbox;   // per-tile bounding boxes of rows / columns (d x (min, max))
    int cull;              // 1: skip column tiles whose box is eps or more from the row tile's
    int band, blo, bhi;    // union: only column tiles t with t - rb in [blo, bhi) (-1: no limit)
    const int *troot;      // union: common root of each tile's points, or -1; tile pairs
                           // with one common root are skipped
};

// Position of a thread's m-th row (or column) inside a 128-point tile.  Two
// runs of four make each group of 8 threads read 128 contiguous bytes.
__device__ __forceinline__ int slot_of(int g, int m) {
    return (m < 4) ? (4 * g + m) : (64 + 4 * g + (m - 4));
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---- union-find (parent[x] <= x always; roots are component minima) -------
__device__ __noinline__ int uf_find(int *parent, int x, Ctrl *ctrl) {
    for (int it = 0; it < UF_CAP; ++it) {
        int p = __ldcg(parent + x);
        if (p == x) return x;
        int gp = __ldcg(parent + p);
        if (gp != p) __stcg(parent + x, gp);   // path halving
        x = gp;
    }
    set_error(ctrl, DBSCAN_ERR_INTERNAL);
    return x;
}

// Merge the sets of a and b; returns a node that is an ancestor of both
// (their common root at the moment of the merge).
__device__ __noinline__ int uf_unite(int *parent, int a, int b, Ctrl *ctrl) {
    for (int it = 0; it < UF_CAP; ++it) {
        a = uf_find(parent, a, ctrl);
        b = uf_find(parent, b, ctrl);
        if (a == b) return a;
        if (a < b) { int t = a; a = b; b = t; }
        // hook the larger root under the smaller one
        if (atomicCAS(parent + a, a, b) == a) return b;
    }
    set_error(ctrl, DBSCAN_ERR_INTERNAL);
    return min(a, b);
}

// ---- work units ------------------------------------------------------------
struct Sched {
    int nrt, nct, uc, kc;
    unsigned units, ubegin, uend;
};

__device__ __forceinline__ Sched make_sched(int n_rows, int n_cols, int tri, int ulo, int uhi) {
    Sched s;
    s.nrt = (n_rows + BT - 1) / BT;
    s.nct = (n_cols + BT - 1) / BT;
    long long total = tri ? (long long)s.nrt * (s.nrt + 1) / 2 : (long long)s.nrt * s.nct;
    long long target = 8LL * gridDim.x;
    long long uc = (total + target - 1) / target;
    if (uc < 1) uc = 1;
    if (uc > s.nct) uc = s.nct;
    s.uc = (int)uc;
    s.kc = (s.nct + s.uc - 1) / s.uc;
    s.units = (unsigned)((long long)s.nrt * s.kc);
    const long long g = gridDim.x;
    s.ubegin = (unsigned)min((long long)s.units, ulo * g);
    s.uend = uhi < 0 ? s.units : (unsigned)min((long long)s.units, uhi * g);
    return s;
}

// Unit u -> row tile rb and column tiles [t0, t1); false when empty.
__device__ __forceinline__ bool decode_unit(unsigned u, const Sched &s, int tri, int &rb,
                                            int &t0, int &t1) {
    rb = (int)(u / s.kc);
    int c = (int)(u % s.kc);
    t0 = tri ? rb + c * s.uc : c * s.uc;
    if (t0 >= s.nct) return false;
    t1 = min(t0 + s.uc, s.nct);
    return true;
}

// ---- per-row state and per-neighbour-pair actions --------------------------
// acc is the row's neighbour count (COUNT), an ancestor of the row point in
// the union-find (UNION), or its smallest neighbouring label (BORDER).
template <int MODE>
__device__ __forceinline__ void row_init(const SweepArgs &a, int p, int n_rows, int &acc) {
    if (MODE == SWEEP_COUNT) acc = 0;
    else if (MODE == SWEEP_UNION) acc = p < n_rows ? uf_find(a.parent, p, a.ctrl) : -1;
    else acc = 0x7fffffff;
}

// aux_q: the staged parent (UNION) or label (BORDER) of column point q.
// last (UNION): the staged parent the row was last joined with, which is in
// the row's set for good, so further neighbours staged with it are skipped.
template <int MODE>
__device__ __forceinline__ void on_neighbour(const SweepArgs &a, int p, int q, bool diag,
                                             int aux_q, int &acc, int &last) {
    if (MODE == SWEEP_COUNT) {
        if (diag && q < p) return;        // counted from the other side
        acc += 1;
        if (q != p) atomicAdd(a.cnt + q, 1);
    } else if (MODE == SWEEP_UNION) {
        if (diag && q <= p) return;
        if (aux_q == acc || aux_q == last) return;   // q's parent is in p's set
        last = aux_q;
        acc = uf_unite(a.parent, acc, aux_q, a.ctrl);
    } else {
        acc = min(acc, aux_q);
    }
}

template <int MODE>
__device__ __forceinline__ void flush_rows(const SweepArgs &a, int rb, int tr, int n_rows,
                                           const int (&acc)[R]) {
#pragma unroll
    for (int m = 0; m < R; ++m) {
        int p = rb * BT + slot_of(tr, m);
        if (p >= n_rows) continue;
        if (MODE == SWEEP_COUNT) {
            if (acc[m]) atomicAdd(a.cnt + p, acc[m]);
        } else if (MODE == SWEEP_BORDER) {
            if (acc[m] != 0x7fffffff) atomicMin(a.labels + a.candidx[p], acc[m]);
        }
    }
}

// Stage of up to tiles_per_stage tiles given by position, tile_of(j0 + q):
// the point tiles, then (with aux) as many x BT ints.
template <bool AUX, typename TileOf>
__device__ __forceinline__ void issue_tiles(float *dst, const SweepArgs &a, TileOf tile_of, int j0,
                                            int ntiles, int tile_floats, int tiles_per_stage) {
    int *adst = reinterpret_cast<int *>(dst + (size_t)tiles_per_stage * tile_floats);
    for (int q = 0; q < ntiles; ++q) {
        const int t = tile_of(j0 + q);
        const float *src = a.cols + (size_t)t * tile_floats;
        for (int c = threadIdx.x; c < tile_floats / 4; c += THREADS)
            cp_async16(dst + (size_t)q * tile_floats + 4 * c, src + 4 * c);
        if (AUX)
            for (int c = threadIdx.x; c < BT / 4; c += THREADS)
                cp_async16(adst + q * BT + 4 * c, a.aux + (size_t)t * BT + 4 * c);
    }
}

// ---- tile culling on CUDA cores ---------------------------------------------
// A column tile whose box is Ctrl::cull_thr or more (squared) from the row
// tile's box holds no pair the sweep's test accepts.  For integer data within
// the exactness bound that is the tensor-core producer's exact test (the gaps
// are integers, their squared sum exact, and cull_thr = thrx); for other data
// cull_thr is eps^2 plus a bound on the rounding of the sweep's float test and
// of the gap sum (prep.cu).  A unit's column tiles go KEEP_SPAN at a time:
// every thread tests one, and the kept ones are listed in ascending order in
// shared memory; only those are copied and evaluated.
constexpr int KEEP_SPAN = THREADS;

// The union sweep also skips the column tiles whose points all share the row
// tile's common root (rroot >= 0), a test that holds for any data.
// Kept tiles of [c0, c1) (c1 - c0 <= KEEP_SPAN) into s_list; returns their
// number.  Every thread of the block calls it.
__device__ __forceinline__ int keep_tiles(const SweepArgs &a, int d, int c0, int c1, bool box,
                                          const float *s_rbox, float thrx, int rroot, int *s_list,
                                          int *s_wtot) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int t = c0 + tid;
    bool keep = false;
    if (t < c1) {
        keep = !(rroot >= 0 && a.troot[t] == rroot);
        if (keep && box) {
            const float *bx = a.cbox + (size_t)t * 2 * d;
            float g2 = 0.f;
            for (int k = 0; k < d; ++k) {
                const float gp =
                    fmaxf(0.f, fmaxf(bx[2 * k] - s_rbox[2 * k + 1], s_rbox[2 * k] - bx[2 * k + 1]));
                g2 = fmaf(gp, gp, g2);
            }
            keep = g2 < thrx;
        }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_wtot[wid] = __popc(bal);
    __syncthreads();
    int base = 0, total = 0;
    for (int w = 0; w < THREADS / 32; ++w) {
        base += w < wid ? s_wtot[w] : 0;
        total += s_wtot[w];
    }
    if (keep) s_list[base + __popc(bal & ((1u << lane) - 1u))] = t;
    __syncthreads();
    return total;
}

// ===========================================================================
// d <= 4: rows in registers, packed f32x2 FMAs.
// ===========================================================================
// DIRECT: the direct form of the test (data off the exact path), else the
// expanded form (dbscan_internal.cuh); the kernels below pick one per call.
template <int D, int MODE, bool DIRECT>
__device__ __forceinline__ void sweep_small(const SweepArgs &a) {
    constexpr bool AUX = MODE != SWEEP_COUNT;
    constexpr float RSCALE = DIRECT ? -1.f : -2.f;   // the row's staged scale of c_i
    constexpr int TILE = (D + 1) * BT;
    constexpr int CT = 4;   // tiles per stage
    constexpr int S = 3;    // stages
    constexpr int STAGE = CT * TILE + (AUX ? CT * BT : 0);
    extern __shared__ __align__(16) float smem[];
    __shared__ unsigned s_unit;
    __shared__ int s_list[KEEP_SPAN], s_wtot[THREADS / 32];
    __shared__ float s_rbox[2 * D];

    if (a.ctrl->tc_kind != TC_NONE) return;   // the tensor-core sweep handles this data
    const int tid = threadIdx.x;
    const int tr = tid >> 4, tc = tid & 15;
    const int n_rows = *a.n_rows, n_cols = *a.n_cols;
    if (n_rows <= 0 || n_cols <= 0) return;
    const Sched sc = make_sched(n_rows, n_cols, a.tri, a.ulo, a.uhi);
    const bool cull = a.cull && a.rbox && a.cbox;
    const float thrx = a.ctrl->cull_thr;

    for (;;) {
        if (tid == 0) s_unit = sc.ubegin + atomicAdd(a.ctr, 1u) * (unsigned)a.sworld + (unsigned)a.srank;
        __syncthreads();
        const unsigned u = s_unit;
        __syncthreads();
        if (u >= sc.uend) break;
        int rb, t0, t1;
        if (!decode_unit(u, sc, a.tri, rb, t0, t1)) continue;
        if (a.band) {
            t0 = max(t0, rb + a.blo);
            if (a.bhi >= 0) t1 = min(t1, rb + a.bhi);
            if (t0 >= t1) continue;
        }
        const int rroot = a.troot ? a.troot[rb] : -1;
        const bool filt = cull || rroot >= 0;

        // rows of this unit: packed (A, A), A = -2c or -c, and thresholds
        float2 ra[R][D];
        float rT[R];
        {
            const float *rt = a.rows + (size_t)rb * TILE;
#pragma unroll
            for (int k = 0; k < D; ++k) {
                float4 lo = *reinterpret_cast<const float4 *>(rt + k * BT + 4 * tr);
                float4 hi = *reinterpret_cast<const float4 *>(rt + k * BT + 64 + 4 * tr);
                float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                for (int m = 0; m < R; ++m) ra[m][k] = make_float2(RSCALE * v[m], RSCALE * v[m]);
            }
            const float *tt = a.rowT + (size_t)rb * BT;
            float4 lo = *reinterpret_cast<const float4 *>(tt + 4 * tr);
            float4 hi = *reinterpret_cast<const float4 *>(tt + 64 + 4 * tr);
            rT[0] = lo.x; rT[1] = lo.y; rT[2] = lo.z; rT[3] = lo.w;
            rT[4] = hi.x; rT[5] = hi.y; rT[6] = hi.z; rT[7] = hi.w;
        }
        int acc[R], last[R];
#pragma unroll
        for (int m = 0; m < R; ++m) {
            row_init<MODE>(a, rb * BT + slot_of(tr, m), n_rows, acc[m]);
            last[m] = -1;
        }
        if (cull) {
            for (int e = tid; e < 2 * D; e += THREADS) s_rbox[e] = a.rbox[(size_t)rb * 2 * D + e];
            __syncthreads();
        }

      // column tiles in spans: all of [t0, t1) at once, or KEEP_SPAN at a time
      // listing the kept ones when tiles are skipped
      for (int c0 = t0; c0 < t1; c0 = filt ? c0 + KEEP_SPAN : t1) {
        const int c1 = filt ? min(c0 + KEEP_SPAN, t1) : t1;
        const int nk = filt ? keep_tiles(a, D, c0, c1, cull, s_rbox, thrx, rroot, s_list, s_wtot)
                            : c1 - c0;
        auto tile_of = [&](int j) { return filt ? s_list[j] : c0 + j; };
        const int nst = (nk + CT - 1) / CT;
#pragma unroll
        for (int s = 0; s < S - 1; ++s) {
            if (s < nst) issue_tiles<AUX>(smem + s * STAGE, a, tile_of, s * CT, min(CT, nk - s * CT), TILE, CT);
            cp_async_commit();
        }
        for (int g = 0; g < nst; ++g) {
            cp_async_wait<S - 2>();
            __syncthreads();
            {
                int gn = g + S - 1;
                if (gn < nst)
                    issue_tiles<AUX>(smem + (gn % S) * STAGE, a, tile_of, gn * CT, min(CT, nk - gn * CT), TILE, CT);
                cp_async_commit();
            }
            const float *sb = smem + (g % S) * STAGE;
            const int *saux = reinterpret_cast<const int *>(sb + CT * TILE);
            const int ntile = min(CT, nk - g * CT);
            for (int q = 0; q < ntile; ++q) {
                const int tile = tile_of(g * CT + q);
                const float *st = sb + q * TILE;
                float xc[D + 1][C];
#pragma unroll
                for (int k = 0; k <= D; ++k) {
                    float4 lo = *reinterpret_cast<const float4 *>(st + k * BT + 4 * tc);
                    float4 hi = *reinterpret_cast<const float4 *>(st + k * BT + 64 + 4 * tc);
                    xc[k][0] = lo.x; xc[k][1] = lo.y; xc[k][2] = lo.z; xc[k][3] = lo.w;
                    xc[k][4] = hi.x; xc[k][5] = hi.y; xc[k][6] = hi.z; xc[k][7] = hi.w;
                }
                unsigned hit = 0;
#pragma unroll
                for (int m = 0; m < R; ++m) {
                    float2 v[C / 2];
#pragma unroll
                    for (int p2 = 0; p2 < C / 2; ++p2) {
                        float2 t = make_float2(xc[D][2 * p2], xc[D][2 * p2 + 1]);
#pragma unroll
                        for (int k = 0; k < D; ++k) {
                            const float2 x = make_float2(xc[k][2 * p2], xc[k][2 * p2 + 1]);
                            if (DIRECT) {
                                const float2 q = __fadd2_rn(x, ra[m][k]);
                                t = __ffma2_rn(q, q, t);
                            } else {
                                t = __ffma2_rn(ra[m][k], x, t);
                            }
                        }
                        v[p2] = t;
                    }
                    float mn = min3f(min3f(v[0].x, v[0].y, v[1].x), min3f(v[1].y, v[2].x, v[2].y),
                                     fminf(v[3].x, v[3].y));
                    hit |= (mn < rT[m]) ? (1u << m) : 0u;
                }
                if (hit) {
                    const bool diag = a.tri && tile == rb;
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        if (!((hit >> m) & 1u)) continue;
                        const int p = rb * BT + slot_of(tr, m);
#pragma unroll
                        for (int c = 0; c < C; ++c) {
                            float v = xc[D][c];
#pragma unroll
                            for (int k = 0; k < D; ++k) {
                                if (DIRECT) {
                                    const float q = xc[k][c] + ra[m][k].x;
                                    v = fmaf(q, q, v);
                                } else {
                                    v = fmaf(ra[m][k].x, xc[k][c], v);
                                }
                            }
                            if (v < rT[m]) {
                                const int slot = slot_of(tc, c);
                                on_neighbour<MODE>(a, p, tile * BT + slot, diag,
                                                   AUX ? saux[q * BT + slot] : 0, acc[m], last[m]);
                            }
                        }
                    }
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();   // every thread is done with the stages and the list
      }
        flush_rows<MODE>(a, rb, tr, n_rows, acc);
    }
}

// One kernel per form (both are launched; the one the data did not select
// returns at once): a kernel holding both bodies spilled registers in the
// expanded count (1M x 3 FFMA count 73.3 -> 74.2 ms).
template <int D, int MODE, bool DIRECT>
__global__ void __launch_bounds__(THREADS, 2) k_sweep_small(SweepArgs a) {
    if ((a.ctrl->exact == 0) != DIRECT) return;
    sweep_small<D, MODE, DIRECT>(a);
}

// ===========================================================================
// d > 4: rows and columns from shared memory, 8x8 register accumulators.
// S = 1 (d > 128, where a row tile and two column stages exceed shared
// memory): one column stage, loaded and used in turn, and the row values read
// from the staged row tile in global memory (L2-resident).
// ===========================================================================
template <int MODE, int S, bool DIRECT>
__device__ __forceinline__ void sweep_gen(const SweepArgs &a, int D) {
    constexpr bool AUX = MODE != SWEEP_COUNT;
    constexpr float RSCALE = DIRECT ? -1.f : -2.f;   // the row's staged scale of c_i
    constexpr bool ROWS_GLOBAL = S == 1;
    extern __shared__ __align__(16) float smem[];
    __shared__ unsigned s_unit;
    const int TILE = (D + 1) * BT;
    const int STAGE = TILE + (AUX ? BT : 0);
    float *rowbuf = smem;                                 // D * BT floats: A of the row tile
    float *stages = smem + (ROWS_GLOBAL ? 0 : D * BT);    // S * STAGE floats
    __shared__ int s_list[KEEP_SPAN], s_wtot[THREADS / 32];
    __shared__ float s_rbox[2 * CULL_MAX_D];

    if (a.ctrl->tc_kind != TC_NONE) return;   // the tensor-core sweep handles this data
    const int tid = threadIdx.x;
    const int tr = tid >> 4, tc = tid & 15;
    const int n_rows = *a.n_rows, n_cols = *a.n_cols;
    if (n_rows <= 0 || n_cols <= 0) return;
    const Sched sc = make_sched(n_rows, n_cols, a.tri, a.ulo, a.uhi);
    const bool cull = a.cull && a.rbox && a.cbox && D <= CULL_MAX_D;
    const float thrx = a.ctrl->cull_thr;

    for (;;) {
        if (tid == 0) s_unit = sc.ubegin + atomicAdd(a.ctr, 1u) * (unsigned)a.sworld + (unsigned)a.srank;
        __syncthreads();
        const unsigned u = s_unit;
        __syncthreads();
        if (u >= sc.uend) break;
        int rb, t0, t1;
        if (!decode_unit(u, sc, a.tri, rb, t0, t1)) continue;
        if (a.band) {
            t0 = max(t0, rb + a.blo);
            if (a.bhi >= 0) t1 = min(t1, rb + a.bhi);
            if (t0 >= t1) continue;
        }
        const int rroot = a.troot ? a.troot[rb] : -1;
        const bool filt = cull || rroot >= 0;

        const float *rowsrc = ROWS_GLOBAL ? a.rows + (size_t)rb * TILE : rowbuf;
        const float rscale = ROWS_GLOBAL ? RSCALE : 1.f;
        if (!ROWS_GLOBAL) {
            const float *rt = a.rows + (size_t)rb * TILE;
            for (int e = tid; e < D * BT; e += THREADS) rowbuf[e] = RSCALE * rt[e];
        }
        float rT[R];
        {
            const float *tt = a.rowT + (size_t)rb * BT;
            float4 lo = *reinterpret_cast<const float4 *>(tt + 4 * tr);
            float4 hi = *reinterpret_cast<const float4 *>(tt + 64 + 4 * tr);
            rT[0] = lo.x; rT[1] = lo.y; rT[2] = lo.z; rT[3] = lo.w;
            rT[4] = hi.x; rT[5] = hi.y; rT[6] = hi.z; rT[7] = hi.w;
        }
        int acc[R], last[R];
#pragma unroll
        for (int m = 0; m < R; ++m) {
            row_init<MODE>(a, rb * BT + slot_of(tr, m), n_rows, acc[m]);
            last[m] = -1;
        }
        if (cull) {
            for (int e = tid; e < 2 * D; e += THREADS) s_rbox[e] = a.rbox[(size_t)rb * 2 * D + e];
            __syncthreads();
        }

      // column tiles in spans: all of [t0, t1) at once, or KEEP_SPAN at a time
      // listing the kept ones when tiles are skipped
      for (int c0 = t0; c0 < t1; c0 = filt ? c0 + KEEP_SPAN : t1) {
        const int c1 = filt ? min(c0 + KEEP_SPAN, t1) : t1;
        const int nk = filt ? keep_tiles(a, D, c0, c1, cull, s_rbox, thrx, rroot, s_list, s_wtot)
                            : c1 - c0;
        auto tile_of = [&](int j) { return filt ? s_list[j] : c0 + j; };
        const int nst = nk;   // one tile per stage
        if constexpr (S > 1) {
#pragma unroll
            for (int s = 0; s < S - 1; ++s) {
                if (s < nst) issue_tiles<AUX>(stages + s * STAGE, a, tile_of, s, 1, TILE, 1);
                cp_async_commit();
            }
        }
        for (int g = 0; g < nst; ++g) {
            if constexpr (S > 1) {
                cp_async_wait<S - 2>();
                __syncthreads();
                int gn = g + S - 1;
                if (gn < nst) issue_tiles<AUX>(stages + (gn % S) * STAGE, a, tile_of, gn, 1, TILE, 1);
                cp_async_commit();
            } else {
                __syncthreads();   // every thread is done with the previous tile
                issue_tiles<AUX>(stages, a, tile_of, g, 1, TILE, 1);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
            }
            const int tile = tile_of(g);
            const float *st = stages + (g % S) * STAGE;
            const int *saux = reinterpret_cast<const int *>(st + TILE);
            float v[R][C];
            {
                float4 lo = *reinterpret_cast<const float4 *>(st + D * BT + 4 * tc);
                float4 hi = *reinterpret_cast<const float4 *>(st + D * BT + 64 + 4 * tc);
                float nn[C] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                for (int m = 0; m < R; ++m)
#pragma unroll
                    for (int c = 0; c < C; ++c) v[m][c] = nn[c];
            }
#pragma unroll 2
            for (int k = 0; k < D; ++k) {
                const float4 rlo = *reinterpret_cast<const float4 *>(rowsrc + k * BT + 4 * tr);
                const float4 rhi = *reinterpret_cast<const float4 *>(rowsrc + k * BT + 64 + 4 * tr);
                float4 xlo = *reinterpret_cast<const float4 *>(st + k * BT + 4 * tc);
                float4 xhi = *reinterpret_cast<const float4 *>(st + k * BT + 64 + 4 * tc);
                float rr[R] = {rscale * rlo.x, rscale * rlo.y, rscale * rlo.z, rscale * rlo.w,
                               rscale * rhi.x, rscale * rhi.y, rscale * rhi.z, rscale * rhi.w};
                float xx[C] = {xlo.x, xlo.y, xlo.z, xlo.w, xhi.x, xhi.y, xhi.z, xhi.w};
#pragma unroll
                for (int m = 0; m < R; ++m)
#pragma unroll
                    for (int c = 0; c < C; ++c) {
                        if (DIRECT) {
                            const float q = xx[c] + rr[m];
                            v[m][c] = fmaf(q, q, v[m][c]);
                        } else {
                            v[m][c] = fmaf(rr[m], xx[c], v[m][c]);
                        }
                    }
            }
            unsigned hit = 0;
#pragma unroll
            for (int m = 0; m < R; ++m) {
                float mn = min3f(min3f(v[m][0], v[m][1], v[m][2]), min3f(v[m][3], v[m][4], v[m][5]),
                                 fminf(v[m][6], v[m][7]));
                hit |= (mn < rT[m]) ? (1u << m) : 0u;
            }
            if (hit) {
                const bool diag = a.tri && tile == rb;
#pragma unroll
                for (int m = 0; m < R; ++m) {
                    if (!((hit >> m) & 1u)) continue;
                    const int p = rb * BT + slot_of(tr, m);
#pragma unroll
                    for (int c = 0; c < C; ++c)
                        if (v[m][c] < rT[m]) {
                            const int slot = slot_of(tc, c);
                            on_neighbour<MODE>(a, p, tile * BT + slot, diag, AUX ? saux[slot] : 0,
                                               acc[m], last[m]);
                        }
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();   // every thread is done with the stages and the list
      }
        flush_rows<MODE>(a, rb, tr, n_rows, acc);
    }
}

template <int MODE, int S, bool DIRECT>
__global__ void __launch_bounds__(THREADS, 2) k_sweep_gen(SweepArgs a, int D) {
    if ((a.ctrl->exact == 0) != DIRECT) return;
    sweep_gen<MODE, S, DIRECT>(a, D);
}

// ---- tile-local union before the core-core sweep -------------------------------
// With the points in locality order most core-core neighbour pairs fall inside
// a diagonal tile.  One CTA per core tile joins the tile's own neighbour pairs
// in a shared-memory union-find and points every position at the smallest
// position of its tile-local component, so that the sweep's staged parent
// snapshots already carry those roots and the sweep skips such pairs without
// touching global memory.  Same hit test as the sweep (v_ij < T_i).
// Find with path halving: parents only ever move towards the root, so a
// racing write of a grandparent is always a valid ancestor.
__device__ __forceinline__ int sm_find(volatile int *sp, int x) {
    for (int it = 0; it < BT; ++it) {
        const int p = sp[x];
        if (p == x) break;
        const int gp = sp[p];
        if (gp != p) sp[x] = gp;
        x = gp;
    }
    return x;
}

// DMAX > 0 (d <= DMAX): the thread's own point, scaled by -2, sits in
// registers, so every FMA reads one shared-memory word instead of two (the
// products and their order are those of the generic form).
template <int DMAX, bool DIRECT>
__device__ __forceinline__ void local_union(const Ctrl *ctrl, const float *staged, const float *T,
                                            int d, int *parent) {
    constexpr float RSCALE = DIRECT ? -1.f : -2.f;   // the row's staged scale of c_i
    extern __shared__ float s_pts[];   // (d + 1) * BT staged floats, then BT parents
    volatile int *sp = reinterpret_cast<volatile int *>(s_pts + (size_t)(d + 1) * BT);
    const int n_core = ctrl->n_core;
    const int ntiles = (n_core + BT - 1) / BT;
    const int i = threadIdx.x;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int base = t * BT;
        const int nv = min(BT, n_core - base);
        __syncthreads();
        const float *src = staged + (size_t)t * (size_t)(d + 1) * BT;
        for (int e = i; e < (d + 1) * BT; e += BT) s_pts[e] = src[e];
        sp[i] = i;
        __syncthreads();
        if (i < nv) {
            const float Ti = T[base + i];
            float ri[DMAX > 0 ? DMAX : 1];
            if constexpr (DMAX > 0) {
#pragma unroll
                for (int k = 0; k < DMAX; ++k) ri[k] = k < d ? RSCALE * s_pts[(size_t)k * BT + i] : 0.f;
            }
            // pairs (i, i + sh mod BT), sh = 1..63, and sh = 64 for i < 64: every
            // unordered pair of the tile once, 63 or 64 per thread
            const int shmax = i < BT / 2 ? BT / 2 : BT / 2 - 1;
            for (int sh = 1; sh <= shmax; ++sh) {
                const int j = (i + sh) & (BT - 1);
                if (j >= nv) continue;
                float v = s_pts[(size_t)d * BT + j];
                if constexpr (DMAX > 0) {
#pragma unroll
                    for (int k = 0; k < DMAX; ++k)
                        if (k < d) {
                            if (DIRECT) {
                                const float q = s_pts[(size_t)k * BT + j] + ri[k];
                                v = fmaf(q, q, v);
                            } else {
                                v = fmaf(ri[k], s_pts[(size_t)k * BT + j], v);
                            }
                        }
                } else {
                    for (int k = 0; k < d; ++k) {
                        if (DIRECT) {
                            const float q = s_pts[(size_t)k * BT + j] + RSCALE * s_pts[(size_t)k * BT + i];
                            v = fmaf(q, q, v);
                        } else {
                            v = fmaf(RSCALE * s_pts[(size_t)k * BT + i], s_pts[(size_t)k * BT + j], v);
                        }
                    }
                }
                if (!(v < Ti)) continue;
                int ra = i, rb = j;
                for (int it = 0; it < 2 * BT; ++it) {
                    ra = sm_find(sp, ra);
                    rb = sm_find(sp, rb);
                    if (ra == rb) break;
                    if (ra < rb) { const int tmp = ra; ra = rb; rb = tmp; }
                    if (atomicCAS((int *)&sp[ra], ra, rb) == ra) break;
                }
            }
        }
        __syncthreads();
        if (i < nv) parent[base + i] = base + sm_find(sp, i);
    }
}

template <int DMAX>
__global__ void k_local_union(const Ctrl *ctrl, const float *staged, const float *T, int d,
                              int *parent) {
    if (ctrl->exact) local_union<DMAX, false>(ctrl, staged, T, d, parent);
    else local_union<DMAX, true>(ctrl, staged, T, d, parent);
}

// Point every core position straight at its root (between union bands);
// tc = 1 runs only on the tensor-core path, tc = 0 only on the CUDA-core path.
__global__ void k_compress(Ctrl *ctrl, int *parent, int tc) {
    if ((ctrl->tc_kind != TC_NONE) != (tc != 0)) return;
    const int n_core = ctrl->n_core;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_core; p += gridDim.x * blockDim.x) {
        int r = uf_find(parent, p, ctrl);
        if (__ldcg(parent + p) != r) __stcg(parent + p, r);
    }
}

// Common root of each core tile's points, or -1 when they are not all in one
// set (tensor-core path, after k_compress: every parent is then a root).  A
// union tile pair whose row and column tiles share one common root holds no
// pair the union could still join, and the sweep skips it; sets only merge,
// so a snapshot taken before a band stays safe through it.
__global__ void k_tile_roots(const Ctrl *ctrl, const int *parent, int *troot, int tc) {
    if ((ctrl->tc_kind != TC_NONE) != (tc != 0)) return;
    const int n_core = ctrl->n_core;
    const int nt = (n_core + BT - 1) / BT;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < nt; t += gridDim.x * wpb) {
        int mn = 0x7fffffff, mx = -1;
        for (int j = lane; j < BT; j += 32) {
            const int p = t * BT + j;
            if (p < n_core) {
                const int r = __ldcg(parent + p);
                mn = min(mn, r);
                mx = max(mx, r);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        if (lane == 0) troot[t] = mn == mx ? mn : -1;
    }
}

// ===========================================================================
// host side
// ===========================================================================
int persistent_ctas(const void *kernel, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_pair(dev, kernel);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int sms = 0, per = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, threads, smem);
    if (per < 1) per = 1;
    if (sms < 1) sms = 1;
    int v = sms * per;
    cache[key] = v;
    return v;
}

template <int D, int MODE, bool DIRECT>
static cudaError_t run_small_form(const SweepArgs &args, cudaStream_t s) {
    auto kernel = k_sweep_small<D, MODE, DIRECT>;
    const int aux = MODE != SWEEP_COUNT ? 4 * BT : 0;
    const size_t smem = (size_t)3 * (4 * (D + 1) * BT + aux) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute((const void *)kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = persistent_ctas((const void *)kernel, THREADS, smem);
    kernel<<<grid, THREADS, smem, s>>>(args);
    return cudaGetLastError();
}

template <int MODE, int S, bool DIRECT>
static cudaError_t run_gen_form(const SweepArgs &args, int d, cudaStream_t s) {
    auto kernel = k_sweep_gen<MODE, S, DIRECT>;
    const int aux = MODE != SWEEP_COUNT ? BT : 0;
    const size_t smem = ((S == 1 ? 0 : (size_t)d * BT) + (size_t)S * ((d + 1) * BT + aux)) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute((const void *)kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = persistent_ctas((const void *)kernel, THREADS, smem);
    kernel<<<grid, THREADS, smem, s>>>(args, d);
    return cudaGetLastError();
}

template <int D, int MODE>
static cudaError_t run_small(const SweepArgs &args, cudaStream_t s) {
    cudaError_t e = run_small_form<D, MODE, false>(args, s);
    return e != cudaSuccess ? e : run_small_form<D, MODE, true>(args, s);
}

template <int MODE, int S>
static cudaError_t run_gen(const SweepArgs &args, int d, cudaStream_t s) {
    cudaError_t e = run_gen_form<MODE, S, false>(args, d, s);
    return e != cudaSuccess ? e : run_gen_form<MODE, S, true>(args, d, s);
}

template <int MODE>
static cudaError_t dispatch(const SweepArgs &args, int d, cudaStream_t s) {
    switch (d) {
    case 1: return run_small<1, MODE>(args, s);
    case 2: return run_small<2, MODE>(args, s);
    case 3: return run_small<3, MODE>(args, s);
    case 4: return run_small<4, MODE>(args, s);
    default:
        // shared memory: a row tile and S column stages of (d + 1) x 128 floats
        return d <= 32 ? run_gen<MODE, 3>(args, d, s)
                       : (d <= 128 ? run_gen<MODE, 2>(args, d, s) : run_gen<MODE, 1>(args, d, s));
    }
}

cudaError_t launch_count(const Work &w, const Layout &L, cudaStream_t s) {
    SweepArgs a{};
    a.srank = L.rank; a.sworld = L.world;
    a.rows = w.staged_all; a.rowT = w.T_all; a.n_rows = &w.ctrl->n_all;
    a.cols = w.staged_all; a.n_cols = &w.ctrl->n_all;
    a.tri = 1; a.ulo = 0; a.uhi = -1;
    a.ctr = &w.ctrl->unit_ctr[CTR_COUNT]; a.ctrl = w.ctrl; a.cnt = w.cnt;
    a.rbox = w.box_all; a.cbox = w.box_all; a.cull = L.cull;
    cudaError_t e = dispatch<SWEEP_COUNT>(a, L.d, s);
    if (e != cudaSuccess) return e;
    return launch_count_tc(w, L, s);
}

// Tensor-core union bands of a call: the three of tc_schedule.h, or for at
// most ONE_BAND_MAX_TILES tiles a single band (every tile distance from 1):
// every band costs a compression, a tile-root snapshot and the sweep's
// start-up, and with few tiles a band holds too little work to repay them
// (100k x 2 union 0.44 -> 0.38 ms).  The CUDA-core union keeps three bands:
// its sweeps gain more from the compressions between them (forced onto CUDA
// cores, 100k x 2 union 1.37 -> 1.80 ms with one band).
#ifndef ONE_BAND_MAX_TILES
#define ONE_BAND_MAX_TILES 2048
#endif
int union_band_count(int64_t ntiles) { return ntiles <= ONE_BAND_MAX_TILES ? 1 : UNION_BANDS; }
static void union_band(int64_t ntiles, int bd, int &lo, int &hi) {
    if (union_band_count(ntiles) == 1) {
        lo = 1;
        hi = -1;
    } else {
        lo = kUnionBandEdges[bd];
        hi = kUnionBandEdges[bd + 1];
    }
}

cudaError_t launch_union(const Work &w, const Layout &L, cudaStream_t s) {
    SweepArgs a{};
    a.srank = L.rank; a.sworld = L.world;
    a.rows = w.staged_core; a.rowT = w.T_core; a.n_rows = &w.ctrl->n_core;
    a.cols = w.staged_core; a.n_cols = &w.ctrl->n_core; a.aux = w.parent;
    a.tri = 1; a.ctrl = w.ctrl; a.parent = w.parent;
    a.rbox = w.box_core; a.cbox = w.box_core; a.cull = L.cull_nbr;
    const int grid = persistent_ctas((const void *)k_compress, 256, 0);
    const size_t lsmem = (size_t)(L.d + 1) * BT * sizeof(float) + BT * sizeof(int);
    auto local = L.d <= 4 ? k_local_union<4>
                          : (L.d <= 16 ? k_local_union<16> : (L.d <= 64 ? k_local_union<64> : k_local_union<0>));
    if (cudaFuncSetAttribute((const void *)local,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lsmem) != cudaSuccess)
        return cudaGetLastError();
    int dev = 0, sms = 1, per = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, (const void *)local, BT, lsmem);
    int64_t lgrid = (int64_t)sms * (per < 1 ? 1 : per);
    if (lgrid > L.ntiles) lgrid = L.ntiles;
    if (lgrid < 1) lgrid = 1;
    local<<<(unsigned)lgrid, BT, lsmem, s>>>(w.ctrl, w.staged_core, w.T_core, L.d, w.parent);
    // Both paths go by bands of tile distance from the diagonal, nearest
    // first, compressed between bands: in locality order most neighbour pairs
    // lie near the diagonal, so the far bands find merged roots in their
    // staged parent snapshots and skip their pairs without a global access.
    // Each band also skips the tile pairs whose tiles share one root (a
    // snapshot per band, k_tile_roots; the tile-local union leaves every
    // parent a root, so the first snapshot needs no compression).  The
    // kernels of the path not taken return at once.
    const unsigned rgrid = (unsigned)((L.ntiles + 7) / 8);
    // CUDA-core path
    a.ulo = 0; a.uhi = -1;
    a.band = 1; a.troot = w.troot;
    for (int bd = 0; bd < UNION_BANDS; ++bd) {
        cudaError_t e;
        if (bd > 0) {
            k_compress<<<grid, 256, 0, s>>>(w.ctrl, w.parent, 0);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        k_tile_roots<<<rgrid, 256, 0, s>>>(w.ctrl, w.parent, w.troot, 0);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        a.blo = kUnionBandEdges[bd];
        a.bhi = kUnionBandEdges[bd + 1];
        a.ctr = &w.ctrl->unit_ctr[CTR_UNION0 + bd];
        if ((e = dispatch<SWEEP_UNION>(a, L.d, s)) != cudaSuccess) return e;
    }
    // tensor-core path
    const int nbands = union_band_count(L.ntiles);
    for (int bd = 0; bd < nbands; ++bd) {
        cudaError_t e;
        if (bd > 0) {
            k_compress<<<grid, 256, 0, s>>>(w.ctrl, w.parent, 1);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        k_tile_roots<<<rgrid, 256, 0, s>>>(w.ctrl, w.parent, w.troot, 1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        int lo, hi;
        union_band(L.ntiles, bd, lo, hi);
        e = launch_union_tc_band(w, L, bd, lo, hi, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Sharding: every rank's union-find forest links core positions of one
// component (each link is a neighbour pair or a chain of them), so uniting
// every core position i with every rank's parent of i joins exactly the union
// of the neighbour pairs all ranks evaluated.
__global__ void k_merge_forests(Ctrl *ctrl, int *parent, const int *gathered, int64_t stride,
                                int world) {
    const int nc = ctrl->n_core;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nc; i += gridDim.x * blockDim.x) {
        for (int r = 0; r < world; ++r) {
            const int p = gathered[(size_t)r * stride + i];
            if (p != i && p >= 0 && p < nc) uf_unite(parent, i, p, ctrl);
        }
    }
}

cudaError_t launch_merge_forests(const Work &w, const Layout &L, const int *gathered, int64_t stride,
                                 int world, cudaStream_t s) {
    const int grid = persistent_ctas((const void *)k_compress, 256, 0);
    k_merge_forests<<<grid, 256, 0, s>>>(w.ctrl, w.parent, gathered, stride, world);
    return cudaGetLastError();   // k_flatten follows every position to its root
}

cudaError_t launch_border(const Work &w, const Layout &L, int32_t *labels, cudaStream_t s) {
    SweepArgs a{};
    a.srank = L.rank; a.sworld = L.world;
    a.rows = w.staged_cand; a.rowT = w.T_cand; a.n_rows = &w.ctrl->n_cand;
    a.cols = w.staged_core; a.n_cols = &w.ctrl->n_core; a.aux = w.clabel;
    a.tri = 0; a.ulo = 0; a.uhi = -1;
    a.ctr = &w.ctrl->unit_ctr[CTR_BORDER]; a.ctrl = w.ctrl;
    a.candidx = w.candidx; a.labels = labels;
    a.rbox = w.box_cand; a.cbox = w.box_core; a.cull = L.cull_nbr;
    cudaError_t e = dispatch<SWEEP_BORDER>(a, L.d, s);
    if (e != cudaSuccess) return e;
    return launch_border_tc(w, L, labels, s);
}

}  // namespace dbscan
