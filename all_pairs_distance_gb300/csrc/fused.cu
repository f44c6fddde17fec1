// Fused small-problem pipeline: every stage of the DBSCAN path in ONE
// persistent, cooperative launch with grid-wide phases.
//
// "Design and optimization of DBSCAN Algorithm based on CUDA", §IV-B1, fuses
// the distance evaluation with building the primitive clusters so that one
// kernel does both.  For small problems the multi-kernel path is bound by its
// ~60 launches (a tensor-core sweep costs ~14 us even with almost no work), so
// here the fusion is carried through the whole path: statistics, centring,
// counting, core flags, the union-find merge (§IV-C), flattening and border
// assignment run as phases of one kernel, separated by a grid-wide barrier.
// Points stay in input order (no locality order), so cluster names come out
// directly as the smallest core input index: the union-find hooks the larger
// root under the smaller one, so a component's root is its smallest member.
//
// Phases (B = grid-wide barrier):
//   stats      per-dimension min/max, integer and finiteness flags        B
//   stage      centre, threshold constant (every block, from the stats),
//              centred coordinates, squared norms, row thresholds,
//              per-tile counters cleared                                   B
//   count      upper triangle of 128 x 128 tile pairs, each pair credited
//              to both points (row count in a register, column counts in
//              shared memory)                                              B
//   core       core flags, union-find init, per-tile core counts, the list
//              of border candidates                                        B
//   union      every core-core neighbour pair of the upper triangle hooks
//              the larger index under the smaller (atomicMin), B, parents
//              compressed to roots, B, then a lock-free union-find (CAS of
//              the larger root) over the same pairs, skipping pairs already
//              joined by a shared-memory snapshot of the roots             B
//   flatten    labels of core points = their root; candidates get a
//              sentinel, other non-core points -1                          B
//   border     candidate list x core tiles, smallest neighbouring label
//              by atomicMin                                                B
//   finalize   candidates without a core neighbour become noise
//
// Arithmetic is that of the CUDA-core sweeps: fp32 FMAs on centred
// coordinates, v_ij = nrm_j + sum_k (-2 c_ik) c_jk tested against
// T_i = thrx - nrm_i, exact for integer data while sum_k range_k^2 < 2^24,
// and for other data the direct form v_ij = sum_k (c_jk - c_ik)^2 against
// the common threshold (dbscan_internal.cuh).
// Every barrier wait is bounded; on timeout the kernel records
// DBSCAN_ERR_INTERNAL and every block leaves at its next barrier.
#include "dbscan_internal.cuh"

#include <math.h>

namespace dbscan {
namespace {

constexpr int FT = BT;                 // points per tile = threads per block
constexpr long long F_WAIT = 4000000000LL;   // clock cycles (about 2 s)
constexpr int F_UF_CAP = 1 << 22;

struct FusedArgs {
    const void *pts;
    int dtype, n, d, min_pts, ntiles;
    float eps2;
    Ctrl *ctrl;
    unsigned *smin, *smax;   // per dimension: max of ~u and of u (u: ordered key), zeroed
    float *staged, *T;
    int *cnt, *parent, *clabel, *tcore, *candlist;
    int32_t *labels;
    uint8_t *is_core;
    int32_t *cnt_out;        // counts only: the counts in input order, then stop
};

// ---- grid-wide barrier (all blocks co-resident: cooperative launch) --------
// Sense by generation: read the generation, arrive; the last block to arrive
// resets the count and advances the generation; the others wait for it.
__device__ bool grid_sync(Ctrl *ctrl, unsigned nblocks) {
    volatile unsigned *gen = &ctrl->bar_gen;
    unsigned *count = &ctrl->bar_count;
    volatile int *abort_flag = &ctrl->bar_abort;
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = *abort_flag == 0;
        if (ok) {
            const unsigned g = *gen;
            __threadfence();
            if (atomicAdd(count, 1u) == nblocks - 1) {
                *count = 0;
                __threadfence();
                atomicAdd(const_cast<unsigned *>(gen), 1u);
            } else {
                const long long t0 = clock64();
                while (*gen == g) {
                    if (*abort_flag) { ok = 0; break; }
                    if (clock64() - t0 > F_WAIT) {
                        set_error(ctrl, DBSCAN_ERR_INTERNAL);
                        *abort_flag = 1;
                        ok = 0;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            __threadfence();
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// ---- union-find: parent[x] <= x always, roots are component minima --------
__device__ int f_find(int *parent, int x, Ctrl *ctrl) {
    for (int it = 0; it < F_UF_CAP; ++it) {
        const int p = __ldcg(parent + x);
        if (p == x) return x;
        const int gp = __ldcg(parent + p);
        if (gp != p) __stcg(parent + x, gp);   // path halving
        x = gp;
    }
    set_error(ctrl, DBSCAN_ERR_INTERNAL);
    return x;
}
// Merge the sets of a and b; returns their common root at the merge.
__device__ int f_unite(int *parent, int a, int b, Ctrl *ctrl) {
    for (int it = 0; it < F_UF_CAP; ++it) {
        a = f_find(parent, a, ctrl);
        b = f_find(parent, b, ctrl);
        if (a == b) return a;
        if (a < b) { const int t = a; a = b; b = t; }
        if (atomicCAS(parent + a, a, b) == a) return b;
    }
    set_error(ctrl, DBSCAN_ERR_INTERNAL);
    return min(a, b);
}

// Upper-triangle tile pair u -> (rb, cb), rb <= cb, row by row: row r holds
// nt - r pairs and S(r) = r nt - r (r - 1) / 2 pairs precede it.
__device__ __forceinline__ void tri_pair(int u, int nt, int &rb, int &cb) {
    auto S = [nt](int r) { return r * nt - r * (r - 1) / 2; };
    const float b = 2.f * nt + 1.f;
    int r = (int)floorf((b - sqrtf(fmaxf(b * b - 8.f * (float)u, 0.f))) * 0.5f);
    r = min(max(r, 0), nt - 1);
    while (r > 0 && S(r) > u) --r;
    while (r + 1 < nt && S(r + 1) <= u) ++r;
    rb = r;
    cb = r + (u - S(r));
}

// Row thread state: A = -2 c_i (expanded form) or -c_i (direct form) in
// registers (D > 0) or in shared memory (D = 0).
template <int D>
struct RowPoint {
    float a[D > 0 ? D : 1];
};

// One term of v_ij: a_k c_jk (expanded) or (c_jk + a_k)^2 (direct).
__device__ __forceinline__ float pair_term(bool direct, float ak, float ck, float v) {
    if (direct) {
        const float q = ck + ak;
        return fmaf(q, q, v);
    }
    return fmaf(ak, ck, v);
}

// v_ij = slot_j + the sum of the terms for column j of the staged column tile
// s (structure of arrays: (d + 1) x FT floats, the norm slots last).
template <int D>
__device__ __forceinline__ float pair_value(bool direct, const RowPoint<D> &r, const float *sa,
                                            const float *s, int d, int j) {
    if (D > 0) {
        float v = s[D * FT + j];
#pragma unroll
        for (int k = 0; k < D; ++k) v = pair_term(direct, r.a[k], s[k * FT + j], v);
        return v;
    }
    float v = s[d * FT + j];
    for (int k = 0; k < d; ++k) v = pair_term(direct, sa[k * FT + threadIdx.x], s[k * FT + j], v);
    return v;
}

template <int D>
__global__ void __launch_bounds__(FT) k_fused(FusedArgs a) {
    extern __shared__ float sm[];
    const int d = D > 0 ? D : a.d;
    const int n = a.n, nt = a.ntiles, tid = threadIdx.x;
    const unsigned nb = gridDim.x;
    Ctrl *ctrl = a.ctrl;
    float *s_col = sm;                            // (d + 1) x FT column tile
    float *s_row = sm + (size_t)(d + 1) * FT;     // D = 0: -2 c of the row tile, d x FT
    int *s_aux = reinterpret_cast<int *>(s_row + (D > 0 ? 0 : (size_t)d * FT));   // 2 x FT ints
    __shared__ float s_centre[DBSCAN_MAX_D];
    __shared__ float s_thrx;
    __shared__ int s_integral, s_direct;

    // ---- stats ----------------------------------------------------------------
    {
        // with a stride that is a multiple of d every thread stays on one
        // dimension; min and max go through the order-preserving unsigned key
        // u, the minimum as the maximum of ~u, so zero is the neutral value
        __shared__ unsigned bmin[DBSCAN_MAX_D], bmax[DBSCAN_MAX_D];
        for (int k = tid; k < d; k += FT) bmin[k] = bmax[k] = 0u;
        __syncthreads();
        int nonint = 0, nonfin = 0;
        const int64_t total = (int64_t)n * d;
        const int64_t stride = ((int64_t)nb * FT / d) * d;
        const int64_t t0 = (int64_t)blockIdx.x * FT + tid;
        unsigned umin = 0u, umax = 0u;
        if (t0 < stride) {
            for (int64_t e = t0; e < total; e += stride) {
                const float x = load_point(a.pts, a.dtype, (size_t)e);
                if (!isfinite(x)) { nonfin = 1; continue; }
                if (x != rintf(x)) nonint = 1;
                const unsigned u = (unsigned)float_key(x) ^ 0x80000000u;
                umin = max(umin, ~u);
                umax = max(umax, u);
            }
            if (umax) {
                atomicMax(&bmin[t0 % d], umin);
                atomicMax(&bmax[t0 % d], umax);
            }
        }
        if (__syncthreads_or(nonint) && tid == 0) atomicOr(&ctrl->nonint, 1);
        if (__syncthreads_or(nonfin) && tid == 0) atomicOr(&ctrl->nonfinite, 1);
        for (int k = tid; k < d; k += FT) {
            if (bmax[k]) {
                atomicMax(&a.smin[k], bmin[k]);
                atomicMax(&a.smax[k], bmax[k]);
            }
        }
    }
    if (!grid_sync(ctrl, nb)) return;

    // ---- stage: every block derives the centre and threshold from the stats -----
    if (tid == 0) s_integral = ctrl->nonint == 0;
    __syncthreads();
    const bool integral = s_integral != 0;
    for (int k = tid; k < d; k += FT) {
        float lo = 0.f, hi = 0.f;
        if (a.smax[k]) {   // some finite value in this dimension
            lo = key_float((int)(~a.smin[k] ^ 0x80000000u));
            hi = key_float((int)(a.smax[k] ^ 0x80000000u));
        }
        s_centre[k] = integral ? floorf(0.5f * lo + 0.5f * hi) : 0.5f * lo + 0.5f * hi;
        s_row[k] = (float)((double)hi - (double)lo);   // scratch: the ranges
    }
    __syncthreads();
    if (tid == 0) {
        double R = 0.0;
        for (int k = 0; k < d; ++k) R += (double)s_row[k] * (double)s_row[k];
        float thrx = a.eps2;
        if (integral) {
            double t = floor((double)a.eps2);
            if (t > R) t = R;
            thrx = (float)(t + 1.0);
        }
        s_thrx = thrx;
        s_direct = (integral && R < 16777215.0) ? 0 : 1;
        if (blockIdx.x == 0) {
            ctrl->n_all = n;
            ctrl->range_sq = (float)R;
            ctrl->thrx = thrx;
            ctrl->exact = (integral && R < 16777215.0) ? 1 : 0;
            ctrl->tc_kind = TC_NONE;
            ctrl->tc_kpad = 0;
            ctrl->tc_kbytes = 0;
            ctrl->fused = 1;
            if (ctrl->nonfinite) set_error(ctrl, DBSCAN_ERR_INVALID_ARG);
        }
    }
    __syncthreads();
    const bool direct = s_direct != 0;             // the form of the test, uniform
    const float ascale = direct ? -1.f : -2.f;     // the row's scale of c_i
    {
        const float thrx = s_thrx;
        const int npad = nt * FT;
        for (int i = blockIdx.x * FT + tid; i < npad; i += nb * FT) {
            float *base = a.staged + (size_t)(i / FT) * (size_t)(d + 1) * FT + (i % FT);
            if (i >= n) {
                for (int k = 0; k < d; ++k) base[(size_t)k * FT] = 0.f;
                base[(size_t)d * FT] = PAD_NORM;
                a.T[i] = PAD_THRESH;
                continue;
            }
            float nrm = 0.f;
            for (int k = 0; k < d; ++k) {
                // the direct form takes the coordinates as they are (prep.cu)
                const float c = load_point(a.pts, a.dtype, (size_t)i * d + k) - (direct ? 0.f : s_centre[k]);
                base[(size_t)k * FT] = c;
                nrm = fmaf(c, c, nrm);
            }
            if (s_direct) {
                base[(size_t)d * FT] = 0.f;
                a.T[i] = direct_threshold(thrx, integral);
            } else {
                base[(size_t)d * FT] = nrm;
                a.T[i] = integral ? thrx - nrm : nextafterf(thrx - nrm, INFINITY);
            }
        }
        for (int t = blockIdx.x * FT + tid; t < nt; t += nb * FT) a.tcore[t] = 0;
    }
    if (!grid_sync(ctrl, nb)) return;

    // ---- count: upper triangle, each pair credited to both points ---------------
    const int npairs = nt * (nt + 1) / 2;
    for (int u = blockIdx.x; u < npairs; u += nb) {
        int rb, cb;
        tri_pair(u, nt, rb, cb);
        const float *gc = a.staged + (size_t)cb * (d + 1) * FT;
        const float *gr = a.staged + (size_t)rb * (d + 1) * FT;
        for (int e = tid; e < (d + 1) * FT; e += FT) s_col[e] = gc[e];
        RowPoint<D> r;
        if (D > 0) {
#pragma unroll
            for (int k = 0; k < (D > 0 ? D : 1); ++k) r.a[k] = ascale * gr[k * FT + tid];
        } else {
            for (int k = 0; k < d; ++k) s_row[k * FT + tid] = ascale * gr[k * FT + tid];
        }
        s_aux[tid] = 0;
        __syncthreads();
        const float Ti = a.T[rb * FT + tid];
        int rowc = 0;
        if (rb == cb) {
            for (int j = 0; j < FT; ++j) rowc += pair_value<D>(direct, r, s_row, s_col, d, j) < Ti;
        } else {
            for (int j = 0; j < FT; ++j) {
                if (pair_value<D>(direct, r, s_row, s_col, d, j) < Ti) {
                    ++rowc;
                    atomicAdd(&s_aux[j], 1);
                }
            }
        }
        if (rowc) atomicAdd(&a.cnt[rb * FT + tid], rowc);
        __syncthreads();
        if (rb != cb && s_aux[tid]) atomicAdd(&a.cnt[cb * FT + tid], s_aux[tid]);
        __syncthreads();
    }
    if (!grid_sync(ctrl, nb)) return;

    if (a.cnt_out) {   // counts only
        for (int i = blockIdx.x * FT + tid; i < n; i += nb * FT) a.cnt_out[i] = a.cnt[i];
        return;
    }

    // ---- core flags, union-find init, per-tile core counts, candidate list -------
    for (int i = blockIdx.x * FT + tid; i < nt * FT; i += nb * FT) {
        const bool valid = i < n;
        const int c = valid ? a.cnt[i] : 0;
        const bool core = valid && c >= a.min_pts;
        const bool cand = valid && !core && c >= 2;
        if (valid) a.is_core[i] = core ? 1 : 0;
        a.parent[i] = i;
        if (core) { atomicAdd(&a.tcore[i / FT], 1); atomicAdd(&ctrl->n_core, 1); }
        if (cand) a.candlist[atomicAdd(&ctrl->n_cand, 1)] = i;   // any order: a minimum follows
    }
    if (!grid_sync(ctrl, nb)) return;

    // ---- union: core-core pairs of the upper triangle, in two passes ------------
    // In input order every tile pair holds pairs of every cluster, and hooking
    // roots in arbitrary index order grows long parent chains, each step of a
    // find an L2 round trip.  Pass 0 therefore only hooks: for every core-core
    // neighbour pair the larger index's parent takes the smaller index by
    // atomicMin (no finds; parent[x] <= x still holds, and every link is a
    // neighbour pair).  Every core's parent is then compressed to its root.
    // Pass 1 unites the sets of every core-core neighbour pair, staging the
    // column tile's compressed parents in shared memory and skipping each pair
    // whose two sides already had one root (sets only merge, so such a pair
    // stays joined); after pass 0 most pairs are skipped.
    int *s_par = s_aux + FT;
    for (int pass = 0; pass < 2; ++pass) {
        for (int u = blockIdx.x; u < npairs; u += nb) {
            int rb, cb;
            tri_pair(u, nt, rb, cb);
            if (a.tcore[rb] == 0 || a.tcore[cb] == 0) continue;   // uniform over the block
            const float *gc = a.staged + (size_t)cb * (d + 1) * FT;
            const float *gr = a.staged + (size_t)rb * (d + 1) * FT;
            for (int e = tid; e < (d + 1) * FT; e += FT) s_col[e] = gc[e];
            RowPoint<D> r;
            if (D > 0) {
#pragma unroll
                for (int k = 0; k < (D > 0 ? D : 1); ++k) r.a[k] = ascale * gr[k * FT + tid];
            } else {
                for (int k = 0; k < d; ++k) s_row[k * FT + tid] = ascale * gr[k * FT + tid];
            }
            const int q = cb * FT + tid;
            const bool qcore = q < n && a.cnt[q] >= a.min_pts;
            s_aux[tid] = qcore ? 1 : 0;
            s_par[tid] = qcore ? __ldcg(a.parent + q) : -1;
            __syncthreads();
            const int p = rb * FT + tid;
            if (p < n && a.cnt[p] >= a.min_pts) {
                const float Ti = a.T[p];
                if (pass == 0) {
                    int lo = p;   // the smallest neighbour index of this row so far
                    for (int j = (rb == cb ? tid + 1 : 0); j < FT; ++j) {
                        if (!s_aux[j] || !(pair_value<D>(direct, r, s_row, s_col, d, j) < Ti)) continue;
                        const int qj = cb * FT + j;
                        if (qj < p) lo = min(lo, qj);
                        else atomicMin(a.parent + qj, p);
                    }
                    if (lo < p) atomicMin(a.parent + p, lo);
                } else {
                    // root: this row's set; j0, j1: the last two snapshot roots
                    // joined to it (their whole trees are in the set)
                    int root = __ldcg(a.parent + p), j0 = root, j1 = root;
                    for (int j = (rb == cb ? tid + 1 : 0); j < FT; ++j) {
                        const int sj = s_par[j];
                        if (!s_aux[j] || sj == root || sj == j0 || sj == j1 ||
                            !(pair_value<D>(direct, r, s_row, s_col, d, j) < Ti))
                            continue;
                        j1 = j0;
                        j0 = sj;
                        if (__ldcg(a.parent + sj) == root) continue;   // already joined
                        root = f_unite(a.parent, root, sj, ctrl);
                    }
                }
            }
            __syncthreads();
        }
        if (!grid_sync(ctrl, nb)) return;
        if (pass == 0) {   // compress: every core position points at its root
            for (int i = blockIdx.x * FT + tid; i < n; i += nb * FT)
                if (a.cnt[i] >= a.min_pts) __stcg(a.parent + i, f_find(a.parent, i, ctrl));
            if (!grid_sync(ctrl, nb)) return;
        }
    }

    // ---- flatten: core labels are roots (the smallest core input index) ---------
    for (int i = blockIdx.x * FT + tid; i < n; i += nb * FT) {
        const int c = a.cnt[i];
        int lab = -1;
        if (c >= a.min_pts) lab = f_find(a.parent, i, ctrl);
        else if (c >= 2) lab = 0x7fffffff;   // candidate: smallest neighbouring label below
        a.clabel[i] = lab;
        a.labels[i] = lab;
    }
    if (!grid_sync(ctrl, nb)) return;

    // ---- border: the candidate list (128 at a time) x core tiles -----------------
    const int ncand = __ldcg(&ctrl->n_cand);
    const int ncb = (ncand + FT - 1) / FT;
    for (int u = blockIdx.x; u < ncb * nt; u += nb) {
        const int kb = u / nt, cb = u % nt;
        if (a.tcore[cb] == 0) continue;
        const float *gc = a.staged + (size_t)cb * (d + 1) * FT;
        for (int e = tid; e < (d + 1) * FT; e += FT) s_col[e] = gc[e];
        const int k = kb * FT + tid;
        const int p = k < ncand ? a.candlist[k] : -1;
        RowPoint<D> r;
        if (p >= 0) {
            const float *gp = a.staged + (size_t)(p / FT) * (d + 1) * FT + (p % FT);
            if (D > 0) {
#pragma unroll
                for (int kk = 0; kk < (D > 0 ? D : 1); ++kk) r.a[kk] = ascale * gp[kk * FT];
            } else {
                for (int kk = 0; kk < d; ++kk) s_row[kk * FT + tid] = ascale * gp[kk * FT];
            }
        }
        const int q = cb * FT + tid;
        // the column's label if it is a core point, else -1
        s_aux[tid] = (q < n && a.cnt[q] >= a.min_pts) ? a.clabel[q] : -1;
        __syncthreads();
        if (p >= 0) {
            const float Ti = a.T[p];
            int best = 0x7fffffff;
            for (int j = 0; j < FT; ++j)
                if (s_aux[j] >= 0 && pair_value<D>(direct, r, s_row, s_col, d, j) < Ti) best = min(best, s_aux[j]);
            if (best != 0x7fffffff) atomicMin(&a.labels[p], best);
        }
        __syncthreads();
    }
    if (!grid_sync(ctrl, nb)) return;

    // ---- finalize: candidates without a core neighbour are noise -----------------
    for (int i = blockIdx.x * FT + tid; i < n; i += nb * FT)
        if (a.labels[i] == 0x7fffffff) a.labels[i] = -1;
}

template <int D>
cudaError_t launch_d(const FusedArgs &args, cudaStream_t s) {
    const int d = D > 0 ? D : args.d;
    const size_t smem = ((size_t)(d + 1) * FT + (D > 0 ? 0 : (size_t)d * FT)) * sizeof(float) +
                        2 * FT * sizeof(int);
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fused<D>, FT, smem)) != cudaSuccess)
        return e;
    const int npairs = args.ntiles * (args.ntiles + 1) / 2;
    int blocks = min(max(per_sm, 1) * sms, max(npairs, 1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(FT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every block resident: the barriers hold
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_fused<D>, args);
}

}  // namespace

bool fused_eligible(int64_t n, int d) {
    return n > 0 && d <= FUSED_MAX_D && n <= (d <= 4 ? FUSED_MAX_N_LOW_D : FUSED_MAX_N);
}

cudaError_t launch_fused(const void *points, int dtype, int64_t n, int d, float eps, int min_pts,
                         int32_t *labels, uint8_t *is_core, int32_t *cnt_out, const Work &w,
                         const Layout &L, cudaStream_t s) {
    FusedArgs a{};
    a.pts = points;
    a.dtype = dtype;
    a.n = (int)n;
    a.d = d;
    a.min_pts = min_pts;
    a.ntiles = (int)L.ntiles;
    a.eps2 = eps * eps;
    a.ctrl = w.ctrl;
    a.smin = reinterpret_cast<unsigned *>(w.stat_min);
    a.smax = reinterpret_cast<unsigned *>(w.stat_max);
    a.staged = w.staged_all;
    a.T = w.T_all;
    a.cnt = w.cnt;
    a.parent = w.parent;
    a.clabel = w.clabel;
    a.tcore = w.troot;       // per-tile core counts (ntiles ints)
    a.candlist = w.candidx;  // border candidates' positions (n ints)
    a.labels = labels;
    a.is_core = is_core;
    a.cnt_out = cnt_out;
    switch (d) {
    case 1: return launch_d<1>(a, s);
    case 2: return launch_d<2>(a, s);
    case 3: return launch_d<3>(a, s);
    case 4: return launch_d<4>(a, s);
    default: return launch_d<0>(a, s);
    }
}

}  // namespace dbscan
