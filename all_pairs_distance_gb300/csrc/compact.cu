// Core flags, stable compaction of core points and border candidates,
// union-find flatten and label finalisation.
//
// Core points follow "Design and optimization of DBSCAN Algorithm based on
// CUDA", §II (a point is core when at least MinPts points lie within eps of
// it).  The page's primitive-cluster construction (§IV-B, a cluster matrix
// with a valid flag per column) and its merge kernel (§IV-C) need O(N^2)
// memory; here the core points are compacted (stable, in the staged locality
// order), merged by union-find in the core-core sweep, and each component is
// named by the smallest input index among its core points.  Non-core points
// with at least one neighbour besides themselves are the border candidates
// scanned by the border sweep; the rest are noise.  Every array indexed by
// position p maps to the caller's numbering through perm[p].
#include "dbscan_internal.cuh"

#include <math.h>

namespace dbscan {

constexpr int CT_THREADS = 256;
constexpr int PER_THREAD = SCAN_BLOCK / CT_THREADS;  // 4

// Pass A: flags, is_core output, initial labels, per-block counts.
__global__ void k_flags(const int *cnt, const int *perm, int64_t n, int min_pts,
                        uint8_t *is_core, int32_t *labels, int *bsum, int64_t nblocks) {
    __shared__ int s_core, s_cand;
    if (threadIdx.x == 0) { s_core = 0; s_cand = 0; }
    __syncthreads();
    int ncore = 0, ncand = 0;
    const int64_t base = blockIdx.x * (int64_t)SCAN_BLOCK;
    for (int r = 0; r < PER_THREAD; ++r) {
        int64_t i = base + r * CT_THREADS + threadIdx.x;
        if (i >= n) break;
        int c = cnt[i];
        bool core = c >= min_pts;
        bool cand = !core && c >= 2;
        const int src = perm[i];
        is_core[src] = core ? 1 : 0;
        labels[src] = cand ? 0x7fffffff : -1;
        ncore += core;
        ncand += cand;
    }
    atomicAdd(&s_core, ncore);
    atomicAdd(&s_cand, ncand);
    __syncthreads();
    if (threadIdx.x == 0) {
        bsum[blockIdx.x] = s_core;
        bsum[nblocks + blockIdx.x] = s_cand;
    }
}

// Pass B (one block): exclusive scan of the per-block counts, totals to Ctrl.
__global__ void k_scan_blocks(int *bsum, int64_t nblocks, Ctrl *ctrl) {
    __shared__ int warp_tot[32];
    __shared__ int carry[2];
    if (threadIdx.x < 2) carry[threadIdx.x] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int which = 0; which < 2; ++which) {
        int *arr = bsum + which * nblocks;
        for (int64_t base = 0; base < nblocks; base += blockDim.x) {
            int64_t i = base + threadIdx.x;
            int v = i < nblocks ? arr[i] : 0;
            int x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) warp_tot[wid] = x;
            __syncthreads();
            if (wid == 0) {
                int t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    int y = __shfl_up_sync(0xffffffffu, t, o);
                    if (lane >= o) t += y;
                }
                warp_tot[lane] = t;   // inclusive over warps
            }
            __syncthreads();
            int warp_off = wid ? warp_tot[wid - 1] : 0;
            int excl = carry[which] + warp_off + x - v;
            if (i < nblocks) arr[i] = excl;
            __syncthreads();
            if (threadIdx.x == blockDim.x - 1) carry[which] = excl + v;
            __syncthreads();
        }
    }
    if (threadIdx.x == 0) {
        ctrl->n_core = carry[0];
        ctrl->n_cand = carry[1];
    }
}

__device__ __forceinline__ void copy_staged(const float *src_tiles, float *dst_tiles, int d,
                                            int64_t from, int64_t to) {
    const size_t tf = (size_t)(d + 1) * BT;
    const float *s = src_tiles + (size_t)(from / BT) * tf + (from % BT);
    float *t = dst_tiles + (size_t)(to / BT) * tf + (to % BT);
    for (int k = 0; k <= d; ++k) t[(size_t)k * BT] = s[(size_t)k * BT];
}

// Pass C: stable scatter of core points and candidates with their staged
// coordinates and thresholds; parent[pos] = pos.
__global__ void k_scatter(const int *cnt, const int *perm, int64_t n, int d, int min_pts,
                          const int *bsum, int64_t nblocks, const float *staged_all,
                          const float *T_all, float *staged_core, float *T_core, int *cidx,
                          int *parent, int *rootmin, float *staged_cand, float *T_cand,
                          int *candidx) {
    __shared__ int wsum[2][CT_THREADS / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int off_core = bsum[blockIdx.x];
    int off_cand = bsum[nblocks + blockIdx.x];
    const int64_t base = blockIdx.x * (int64_t)SCAN_BLOCK;
    for (int r = 0; r < PER_THREAD; ++r) {
        int64_t i = base + r * CT_THREADS + threadIdx.x;
        bool core = false, cand = false;
        if (i < n) {
            int c = cnt[i];
            core = c >= min_pts;
            cand = !core && c >= 2;
        }
        unsigned bc = __ballot_sync(0xffffffffu, core);
        unsigned bd = __ballot_sync(0xffffffffu, cand);
        if (lane == 0) { wsum[0][wid] = __popc(bc); wsum[1][wid] = __popc(bd); }
        __syncthreads();
        int pc = off_core, pd = off_cand, tc = 0, td = 0;
        for (int w = 0; w < CT_THREADS / 32; ++w) {
            if (w < wid) { pc += wsum[0][w]; pd += wsum[1][w]; }
            tc += wsum[0][w];
            td += wsum[1][w];
        }
        const unsigned below = (1u << lane) - 1u;
        pc += __popc(bc & below);
        pd += __popc(bd & below);
        if (core) {
            cidx[pc] = perm[i];
            parent[pc] = pc;
            rootmin[pc] = 0x7fffffff;
            copy_staged(staged_all, staged_core, d, i, pc);
            T_core[pc] = T_all[i];
        } else if (cand) {
            candidx[pd] = perm[i];
            copy_staged(staged_all, staged_cand, d, i, pd);
            T_cand[pd] = T_all[i];
        }
        off_core += tc;
        off_cand += td;
        __syncthreads();
    }
}

// Bounding box of every tile of a staged array (min and max of each centred
// coordinate over the tile's valid points): one block of BT threads per tile.
__global__ void k_tile_boxes(const float *staged, const int *count, int d, float *box) {
    __shared__ float red[2][BT / 32];
    const int t = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int cnt = *count;
    if ((int64_t)t * BT >= cnt) return;
    const bool valid = (int64_t)t * BT + threadIdx.x < cnt;
    const float *src = staged + (size_t)t * (size_t)(d + 1) * BT + threadIdx.x;
    for (int k = 0; k < d; ++k) {
        const float v = src[(size_t)k * BT];
        float lo = valid ? v : INFINITY, hi = valid ? v : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (lane == 0) { red[0][wid] = lo; red[1][wid] = hi; }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w2 = 1; w2 < BT / 32; ++w2) {
                lo = fminf(lo, red[0][w2]);
                hi = fmaxf(hi, red[1][w2]);
            }
            box[((size_t)t * d + k) * 2] = lo;
            box[((size_t)t * d + k) * 2 + 1] = hi;
        }
        __syncthreads();
    }
}

// Box of every group of 32 consecutive tiles (over its valid tiles), so that
// the sweeps can skip a whole group with one test: one thread per group and
// dimension.
__global__ void k_group_boxes(const float *box, const int *count, int d, int64_t ngroups,
                              float *gbox) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= ngroups * d) return;
    const int64_t g = e / d;
    const int k = (int)(e % d);
    const int64_t ntv = ((int64_t)*count + BT - 1) / BT;   // valid tiles
    float lo = INFINITY, hi = -INFINITY;
    for (int64_t t = g * CULL_GROUP; t < (g + 1) * CULL_GROUP && t < ntv; ++t) {
        lo = fminf(lo, box[(t * d + k) * 2]);
        hi = fmaxf(hi, box[(t * d + k) * 2 + 1]);
    }
    gbox[(g * d + k) * 2] = lo;
    gbox[(g * d + k) * 2 + 1] = hi;
}

cudaError_t launch_tile_boxes(const Work &w, const Layout &L, int which, cudaStream_t s) {
    if (L.box_floats == 0) return cudaSuccess;
    const float *st = which == 0 ? w.staged_all : (which == 1 ? w.staged_core : w.staged_cand);
    const int *cnt = which == 0 ? &w.ctrl->n_all : (which == 1 ? &w.ctrl->n_core : &w.ctrl->n_cand);
    float *box = which == 0 ? w.box_all : (which == 1 ? w.box_core : w.box_cand);
    k_tile_boxes<<<(unsigned)L.ntiles, BT, 0, s>>>(st, cnt, L.d, box);
    if (which != 2) {   // column arrays (all points, core points) also get group boxes
        const int64_t ngroups = (L.ntiles + CULL_GROUP - 1) / CULL_GROUP;
        k_group_boxes<<<(unsigned)((ngroups * L.d + 255) / 256), 256, 0, s>>>(
            box, cnt, L.d, ngroups, which == 0 ? w.gbox_all : w.gbox_core);
    }
    return cudaGetLastError();
}

// Padding slots of the last tile of the core and candidate arrays.
__global__ void k_pad_tails(const Ctrl *ctrl, int d, float *staged_core, float *T_core,
                            float *staged_cand, float *T_cand) {
    const size_t tf = (size_t)(d + 1) * BT;
    for (int which = 0; which < 2; ++which) {
        const int cnt = which == 0 ? ctrl->n_core : ctrl->n_cand;
        float *st = which == 0 ? staged_core : staged_cand;
        float *T = which == 0 ? T_core : T_cand;
        const int end = ((cnt + BT - 1) / BT) * BT;
        for (int p = cnt + threadIdx.x; p < end; p += blockDim.x) {
            float *t = st + (size_t)(p / BT) * tf + (p % BT);
            for (int k = 0; k < d; ++k) t[(size_t)k * BT] = 0.f;
            t[(size_t)d * BT] = PAD_NORM;
            T[p] = PAD_THRESH;
        }
    }
}

// Flatten: every core position to its root (the smallest position of its
// component); the root collects the smallest input index of its component.
__global__ void k_flatten(Ctrl *ctrl, const int *parent, const int *cidx, int *clabel,
                          int *rootmin) {
    const int n_core = ctrl->n_core;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_core; p += gridDim.x * blockDim.x) {
        int x = p;
        int it = 0;
        for (; it < (1 << 22); ++it) {
            int q = __ldcg(parent + x);
            if (q == x) break;
            x = q;
        }
        if (it == (1 << 22)) set_error(ctrl, DBSCAN_ERR_INTERNAL);
        clabel[p] = x;
        atomicMin(rootmin + x, cidx[p]);
    }
}

// Label of every core point: its component's smallest input index.
__global__ void k_core_labels(const Ctrl *ctrl, const int *cidx, const int *rootmin,
                              int *clabel, int32_t *labels) {
    const int n_core = ctrl->n_core;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_core; p += gridDim.x * blockDim.x) {
        const int lab = rootmin[clabel[p]];
        clabel[p] = lab;
        labels[cidx[p]] = lab;
    }
}

// Candidates that met no core point are noise.
__global__ void k_finalize(const Ctrl *ctrl, const int *candidx, int32_t *labels) {
    const int n_cand = ctrl->n_cand;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_cand; p += gridDim.x * blockDim.x) {
        int i = candidx[p];
        if (labels[i] == 0x7fffffff) labels[i] = -1;
    }
}

static int grid_for(int64_t n, int threads, const void *kernel) {
    int64_t g = (n + threads - 1) / threads;
    int cap = persistent_ctas(kernel, threads, 0) * 2;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

cudaError_t launch_compact(const Work &w, const Layout &L, int min_pts, int32_t *labels,
                           uint8_t *is_core, cudaStream_t s) {
    const int64_t nb = L.nscan_blocks;
    k_flags<<<(unsigned)nb, CT_THREADS, 0, s>>>(w.cnt, w.perm, L.n, min_pts, is_core, labels,
                                                w.bsum, nb);
    k_scan_blocks<<<1, 1024, 0, s>>>(w.bsum, nb, w.ctrl);
    k_scatter<<<(unsigned)nb, CT_THREADS, 0, s>>>(w.cnt, w.perm, L.n, L.d, min_pts, w.bsum, nb,
                                                  w.staged_all, w.T_all, w.staged_core, w.T_core,
                                                  w.cidx, w.parent, w.rootmin, w.staged_cand,
                                                  w.T_cand, w.candidx);
    k_pad_tails<<<1, 128, 0, s>>>(w.ctrl, L.d, w.staged_core, w.T_core, w.staged_cand, w.T_cand);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_stage_umma(w, L, 1, s);   // core operands (candidate rows: after the union)
}

cudaError_t launch_flatten(const Work &w, const Layout &L, int32_t *labels, cudaStream_t s) {
    k_flatten<<<grid_for(L.n, 256, (const void *)k_flatten), 256, 0, s>>>(w.ctrl, w.parent, w.cidx,
                                                                          w.clabel, w.rootmin);
    k_core_labels<<<grid_for(L.n, 256, (const void *)k_core_labels), 256, 0, s>>>(
        w.ctrl, w.cidx, w.rootmin, w.clabel, labels);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const Work &w, const Layout &L, int32_t *labels, cudaStream_t s) {
    k_finalize<<<grid_for(L.n, 256, (const void *)k_finalize), 256, 0, s>>>(w.ctrl, w.candidx,
                                                                            labels);
    return cudaGetLastError();
}

}  // namespace dbscan
