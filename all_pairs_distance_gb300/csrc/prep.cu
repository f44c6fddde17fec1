// Preparation step: per-dimension ranges, centring, squared norms and row
// thresholds, written into the tiled structure-of-arrays layout the sweep
// kernels read.
//
// "Design and optimization of DBSCAN Algorithm based on CUDA", §IV-B2
// ("Put the iteration code outsides"), rewrites the squared distance as
//     dist(t, p) = T + P[n] - (X p_x + Y p_y + Z p_z),  T = |t|^2, X = 2 t_x, ...
// so that per pair only the dot product remains.  Here the point-only terms
// are hoisted the same way:
//     nrm_j = |c_j|^2                      (per column point)
//     v_ij  = nrm_j + sum_k (-2 c_ik) c_jk  (per pair: d fused multiply-adds)
//     neighbour  <=>  |c_i - c_j|^2 <= eps2  <=>  v_ij < T_i
// with c = x - centre.  For integer data T_i = floor(min(eps2, R)) + 1 - nrm_i
// (R = sum_k range_k^2 bounds every squared distance), which turns "<= eps2"
// into a strict comparison between integers.  Centring each dimension on the
// midpoint of its range keeps every partial sum of v_ij within
// [-sum_k M_k^2, R] (M_k the largest |c_k|), so for integer data with R < 2^24
// every value is an exactly representable integer.  Without centring the
// page's form overflows 2^24 already at d = 3 over [0, 2047].
#include "dbscan_internal.cuh"

#include <math.h>

namespace dbscan {

__device__ __forceinline__ float load_point(const void *p, int dtype, size_t e) {
    if (dtype == DBSCAN_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[e]);
    return reinterpret_cast<const float *>(p)[e];
}

__global__ void k_init_stats(Ctrl *ctrl, int *smin, int *smax, int64_t n, int d) {
    for (int k = threadIdx.x; k < DBSCAN_MAX_D; k += blockDim.x) {
        smin[k] = 0x7fffffff;
        smax[k] = (int)0x80000000;
    }
    if (threadIdx.x == 0) ctrl->n_all = (int)n;
}

// Element-parallel pass over [n, d]: with a grid stride that is a multiple
// of d, every thread stays on one dimension and keeps scalar min/max.
__global__ void k_stats(const void *pts, int dtype, int64_t n, int d, Ctrl *ctrl,
                        int *smin, int *smax) {
    __shared__ int bmin[DBSCAN_MAX_D], bmax[DBSCAN_MAX_D];
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        bmin[k] = 0x7fffffff;
        bmax[k] = (int)0x80000000;
    }
    __syncthreads();
    const int64_t total = n * (int64_t)d;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t stride = (nthreads / d) * d;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int kmin = 0x7fffffff, kmax = (int)0x80000000, nonint = 0, nonfin = 0;
    if (t < stride) {
        for (int64_t e = t; e < total; e += stride) {
            float x = load_point(pts, dtype, (size_t)e);
            if (!isfinite(x)) { nonfin = 1; continue; }
            if (x != rintf(x)) nonint = 1;
            int key = float_key(x);
            kmin = min(kmin, key);
            kmax = max(kmax, key);
        }
        int dim = (int)(t % d);
        if (kmin != 0x7fffffff) {
            atomicMin(&bmin[dim], kmin);
            atomicMax(&bmax[dim], kmax);
        }
    }
    if (__syncthreads_or(nonint) && threadIdx.x == 0) atomicOr(&ctrl->nonint, 1);
    if (__syncthreads_or(nonfin) && threadIdx.x == 0) atomicOr(&ctrl->nonfinite, 1);
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        if (bmin[k] != 0x7fffffff) {
            atomicMin(&smin[k], bmin[k]);
            atomicMax(&smax[k], bmax[k]);
        }
    }
}

// One block: centres, the exactness bound and the threshold constant.
__global__ void k_setup(Ctrl *ctrl, const int *smin, const int *smax, float *centre,
                        int d, float eps2) {
    __shared__ double part[DBSCAN_MAX_D];
    const bool integral = ctrl->nonint == 0;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        float lo = key_float(smin[k]), hi = key_float(smax[k]);
        if (smin[k] == 0x7fffffff) { lo = 0.f; hi = 0.f; }  // only non-finite values
        float c = integral ? floorf(0.5f * lo + 0.5f * hi) : 0.5f * lo + 0.5f * hi;
        centre[k] = c;
        double r = (double)hi - (double)lo;
        part[k] = r * r;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double R = 0.0;
        for (int k = 0; k < d; ++k) R += part[k];
        ctrl->range_sq = (float)R;
        if (integral) {
            double t = floor((double)eps2);
            if (t > R) t = R;
            ctrl->thrx = (float)(t + 1.0);
        } else {
            ctrl->thrx = eps2;
        }
        ctrl->exact = (integral && R < 16777215.0) ? 1 : 0;
        if (ctrl->nonfinite) set_error(ctrl, DBSCAN_ERR_INVALID_ARG);
    }
}

// One thread per (padded) point: centred coordinates and norm into the
// tiled layout, row threshold into T.
__global__ void k_stage(const void *pts, int dtype, int64_t n, int d, const Ctrl *ctrl,
                        const float *centre, float *staged, float *T, int64_t npad) {
    extern __shared__ float s_centre[];
    for (int k = threadIdx.x; k < d; k += blockDim.x) s_centre[k] = centre[k];
    __syncthreads();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= npad) return;
    const int64_t tile = i / BT;
    const int lane = (int)(i % BT);
    float *base = staged + (size_t)tile * (size_t)(d + 1) * BT + lane;
    if (i >= n) {
        for (int k = 0; k < d; ++k) base[(size_t)k * BT] = 0.f;
        base[(size_t)d * BT] = PAD_NORM;
        T[i] = PAD_THRESH;
        return;
    }
    float nrm = 0.f;
    for (int k = 0; k < d; ++k) {
        float c = load_point(pts, dtype, (size_t)i * d + k) - s_centre[k];
        base[(size_t)k * BT] = c;
        nrm = fmaf(c, c, nrm);
    }
    base[(size_t)d * BT] = nrm;
    const float thrx = ctrl->thrx;
    if (ctrl->nonint == 0) {
        T[i] = thrx - nrm;
    } else {
        T[i] = nextafterf(thrx - nrm, INFINITY);
    }
}

cudaError_t launch_prep(const void *points, int dtype, int64_t n, int d, float eps,
                        const Work &w, const Layout &L, cudaStream_t s) {
    const float eps2 = eps * eps;
    k_init_stats<<<1, 256, 0, s>>>(w.ctrl, w.stat_min, w.stat_max, n, d);
    int64_t elems = n * (int64_t)d;
    int blocks = (int)((elems + 255) / 256);
    int cap = persistent_ctas((const void *)k_stats, 256, 0) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_stats<<<blocks, 256, 0, s>>>(points, dtype, n, d, w.ctrl, w.stat_min, w.stat_max);
    k_setup<<<1, 256, 0, s>>>(w.ctrl, w.stat_min, w.stat_max, w.centre, d, eps2);
    const int64_t npad = L.ntiles * BT;
    int sblocks = (int)((npad + 255) / 256);
    k_stage<<<sblocks, 256, d * sizeof(float), s>>>(points, dtype, n, d, w.ctrl, w.centre,
                                                     w.staged_all, w.T_all, npad);
    return cudaGetLastError();
}

}  // namespace dbscan
