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
//
// Tensor-core operands.  When every centred coordinate is an integer small
// enough for the MMA input type (|2c| <= 2048 for tf32 and f16, <= 256 for
// bf16), the
// pair quantity w_ij = |c_i - c_j|^2 - thrx is written as one dot product
//     A_i = [-2 c_i,  1, B, ..,   n0_i, n1_i, ..,  -h0, -h1, ..]
//     B_j = [   c_j,  n0_j, n1_j, .., 1, B, ..,     1,   B, ..]
// with |c|^2 = sum_k n_k B^k and thrx = sum_k h_k B^k (all digits in [0, B)),
// every element exactly representable.  The positive terms sum to at most
// 4 S and the negative ones to at most 2 S + thrx (S = sum_k M_k^2); when both
// are at most 2^24 every partial sum the tensor core forms, in any order, is
// an integer of magnitude at most 2^24, exact in f32, and w_ij < 0 <=>
// neighbour.  Every kind accumulates in f32,
// except the opt-in F16H kind, taken only when the whole row fits one K = 16
// MMA: its f16 accumulator rounds the sum once, which keeps the sign (the
// smallest nonzero |w| is 1; overflow gives +-inf; an exact zero is stored as
// +0) provided the tensor core forms the K = 16 sum exactly first -- not
// documented by NVIDIA, observed on GB300 by the tests.
#include "dbscan_internal.cuh"

#include <math.h>

namespace dbscan {

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

// One block: centres, the exactness bound, the threshold constant and the
// tensor-core path (allow: mask of TC_ALLOW_* the call permits).
__global__ void k_setup(Ctrl *ctrl, const int *smin, const int *smax, float *centre,
                        int d, float eps2, int allow) {
    __shared__ double part[DBSCAN_MAX_D];
    __shared__ double mpart[DBSCAN_MAX_D];
    __shared__ double rpart[DBSCAN_MAX_D];
    const bool integral = ctrl->nonint == 0;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        float lo = key_float(smin[k]), hi = key_float(smax[k]);
        if (smin[k] == 0x7fffffff) { lo = 0.f; hi = 0.f; }  // only non-finite values
        float c = integral ? floorf(0.5f * lo + 0.5f * hi) : 0.5f * lo + 0.5f * hi;
        centre[k] = c;
        double r = (double)hi - (double)lo;
        part[k] = r * r;
        double m = fmax((double)hi - (double)c, (double)c - (double)lo);
        mpart[k] = m * m;
        rpart[k] = r;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double R = 0.0, S = 0.0, rmax = 0.0;
        for (int k = 0; k < d; ++k) {
            R += part[k];
            S += mpart[k];
            rmax = fmax(rmax, rpart[k]);
        }
        ctrl->range_sq = (float)R;
        if (integral) {
            double t = floor((double)eps2);
            if (t > R) t = R;
            ctrl->thrx = (float)(t + 1.0);
        } else {
            ctrl->thrx = eps2;
        }
        ctrl->exact = (integral && R < 16777215.0) ? 1 : 0;
        // Box gap bound of the CUDA-core sweeps' tile test.  Exact data: the
        // gaps are integers and the test is the neighbour test itself (thrx).
        // Otherwise the sweeps' float test v_ij < T_i can accept a pair whose
        // exact squared distance exceeds eps^2 by its rounding error: every
        // partial sum of v_ij and T_i is at most 3 S + eps^2 in magnitude
        // (S bounds |c|^2, the range R <= 4 S bounds every gap), about 5 d + 2
        // roundings of relative size 2^-24 reach the test, and the gap sum
        // adds d + 1 more; 2^-16 (d + 4) (S + eps^2 + 1) covers them all
        // with a factor above 20, so a skipped tile pair holds no pair the
        // sweep would have accepted.
        if (ctrl->exact) {
            ctrl->cull_thr = ctrl->thrx;
        } else {
            const double m = ldexp((double)(d + 4) * (S + (double)eps2 + 1.0), -16);
            ctrl->cull_thr = __double2float_ru((double)eps2 + m);
        }
        // tensor-core eligibility (integer data, exact elements, exact sums)
        const double thrx = (double)ctrl->thrx;
        const int nt = tc_nt_for(TC_TF32, thrx);
        int kind = TC_NONE;
        // every partial sum lies in [-(2 S + thrx), 4 S]; integers of magnitude
        // up to 2^24 are exact in f32 (d = 256 over [0, 255] reaches 4 S = 2^24)
        if (integral && !ctrl->nonfinite && 4.0 * S <= 16777216.0 && 2.0 * S + thrx <= 16777216.0) {
            // preference: the opt-in F16H (one MMA, half-width accumulator reads),
            // then BF16 (ranges up to 256), F16 (up to 2048; the same MMA rate),
            // TF32 (half the rate; threshold constants of three digits)
            const int ntb = tc_nt_for(TC_BF16, thrx);
            if ((allow & TC_ALLOW_F16H) && rmax <= 2048.0 && tc_fits(TC_F16H, d, nt)) {
                kind = TC_F16H;
                ctrl->tc_nt = nt;
            } else if ((allow & TC_ALLOW_BF16) && rmax <= 256.0 && tc_fits(TC_BF16, d, ntb)) {
                kind = TC_BF16;
                ctrl->tc_nt = ntb;
            } else if ((allow & TC_ALLOW_F16) && rmax <= 2048.0 && tc_fits(TC_F16, d, nt)) {
                kind = TC_F16;
                ctrl->tc_nt = nt;
            } else if ((allow & TC_ALLOW_TF32) && rmax <= 2048.0 && tc_fits(TC_TF32, d, nt)) {
                kind = TC_TF32;
                ctrl->tc_nt = nt;
            }
        }
        ctrl->tc_kind = kind;
        ctrl->tc_kpad = kind ? tc_kpad(kind, d, ctrl->tc_nt) : 0;
        ctrl->tc_kbytes = kind ? tc_kbytes(kind, d, ctrl->tc_nt) : 0;
        if (ctrl->nonfinite) set_error(ctrl, DBSCAN_ERR_INVALID_ARG);
    }
}

// Element k of a point's operand row (see the header comment):
//   A (row form)    [-2 c,  base powers,  norm digits,  -threshold digits, 0..]
//   B (column form) [   c,  norm digits,  base powers,   base powers,      0..]
struct OperandRow {
    const float *src;   // the point's staged coordinates (stride BT), then its norm
    int d, nd, nt, base, nrm, th;
    __device__ __forceinline__ float elem(int k, bool col) const {
        if (k < d) {
            const float c = src[(size_t)k * BT];
            return col ? c : -2.f * c;
        }
        k -= d;
        if (k < 2 * nd + nt) {
            const int j = k < nd ? k : (k < 2 * nd ? k - nd : k - 2 * nd);
            int pw = 1;
            for (int t = 0; t < j; ++t) pw *= base;
            if (k < nd) return col ? (float)((nrm / pw) % base) : (float)pw;        // column norm
            if (k < 2 * nd) return col ? (float)pw : (float)((nrm / pw) % base);    // row norm
            return col ? (float)pw : (float)(-((th / pw) % base));                  // threshold
        }
        return 0.f;
    }
};

__device__ __forceinline__ uint32_t pack_pair(int kind, float lo, float hi) {
    uint16_t a, b;
    if (tc_is_f16(kind)) {
        const __half x = __float2half_rn(lo), y = __float2half_rn(hi);
        a = *reinterpret_cast<const uint16_t *>(&x);
        b = *reinterpret_cast<const uint16_t *>(&y);
    } else {
        const __nv_bfloat16 x = __float2bfloat16_rn(lo), y = __float2bfloat16_rn(hi);
        a = *reinterpret_cast<const uint16_t *>(&x);
        b = *reinterpret_cast<const uint16_t *>(&y);
    }
    return (uint32_t)a | ((uint32_t)b << 16);
}

// 16 bytes of an operand row: 4 tf32 or 8 f16/bf16 elements from element k0.
__device__ __forceinline__ uint4 row_chunk(const OperandRow &r, int kind, int k0, bool col) {
    uint4 v;
    if (kind == TC_TF32) {
        v.x = __float_as_uint(r.elem(k0, col));
        v.y = __float_as_uint(r.elem(k0 + 1, col));
        v.z = __float_as_uint(r.elem(k0 + 2, col));
        v.w = __float_as_uint(r.elem(k0 + 3, col));
    } else {
        v.x = pack_pair(kind, r.elem(k0, col), r.elem(k0 + 1, col));
        v.y = pack_pair(kind, r.elem(k0 + 2, col), r.elem(k0 + 3, col));
        v.z = pack_pair(kind, r.elem(k0 + 4, col), r.elem(k0 + 5, col));
        v.w = pack_pair(kind, r.elem(k0 + 6, col), r.elem(k0 + 7, col));
    }
    return v;
}

// Tensor-core operand tiles from the staged points: A (row form) and,
// optionally, B (column form).  Tiles are packed back to back (128 x kbytes
// each) so that consecutive tiles can be copied in one piece.  Slots at or
// beyond *count are zero; the sweep masks them out by index.  Each thread
// writes its row 16 bytes at a time: in the K-major layout 16 bytes of a row
// are contiguous and 8 consecutive rows fill 128 contiguous bytes.
__global__ void k_stage_umma(const Ctrl *ctrl, const int *count, const float *staged, int d,
                             int64_t npad, uint8_t *ua, uint8_t *ub) {
    const int kind = ctrl->tc_kind;
    if (kind == TC_NONE) return;
    const int kbytes = ctrl->tc_kbytes;
    const size_t tile_stride = (size_t)BT * kbytes;
    const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= npad) return;
    const int64_t tile = p / BT;
    const int row = (int)(p % BT);
    uint8_t *ta = ua + (size_t)tile * tile_stride;
    uint8_t *tb = ub ? ub + (size_t)tile * tile_stride : nullptr;
    const int per = kind == TC_TF32 ? 4 : 8;   // elements per 16 bytes
    if (p >= *count) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int q = 0; q < kbytes / 16; ++q) {
            *reinterpret_cast<uint4 *>(ta + umma_offset(row, 16 * q, kbytes)) = z;
            if (tb) *reinterpret_cast<uint4 *>(tb + umma_offset(row, 16 * q, kbytes)) = z;
        }
        return;
    }
    OperandRow r;
    r.src = staged + (size_t)tile * (size_t)(d + 1) * BT + row;
    r.d = d;
    r.nd = tc_norm_digits(kind);
    r.nt = ctrl->tc_nt;
    r.base = kind == TC_BF16 ? 256 : 2048;
    r.nrm = (int)r.src[(size_t)d * BT];
    r.th = (int)ctrl->thrx;
    for (int q = 0; q < kbytes / 16; ++q) {
        *reinterpret_cast<uint4 *>(ta + umma_offset(row, 16 * q, kbytes)) = row_chunk(r, kind, q * per, false);
        if (tb) *reinterpret_cast<uint4 *>(tb + umma_offset(row, 16 * q, kbytes)) = row_chunk(r, kind, q * per, true);
    }
}

cudaError_t launch_stage_umma(const Work &w, const Layout &L, int which, cudaStream_t s) {
    if (L.umma_tile_bytes == 0) return cudaSuccess;
    const int64_t npad = L.ntiles * BT;
    const int blocks = (int)((npad + 255) / 256);
    if (which == 0)
        k_stage_umma<<<blocks, 256, 0, s>>>(w.ctrl, &w.ctrl->n_all, w.staged_all, L.d, npad,
                                            w.ua_all, w.ub_all);
    else if (which == 1)
        k_stage_umma<<<blocks, 256, 0, s>>>(w.ctrl, &w.ctrl->n_core, w.staged_core, L.d, npad,
                                            w.ua_core, w.ub_core);
    else
        k_stage_umma<<<blocks, 256, 0, s>>>(w.ctrl, &w.ctrl->n_cand, w.staged_cand, L.d, npad,
                                            w.ua_cand, nullptr);
    return cudaGetLastError();
}

// One thread per (padded) position p: the centred coordinates and norm of
// input point perm[p] into the tiled layout, its row threshold into T[p].
// Data off the exact path (Ctrl::exact = 0) are tested in the direct form
// sum_k (c_jk - c_ik)^2 < T on CUDA cores: the norm slot then holds 0 (the
// sum's start; PAD_NORM for padding) and T[p] the common threshold
// (dbscan_internal.cuh).
__global__ void k_stage(const void *pts, int dtype, int64_t n, int d, const Ctrl *ctrl,
                        const float *centre, const int *perm, float *staged, float *T,
                        int64_t npad) {
    extern __shared__ float s_centre[];
    // the direct form takes the coordinates as they are: the difference of
    // two nearby floats is exact, while centring rounds each coordinate once
    for (int k = threadIdx.x; k < d; k += blockDim.x) s_centre[k] = ctrl->exact ? centre[k] : 0.f;
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
    const int64_t src = perm[i];
    float nrm = 0.f;
    for (int k = 0; k < d; ++k) {
        float c = load_point(pts, dtype, (size_t)src * d + k) - s_centre[k];
        base[(size_t)k * BT] = c;
        nrm = fmaf(c, c, nrm);
    }
    if (!ctrl->exact) {
        base[(size_t)d * BT] = 0.f;
        T[i] = direct_threshold(ctrl->thrx, ctrl->nonint == 0);
        return;
    }
    base[(size_t)d * BT] = nrm;
    const float thrx = ctrl->thrx;
    if (ctrl->nonint == 0) {
        T[i] = thrx - nrm;
    } else {
        T[i] = nextafterf(thrx - nrm, INFINITY);
    }
}

cudaError_t launch_prep_order(const void *points, int dtype, int64_t n, int d, float eps, int allow_tc,
                              const Work &w, const Layout &L, cudaStream_t s) {
    const float eps2 = eps * eps;
    k_init_stats<<<1, 256, 0, s>>>(w.ctrl, w.stat_min, w.stat_max, n, d);
    int64_t elems = n * (int64_t)d;
    int blocks = (int)((elems + 255) / 256);
    int cap = persistent_ctas((const void *)k_stats, 256, 0) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_stats<<<blocks, 256, 0, s>>>(points, dtype, n, d, w.ctrl, w.stat_min, w.stat_max);
    k_setup<<<1, 256, 0, s>>>(w.ctrl, w.stat_min, w.stat_max, w.centre, d, eps2,
                              L.umma_tile_bytes ? allow_tc : 0);
    return launch_order(points, dtype, n, d, w, L, s);
}

cudaError_t launch_prep_stage(const void *points, int dtype, int64_t n, int d, const Work &w,
                              const Layout &L, cudaStream_t s) {
    const int64_t npad = L.ntiles * BT;
    int sblocks = (int)((npad + 255) / 256);
    k_stage<<<sblocks, 256, d * sizeof(float), s>>>(points, dtype, n, d, w.ctrl, w.centre,
                                                     w.perm, w.staged_all, w.T_all, npad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_stage_umma(w, L, 0, s);
}

cudaError_t launch_prep(const void *points, int dtype, int64_t n, int d, float eps, int allow_tc,
                        const Work &w, const Layout &L, cudaStream_t s) {
    cudaError_t e = launch_prep_order(points, dtype, n, d, eps, allow_tc, w, L, s);
    if (e != cudaSuccess) return e;
    return launch_prep_stage(points, dtype, n, d, w, L, s);
}

}  // namespace dbscan
