// Locality order of the points.
//
// The sweeps evaluate every pair of points, whatever their order; the order
// only decides which pairs meet in the same tile.  "Design and optimization
// of DBSCAN Algorithm based on CUDA" processes points in input order (§IV-A);
// with shuffled input nearly every 32 x 32 block of a sweep then holds some
// neighbour pair, and every such block takes the exact (slow) path of the
// sweep's hit test.  Sorting the points by a Morton (Z-order) key first puts
// neighbours next to each other, so blocks with a neighbour pair become rare
// and the fast test (is any value below the threshold?) decides almost every
// block.  Results do not depend on the order: counts are per point, clusters
// are named by their smallest original core index, and border points take the
// smallest neighbouring label (see compact.cu).
//
// Key: d <= 3 interleaves the quantised coordinates themselves (30 bits for
// d = 1, 15 per axis for d = 2, 10 per axis for d = 3); d > 3 interleaves three
// fixed +-1 projections sum_k s_mk x_k, 10 bits each.  Three projections mix
// clusters once d > 3 (in 64-D, 200 clusters projected to 3-D overlap; in
// 16-D the union's tile boxes stay wide), so for 3 < d <= 64 the key leads
// with the nearest of 512 pivots -- input points spread evenly over the input
// order -- followed by the projection key: a cluster's points share a pivot
// and land next to each other.  The top `bits` bits of the
// 30-bit key name a bin (bits = ceil(log2 n) clamped to [8, 20]); a counting
// sort over the bins gives the permutation (order within a bin is unspecified).
#include "dbscan_internal.cuh"

namespace dbscan {

constexpr int BIN_SCAN = 1024;          // bins per block of the bin scan
constexpr int BIN_SCAN_THREADS = 256;

int order_bits(int64_t n) {
    int b = 0;
    while (b < 30 && ((int64_t)1 << b) < n) ++b;
    if (b < 8) b = 8;
    if (b > 20) b = 20;
    return b;
}

// Sign of projection m on dimension k: a fixed pseudo-random +-1 pattern.
__host__ __device__ inline float proj_sign(int m, int k) {
    uint32_t h = (uint32_t)k * 0x9E3779B1u + (uint32_t)(m + 1) * 0x85EBCA77u;
    h ^= h >> 15;
    h *= 0x2C1B3C6Du;
    h ^= h >> 12;
    return (h & 1u) ? -1.f : 1.f;
}

__device__ __forceinline__ uint32_t spread3(uint32_t x) {   // 10 bits -> every third bit
    x &= 0x3ffu;
    x = (x | (x << 16)) & 0x030000ffu;
    x = (x | (x << 8)) & 0x0300f00fu;
    x = (x | (x << 4)) & 0x030c30c3u;
    x = (x | (x << 2)) & 0x09249249u;
    return x;
}

__device__ __forceinline__ uint32_t spread2(uint32_t x) {   // 15 bits -> every other bit
    x &= 0x7fffu;
    x = (x | (x << 8)) & 0x00ff00ffu;
    x = (x | (x << 4)) & 0x0f0f0f0fu;
    x = (x | (x << 2)) & 0x33333333u;
    x = (x | (x << 1)) & 0x55555555u;
    return x;
}

constexpr int PIVOT_MIN_D = 3;    // PIVOT_MIN_D < d <= PIVOT_MAX_D orders by nearest pivot first
constexpr int PIVOT_MAX_D = 64;   // beyond, tiles stay too wide for the box test
constexpr int PIVOT_BITS = 9;     // 512 pivots
constexpr int PIVOT_DIMS = 16;    // distances to the pivots over at most 16 coordinates

// Coordinate m (< PIVOT_DIMS) of the pivot distance: all d coordinates when
// d <= 16 (slots m >= d hold 0 in points and pivots alike), else 16 spread
// evenly across the d.
__host__ __device__ inline int pivot_dim(int m, int d) {
    return d <= PIVOT_DIMS ? m : (int)((int64_t)m * d / PIVOT_DIMS);
}
__device__ __forceinline__ float pivot_coord(const void *pts, int dtype, int64_t row, int m, int d) {
    return m < d ? load_point(pts, dtype, (size_t)row * d + pivot_dim(m, d)) : 0.f;
}

__host__ __device__ inline bool use_pivots(int d) { return d > PIVOT_MIN_D && d <= PIVOT_MAX_D; }

// Nearest pivot of every point, into pid[i] (ties to the lower pivot), over the
// coordinates pivot_dim picks (at most 16: enough to tell clusters apart).
// Pivots are the input points floor(j n / P).  |x - p|^2 = |x|^2 + |p|^2 - 2 x.p, and
// |x|^2 is the same for every pivot, so each thread minimises |p|^2 - 2 x.p
// for PIVOT_PPT points held in registers, four pivots at a time: one 16-byte
// shared-memory load of -2p feeds 4 x PIVOT_PPT independent FMA chains (the
// pivot table is read once per PIVOT_PPT points, which bounds the kernel).
// Float rounding only perturbs the order, never a result.
constexpr int PIVOT_PPT = 4;
constexpr int PIVOT_THREADS = 256;
__global__ void __launch_bounds__(PIVOT_THREADS) k_pivot_assign(const void *pts, int dtype, int64_t n,
                                                                int d, const int *rank, int *pid) {
    constexpr int P = 1 << PIVOT_BITS;
    __shared__ __align__(16) float s_piv[PIVOT_DIMS * P];   // -2 p_jm at m * P + j
    __shared__ __align__(16) float s_pn[P];                  // |p_j|^2 over those coordinates
    __shared__ int s_rank[P];                                // renumbered pivot ids
    for (int j = threadIdx.x; j < P; j += blockDim.x) s_rank[j] = rank[j];
    for (int e = threadIdx.x; e < P * PIVOT_DIMS; e += blockDim.x) {
        const int j = e % P, m = e / P;
        const int64_t src = (int64_t)j * n / P;
        s_piv[e] = -2.f * pivot_coord(pts, dtype, src, m, d);
    }
    __syncthreads();
    for (int j = threadIdx.x; j < P; j += blockDim.x) {
        float q = 0.f;
        for (int m = 0; m < PIVOT_DIMS; ++m) q = fmaf(s_piv[m * P + j], s_piv[m * P + j], q);
        s_pn[j] = 0.25f * q;
    }
    __syncthreads();
    // point q of this thread: base + q * blockDim.x (consecutive threads,
    // consecutive points)
    const int64_t base = (int64_t)blockIdx.x * blockDim.x * PIVOT_PPT + threadIdx.x;
    float x[PIVOT_PPT][PIVOT_DIMS];
#pragma unroll
    for (int q = 0; q < PIVOT_PPT; ++q) {
        const int64_t i = base + (int64_t)q * blockDim.x;
#pragma unroll
        for (int m = 0; m < PIVOT_DIMS; ++m) x[q][m] = i < n ? pivot_coord(pts, dtype, i, m, d) : 0.f;
    }
    float best[PIVOT_PPT];
    int bj[PIVOT_PPT];
#pragma unroll
    for (int q = 0; q < PIVOT_PPT; ++q) {
        best[q] = INFINITY;
        bj[q] = 0;
    }
    for (int j0 = 0; j0 < P; j0 += 4) {
        const float4 pn = *reinterpret_cast<const float4 *>(s_pn + j0);
        float a[PIVOT_PPT][4];
#pragma unroll
        for (int q = 0; q < PIVOT_PPT; ++q) {
            a[q][0] = pn.x;
            a[q][1] = pn.y;
            a[q][2] = pn.z;
            a[q][3] = pn.w;
        }
#pragma unroll
        for (int m = 0; m < PIVOT_DIMS; ++m) {
            const float4 pv = *reinterpret_cast<const float4 *>(s_piv + m * P + j0);
#pragma unroll
            for (int q = 0; q < PIVOT_PPT; ++q) {
                a[q][0] = fmaf(x[q][m], pv.x, a[q][0]);
                a[q][1] = fmaf(x[q][m], pv.y, a[q][1]);
                a[q][2] = fmaf(x[q][m], pv.z, a[q][2]);
                a[q][3] = fmaf(x[q][m], pv.w, a[q][3]);
            }
        }
#pragma unroll
        for (int q = 0; q < PIVOT_PPT; ++q)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (a[q][c] < best[q]) { best[q] = a[q][c]; bj[q] = j0 + c; }
    }
#pragma unroll
    for (int q = 0; q < PIVOT_PPT; ++q) {
        const int64_t i = base + (int64_t)q * blockDim.x;
        if (i < n) pid[i] = s_rank[bj[q]];
    }
}

// Renumbering of the pivots so that pivots of one cluster are consecutive:
// in input order consecutive pivot ids belong to different clusters, and a
// tile that straddles two pivot groups then spans two clusters, whose box the
// union's tile test cannot cull.  One block: pivots within 2 eps of each other
// (over the pivot coordinates; a distance over some of the coordinates is at
// most the full one) are joined by a shared-memory union-find, and pivot j
// gets rank[j], its position in the order (component, index).  The order only
// decides which points share a tile, never a result.
// 1,024 threads: thread t takes pivot j = t % 512 against every second pivot
// k > j (the half t / 512), its own coordinates in registers.
__global__ void __launch_bounds__(1024) k_pivot_rank(const void *pts, int dtype, int64_t n, int d,
                                                     float eps2, int *rank) {
    constexpr int P = 1 << PIVOT_BITS;
    __shared__ float s_p[PIVOT_DIMS * P];
    __shared__ int par[P];
    const int j = threadIdx.x % P, half = threadIdx.x / P;
    if (half == 0) {
        const int64_t src = (int64_t)j * n / P;
        for (int m = 0; m < PIVOT_DIMS; ++m) s_p[m * P + j] = pivot_coord(pts, dtype, src, m, d);
        par[j] = j;
    }
    __syncthreads();
    float pj[PIVOT_DIMS];
#pragma unroll
    for (int m = 0; m < PIVOT_DIMS; ++m) pj[m] = s_p[m * P + j];
    volatile int *vp = par;
    auto find = [&](int x) {
        for (int it = 0; it < P; ++it) {   // parents only move towards smaller roots
            const int q = vp[x];
            if (q == x) break;
            x = q;
        }
        return x;
    };
    const float thr = 4.f * eps2;
    for (int k = j + 1 + half; k < P; k += 2) {
        float d2 = 0.f;
#pragma unroll
        for (int m = 0; m < PIVOT_DIMS; ++m) {
            const float t = pj[m] - s_p[m * P + k];
            d2 = fmaf(t, t, d2);
        }
        if (!(d2 <= thr)) continue;
        for (int it = 0; it < 4 * P; ++it) {   // hook the larger root under the smaller
            int a = find(j), b = find(k);
            if (a == b) break;
            if (a < b) { const int t = a; a = b; b = t; }
            if (atomicCAS(&par[a], a, b) == a) break;
        }
    }
    __syncthreads();
    const int rj = find(j);
    __syncthreads();
    if (half == 0) par[j] = rj;   // every pivot's root (the smallest pivot of its component)
    __syncthreads();
    if (half == 0) {
        int r = 0;
        for (int k = 0; k < P; ++k) r += (par[k] < rj) || (par[k] == rj && k < j);
        rank[j] = r;
    }
}

// One thread: the axes' lower bounds and quantisation scales into Ctrl.
__global__ void k_order_setup(Ctrl *ctrl, const int *smin, const int *smax, int d) {
    if (threadIdx.x != 0) return;
    const int naxes = d < 3 ? d : 3;
    const int abits = d == 1 ? 30 : (d == 2 ? 15 : 10);
    for (int m = 0; m < naxes; ++m) {
        double lo = 0.0, hi = 0.0;
        if (d <= 3) {
            if (smin[m] != 0x7fffffff) {
                lo = key_float(smin[m]);
                hi = key_float(smax[m]);
            }
        } else {
            for (int k = 0; k < d; ++k) {
                if (smin[k] == 0x7fffffff) continue;
                const double a = key_float(smin[k]), b = key_float(smax[k]);
                if (proj_sign(m, k) > 0.f) { lo += a; hi += b; }
                else { lo -= b; hi -= a; }
            }
        }
        const double span = hi - lo;
        ctrl->ord_lo[m] = (float)lo;
        ctrl->ord_scale[m] = span > 0.0 ? (float)((double)(1 << abits) / (span * 1.0000001 + 1e-30)) : 0.f;
    }
}

__device__ __forceinline__ uint32_t quantise(float v, float lo, float scale, float qmax) {
    float t = (v - lo) * scale;
    t = fminf(fmaxf(t, 0.f), qmax);
    return (uint32_t)t;
}

// Bin of every point, and the bin histogram.
__global__ void k_order_key(const void *pts, int dtype, int64_t n, int d, const Ctrl *ctrl,
                            int shift, int *bin, int *hist) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint32_t key;
    if (d == 1) {
        key = quantise(load_point(pts, dtype, (size_t)i), ctrl->ord_lo[0], ctrl->ord_scale[0],
                       1073741823.f);
        key = key > 0x3fffffffu ? 0x3fffffffu : key;
    } else if (d == 2) {
        uint32_t q0 = quantise(load_point(pts, dtype, (size_t)i * 2), ctrl->ord_lo[0],
                               ctrl->ord_scale[0], 32767.f);
        uint32_t q1 = quantise(load_point(pts, dtype, (size_t)i * 2 + 1), ctrl->ord_lo[1],
                               ctrl->ord_scale[1], 32767.f);
        key = spread2(q0) | (spread2(q1) << 1);
    } else {
        float v[3];
        if (d == 3) {
            for (int m = 0; m < 3; ++m) v[m] = load_point(pts, dtype, (size_t)i * 3 + m);
        } else {
            v[0] = v[1] = v[2] = 0.f;
            for (int k = 0; k < d; ++k) {
                const float x = load_point(pts, dtype, (size_t)i * d + k);
                v[0] += proj_sign(0, k) * x;
                v[1] += proj_sign(1, k) * x;
                v[2] += proj_sign(2, k) * x;
            }
        }
        key = 0;
        for (int m = 0; m < 3; ++m)
            key |= spread3(quantise(v[m], ctrl->ord_lo[m], ctrl->ord_scale[m], 1023.f)) << m;
        if (use_pivots(d))   // nearest pivot first (bin[i] holds it on entry)
            key = ((uint32_t)bin[i] << (30 - PIVOT_BITS)) | (key >> PIVOT_BITS);
    }
    const int b = (int)(key >> shift);
    bin[i] = b;
    atomicAdd(hist + b, 1);
}

// Exclusive scan of the histogram within blocks of BIN_SCAN bins; block totals
// to btot.
__global__ void k_bin_scan(const int *hist, int nbins, int *start, int *btot) {
    __shared__ int wsum[BIN_SCAN_THREADS / 32];
    constexpr int PER = BIN_SCAN / BIN_SCAN_THREADS;
    const int base = blockIdx.x * BIN_SCAN + threadIdx.x * PER;
    int v[PER], s = 0;
    for (int r = 0; r < PER; ++r) {
        v[r] = base + r < nbins ? hist[base + r] : 0;
        s += v[r];
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    int woff = 0, tot = 0;
    for (int w = 0; w < BIN_SCAN_THREADS / 32; ++w) {
        if (w < wid) woff += wsum[w];
        tot += wsum[w];
    }
    int run = woff + x - s;
    for (int r = 0; r < PER; ++r) {
        if (base + r < nbins) start[base + r] = run;
        run += v[r];
    }
    if (threadIdx.x == 0) btot[blockIdx.x] = tot;
}

// One block of 1024 threads: exclusive scan of the block totals, in place.
__global__ void k_bin_top(int *btot, int nblk) {
    __shared__ int wsum[32];
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int v = t < nblk ? btot[t] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    int woff = 0;
    for (int w = 0; w < wid; ++w) woff += wsum[w];
    if (t < nblk) btot[t] = woff + x - v;
}

// perm[position] = original index.
__global__ void k_order_scatter(const int *bin, int64_t n, const int *start, const int *btot,
                                int *hist, int *perm) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int b = bin[i];
    const int pos = start[b] + btot[b / BIN_SCAN] + atomicSub(hist + b, 1) - 1;
    perm[pos] = (int)i;
}

cudaError_t launch_order(const void *points, int dtype, int64_t n, int d, const Work &w,
                         const Layout &L, cudaStream_t s) {
    const int nbins = 1 << L.order_bits;
    const int nblk = (nbins + BIN_SCAN - 1) / BIN_SCAN;
    if (cudaMemsetAsync(w.hist, 0, (size_t)nbins * sizeof(int), s) != cudaSuccess) return cudaGetLastError();
    k_order_setup<<<1, 32, 0, s>>>(w.ctrl, w.stat_min, w.stat_max, d);
    const int blocks = (int)((n + 255) / 256);
    if (use_pivots(d)) {
        const int64_t per = (int64_t)PIVOT_THREADS * PIVOT_PPT;
        k_pivot_rank<<<1, 2 << PIVOT_BITS, 0, s>>>(points, dtype, n, d, L.eps2, w.pivrank);
        k_pivot_assign<<<(unsigned)((n + per - 1) / per), PIVOT_THREADS, 0, s>>>(points, dtype, n, d,
                                                                                  w.pivrank, w.bin);
    }
    k_order_key<<<blocks, 256, 0, s>>>(points, dtype, n, d, w.ctrl, 30 - L.order_bits, w.bin,
                                       w.hist);
    k_bin_scan<<<nblk, BIN_SCAN_THREADS, 0, s>>>(w.hist, nbins, w.bstart, w.btot);
    k_bin_top<<<1, 1024, 0, s>>>(w.btot, nblk);
    k_order_scatter<<<blocks, 256, 0, s>>>(w.bin, n, w.bstart, w.btot, w.hist, w.perm);
    return cudaGetLastError();
}

// Neighbour counts back into input order.
__global__ void k_unpermute(const int *perm, const int *src, int64_t n, int32_t *dst) {
    const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p < n) dst[perm[p]] = src[p];
}

cudaError_t launch_unpermute_counts(const Work &w, const Layout &L, int32_t *cnt_out,
                                    cudaStream_t s) {
    k_unpermute<<<(unsigned)((L.n + 255) / 256), 256, 0, s>>>(w.perm, w.cnt, L.n, cnt_out);
    return cudaGetLastError();
}

}  // namespace dbscan
