// Label compaction: cluster labels renumbered 0..k-1, noise kept at -1.
//
// A label of dbscan_fit* is the smallest input index among its cluster's core
// points, and that point carries its own index as its label.  So the clusters
// are exactly the positions j with labels[j] == j ("representatives"), and the
// new id of label j is the number of representatives below j: one pass flags
// and counts them per block, one block scans the block counts, a third pass
// ranks the representatives, and a fourth maps every label through the ranks.
// The first pass also checks that every label is -1 or a representative
// (anything else was not produced by dbscan_fit*) and flags an error.
#include "dbscan_internal.cuh"

namespace dbscan {
namespace {

constexpr int LB_BLOCK = 1024;    // labels per block of the scan
constexpr int LB_THREADS = 256;

__global__ void k_rep_counts(const int32_t *labels, int64_t n, int *bsum, int *err) {
    __shared__ int s_cnt;
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    int c = 0;
    const int64_t base = (int64_t)blockIdx.x * LB_BLOCK;
    for (int r = 0; r < LB_BLOCK / LB_THREADS; ++r) {
        const int64_t i = base + r * LB_THREADS + threadIdx.x;
        if (i >= n) break;
        const int32_t l = labels[i];
        if (l == i) {
            ++c;
        } else if (l != -1 && (l < 0 || l >= n || labels[l] != l)) {
            atomicExch(err, 1);
        }
    }
    atomicAdd(&s_cnt, c);
    __syncthreads();
    if (threadIdx.x == 0) bsum[blockIdx.x] = s_cnt;
}

// One block: exclusive scan of the block counts in place; the total to *k.
__global__ void k_scan_counts(int *bsum, int64_t nblocks, int *k) {
    __shared__ int warp_tot[32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int64_t base = 0; base < nblocks; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        const int v = i < nblocks ? bsum[i] : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const int excl = carry + (wid ? warp_tot[wid - 1] : 0) + x - v;
        if (i < nblocks) bsum[i] = excl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = excl + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) *k = carry;
}

// rank[j] for every representative j: its block's offset plus the
// representatives before it in the block (a block-wide exclusive scan).
__global__ void k_rank(const int32_t *labels, int64_t n, const int *bsum, int *rank) {
    __shared__ int warp_tot[LB_THREADS / 32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = bsum[blockIdx.x];
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t base = (int64_t)blockIdx.x * LB_BLOCK;
    for (int r = 0; r < LB_BLOCK / LB_THREADS; ++r) {
        const int64_t i = base + r * LB_THREADS + threadIdx.x;
        const int f = i < n && labels[i] == i ? 1 : 0;
        int x = f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[wid] = x;
        __syncthreads();
        int off = 0;
        for (int w = 0; w < wid; ++w) off += warp_tot[w];
        if (f) rank[i] = carry + off + x - 1;
        __syncthreads();
        if (threadIdx.x == LB_THREADS - 1) carry += off + x;
        __syncthreads();
    }
}

__global__ void k_map(const int32_t *labels, int64_t n, const int *rank, int32_t *out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t l = labels[i];
        out[i] = l >= 0 ? rank[l] : -1;
    }
}

}  // namespace

size_t compact_labels_scratch(int64_t n) {
    const int64_t nb = (n + LB_BLOCK - 1) / LB_BLOCK;
    return ((size_t)n * sizeof(int) + 255) / 256 * 256 + (size_t)(nb + 2) * sizeof(int);
}

// Passes 1-3; the scratch's last two ints are then k and the error flag.
cudaError_t launch_compact_labels_rank(const int32_t *labels, int64_t n, void *scratch, int **k_err,
                                       cudaStream_t s) {
    const int64_t nb = (n + LB_BLOCK - 1) / LB_BLOCK;
    int *rank = static_cast<int *>(scratch);
    int *bsum = reinterpret_cast<int *>(static_cast<char *>(scratch) +
                                        ((size_t)n * sizeof(int) + 255) / 256 * 256);
    int *k = bsum + nb;
    *k_err = k;
    cudaError_t e = cudaMemsetAsync(k, 0, 2 * sizeof(int), s);
    if (e != cudaSuccess) return e;
    k_rep_counts<<<(unsigned)nb, LB_THREADS, 0, s>>>(labels, n, bsum, k + 1);
    k_scan_counts<<<1, 1024, 0, s>>>(bsum, nb, k);
    k_rank<<<(unsigned)nb, LB_THREADS, 0, s>>>(labels, n, bsum, rank);
    return cudaGetLastError();
}

// Pass 4: every label through the ranks (out may be labels itself).
cudaError_t launch_compact_labels_map(const int32_t *labels, int64_t n, const void *scratch, int32_t *out,
                                      cudaStream_t s) {
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (n + 255) / 256;
    const unsigned grid = (unsigned)(want < 8 * (int64_t)sms ? want : 8 * (int64_t)sms);
    k_map<<<grid, 256, 0, s>>>(labels, n, static_cast<const int *>(scratch), out);
    return cudaGetLastError();
}

}  // namespace dbscan
