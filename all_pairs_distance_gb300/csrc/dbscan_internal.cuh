// Internal definitions shared by the CUDA translation units of the DBSCAN
// library: workspace layout, the device control block, launch wrappers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>
#include <math.h>

#include "../../include/dbscan.h"

namespace dbscan {

// Points are staged in tiles of BT points.  A tile holds, for each of the d
// dimensions, the BT centred coordinates (structure of arrays), followed by
// the BT squared norms: (d + 1) * BT floats, 512-byte aligned rows.
constexpr int BT = 128;
constexpr int SCAN_BLOCK = 1024;   // elements per block of the compaction scan
// Tile culling keeps per-tile bounding boxes for d up to this dimension (the
// locality order's nearest-pivot key covers 3 < d <= 64 and keeps tiles tight).
constexpr int CULL_MAX_D = 64;
// Tiles per group of the group boxes (the coarse level of the test).
constexpr int CULL_GROUP = 8;

// Sentinels for the padding slots of the last tile: a padding column has a
// huge norm and never tests as a neighbour; a padding row has a hugely
// negative threshold and never tests as a neighbour either.
constexpr float PAD_NORM = 1.0e30f;
constexpr float PAD_THRESH = -1.0e30f;

// Two forms of the CUDA-core neighbour test, with A_ik the row's staged
// scale of c_ik and s_j the column's norm slot:
//   expanded (exact data):  v_ij = s_j + sum_k A_ik c_jk,  A = -2 c_i,
//                           s_j = |c_j|^2, T_i = thrx - |c_i|^2: every sum
//                           is an exact integer below 2^24, so the test is
//                           exact and one FMA per coordinate;
//   direct (other data):    v_ij = s_j + sum_k (c_jk + A_ik)^2,  A = -c_i,
//                           s_j = 0, T_i = direct_threshold: accurate to a
//                           few roundings of d^2 itself (the expanded form
//                           errs by roundings of |c|^2, far above eps^2 when
//                           the coordinates are large), and symmetric --
//                           (c_jk - c_ik)^2 is the same number for either
//                           point as the row, so every pass decides a pair
//                           the same way whatever the order of the points.
// A pair is a neighbour iff v_ij < T_i in both; padding has s_j = PAD_NORM
// and T_i = PAD_THRESH.
__host__ __device__ inline float direct_threshold(float thrx, bool integral) {
    // integer data: d^2 <= floor(eps^2) iff d^2 < thrx; otherwise d^2 <= eps^2
    return integral ? thrx : nextafterf(thrx, INFINITY);
}

// Device control block at offset 0 of every workspace.
struct Ctrl {
    int err;            // first device-side error (a dbscan_status), 0 = none
    int n_core;         // number of core points
    int n_cand;         // number of border candidates (non-core, count >= 2)
    int nonint;         // set when a coordinate is not an integer
    int nonfinite;      // set when a coordinate is NaN or infinite
    int exact;          // 1 when the exactness bound holds (set by setup)
    float thrx;         // row threshold constant, see prep.cu
    int n_all;          // number of points
    unsigned unit_ctr[8];   // CUDA-core work-unit counters: count, union bands 1-3 (slots 1-3), border (5)
    float range_sq;     // sum_k (max_k - min_k)^2
    int tc_kind;        // tensor-core path chosen by setup: a TcKind (TC_NONE = CUDA cores)
    int tc_kpad;        // padded K of the tensor-core operands (elements)
    int tc_kbytes;      // bytes of one operand row (tc_kpad * element size)
    int tc_nt;          // digits of the threshold constant in the operands
    float ord_lo[3];    // locality order: lower bound of each key axis
    float ord_scale[3]; // locality order: quantisation scale of each key axis
    unsigned band_ctr[8];   // work-unit counters of the tensor-core union bands
    int fused;          // 1 when the call ran the fused single-launch pipeline
    unsigned bar_gen;   // fused pipeline: grid barrier generation
    unsigned bar_count; // fused pipeline: blocks arrived at the current barrier
    int bar_abort;      // fused pipeline: set when a barrier wait timed out
    float cull_thr;     // CUDA-core tile test: keep a tile pair whose squared box gap is below
    int pad1[24];
};
static_assert(sizeof(Ctrl) == 256, "Ctrl must be 256 bytes");

// Workspace carve-up (host side).  All offsets are 256-byte aligned.
struct Layout {
    int64_t n;
    int32_t d;
    float eps2;           // fl32(eps * eps) of the call (0 in a bare size query)
    unsigned allow;       // tensor-core kinds the call may take (TC_ALLOW_* bits)
    int rows[3];          // row blocks per unit of count, union, border (0 = automatic)
    int fused;            // 1: the whole call runs as the fused single-launch pipeline
    int rank, world;      // sharding: the sweeps take work units u with u % world == rank
    int64_t ntiles;       // ceil(n / BT)
    size_t tile_floats;   // (d + 1) * BT
    size_t off_ctrl, off_stats, off_staged_all, off_staged_core, off_staged_cand;
    size_t off_T_all, off_T_core, off_T_cand;
    size_t off_cnt, off_cidx, off_candidx, off_parent, off_clabel, off_bsum;
    size_t umma_tile_bytes;   // bytes of one 128-point operand tile (largest path), 0 = none
    size_t off_ua_all, off_ub_all, off_ua_core, off_ub_core, off_ua_cand;
    int order_bits;       // bins of the locality order: 2^order_bits
    size_t off_bin, off_perm, off_hist, off_bstart, off_btot, off_rootmin;
    int cull;             // 1: the count sweep also skips tile pairs whose boxes are eps apart
    int cull_nbr;         // 1: union and border skip tile pairs whose boxes are eps apart
    size_t box_floats;    // floats of one box array (ntiles x 2d), 0 when d > CULL_MAX_D
    size_t gbox_floats;   // floats of one group-box array (ceil(ntiles / CULL_GROUP) x 2d)
    size_t off_box_all, off_box_core, off_box_cand;
    size_t off_gbox_all, off_gbox_core;
    size_t off_troot;     // [ntiles] ints: common root of each core tile's points, or -1
    size_t off_pivrank;   // [512] ints: renumbered pivots of the locality order
    int64_t nscan_blocks;
    size_t total;
};

Layout make_layout(int64_t n, int32_t d);

// Device pointers into one workspace.
struct Work {
    Ctrl *ctrl;
    int *stat_min;        // [DBSCAN_MAX_D] ordered-int keys of per-dimension minima
    int *stat_max;        // [DBSCAN_MAX_D] ordered-int keys of per-dimension maxima
    float *centre;        // [DBSCAN_MAX_D] per-dimension centre
    float *staged_all, *staged_core, *staged_cand;
    float *T_all, *T_core, *T_cand;
    int *cnt;             // [n] neighbour counts
    int *cidx;            // [n] input index of each core position (staged order)
    int *candidx;         // [n] input index of each border-candidate position
    int *parent;          // [n] union-find parents over core positions
    int *clabel;          // [n] root, then final label, of each core position
    int *bsum;            // [2 * nscan_blocks] per-block counts of the compaction scan
    uint8_t *ua_all, *ub_all, *ua_core, *ub_core, *ua_cand;   // tensor-core operand tiles
    int *bin;             // [n] locality bin of each input point
    int *perm;            // [ntiles * BT] input index of each staged position
    int *hist, *bstart;   // [2^order_bits] bin counts and bin starts
    int *btot;            // [2^order_bits / 1024] bin-block offsets
    int *rootmin;         // [n] smallest input index of each union-find root's component
    float *box_all, *box_core, *box_cand;   // [ntiles][d][min, max] tile bounding boxes
    float *gbox_all, *gbox_core;            // [ntiles / CULL_GROUP][d][min, max] group boxes
    int *troot;           // [ntiles] common root of each core tile's points, or -1 (union)
    int *pivrank;         // [512] position of each pivot in the locality order's pivot order
};

Work carve(void *base, const Layout &L);

// Sweep modes.
enum SweepMode { SWEEP_COUNT = 0, SWEEP_UNION = 1, SWEEP_BORDER = 2 };

// Tensor-core paths.  The operands carry, per point, the d coordinates plus
// base-B digits of the squared norms and of the threshold constant, so one
// MMA yields w_ij = |c_i - c_j|^2 - thrx exactly (see prep.cu):
//   TF32: elements exact up to 2048, base 2048, 2 digits per norm, f32 accumulator
//   BF16: elements exact up to 256,  base 256,  3 digits per norm, f32 accumulator
//   F16:  elements exact up to 2048, base 2048, 2 digits per norm, f32 accumulator
//   F16H: the F16 operands with an f16 accumulator, only when the whole operand
//         row fits one K = 16 MMA (so the exact integer sum is rounded to f16
//         once); chosen only when the caller opts in (DBSCAN_PATH_F16_ACC16):
//         that the tensor core forms the K = 16 sum exactly before its one
//         rounding is not documented, only observed on GB300 by the tests
// plus nt digits of thrx (1..3; at most 2 for F16 and F16H, whose largest
// power is B).
enum TcKind { TC_NONE = 0, TC_TF32 = 1, TC_BF16 = 2, TC_F16 = 3, TC_F16H = 4 };
constexpr int TC_NKINDS = 4;
// Allowed-path mask passed from the host: the DBSCAN_PATH_* bits of dbscan.h.
enum {
    TC_ALLOW_TF32 = DBSCAN_PATH_TF32,
    TC_ALLOW_BF16 = DBSCAN_PATH_BF16,
    TC_ALLOW_F16 = DBSCAN_PATH_F16,
    TC_ALLOW_F16H = DBSCAN_PATH_F16_ACC16
};
__host__ __device__ inline unsigned tc_allow_bit(int kind) { return 1u << (kind - 1); }
// Largest operand row the tensor-core sweep stages.  Up to 288 bytes two row
// tiles and two stages of two column tiles (plus their aux ints) fit 224 KB of
// shared memory; wider rows, up to 544 bytes (272 bf16/f16 elements: d = 256
// with its digits; 136 tf32 elements), take one row tile and stages of one
// column tile (sweep_tc.cu).
constexpr int TC_MAX_KBYTES = 544;
constexpr int TC_F16H_KBYTES = 32;   // the one K = 16 MMA of the F16H path

__host__ __device__ inline bool tc_is_f16(int kind) { return kind == TC_F16 || kind == TC_F16H; }
__host__ __device__ inline int tc_norm_digits(int kind) { return kind == TC_BF16 ? 3 : 2; }
__host__ __device__ inline int tc_kpad(int kind, int d, int nt) {
    const int used = d + 2 * tc_norm_digits(kind) + nt;
    return kind == TC_TF32 ? ((used + 7) / 8) * 8 : ((used + 15) / 16) * 16;
}
__host__ __device__ inline int tc_kbytes(int kind, int d, int nt) {
    return tc_kpad(kind, d, nt) * (kind == TC_TF32 ? 4 : 2);
}
// Whether a kind can hold the operand rows of dimension d with nt threshold digits.
__host__ __device__ inline bool tc_fits(int kind, int d, int nt) {
    if (kind == TC_F16H) return nt <= 2 && tc_kbytes(kind, d, nt) <= TC_F16H_KBYTES;
    if (kind == TC_F16) return nt <= 2 && tc_kbytes(kind, d, nt) <= TC_MAX_KBYTES;
    return tc_kbytes(kind, d, nt) <= TC_MAX_KBYTES;
}
// Digits of the threshold constant thrx (<= floor(eps2) + 1, see prep.cu)
// in the operands of a path: the host sizes the sweep's shared-memory tiles
// with this bound, the device takes the digits of the actual thrx.
__host__ __device__ inline int tc_nt_for(int kind, double thrx) {
    if (kind != TC_BF16) return thrx < 2048.0 ? 1 : (thrx < 4194304.0 ? 2 : 3);
    return thrx < 256.0 ? 1 : (thrx < 65536.0 ? 2 : 3);
}
inline int tc_nt_bound(int kind, float eps2) {
    double t = (double)eps2;
    t = t < 16777216.0 ? (double)(long long)t : t;   // floor for the values that matter
    return tc_nt_for(kind, t + 1.0);
}
// Byte offset of (row, byte k) in a 128-row K-major operand tile without
// swizzle: 8-row x 16-byte core matrices, K-adjacent ones 128 B apart,
// 8-row groups (kbytes / 16) * 128 B apart.
__host__ __device__ inline size_t umma_offset(int row, int kbyte, int kbytes) {
    return (size_t)(row >> 3) * (size_t)(kbytes >> 4) * 128 + (size_t)(kbyte >> 4) * 128 +
           (size_t)(row & 7) * 16 + (size_t)(kbyte & 15);
}

// ---- host launch wrappers (each returns cudaGetLastError()) ---------------
int order_bits(int64_t n);
cudaError_t launch_order(const void *points, int dtype, int64_t n, int d, const Work &w,
                         const Layout &L, cudaStream_t s);
cudaError_t launch_unpermute_counts(const Work &w, const Layout &L, int32_t *cnt_out,
                                    cudaStream_t s);
cudaError_t launch_tile_boxes(const Work &w, const Layout &L, int which, cudaStream_t s);
cudaError_t launch_prep(const void *points, int dtype, int64_t n, int d, float eps, int allow_tc,
                        const Work &w, const Layout &L, cudaStream_t s);
// launch_prep in two parts: statistics, setup and the locality order (perm);
// then the staged points and operand rows in that order.
cudaError_t launch_prep_order(const void *points, int dtype, int64_t n, int d, float eps, int allow_tc,
                              const Work &w, const Layout &L, cudaStream_t s);
cudaError_t launch_prep_stage(const void *points, int dtype, int64_t n, int d, const Work &w,
                              const Layout &L, cudaStream_t s);
cudaError_t launch_stage_umma(const Work &w, const Layout &L, int which, cudaStream_t s);
cudaError_t launch_count(const Work &w, const Layout &L, cudaStream_t s);
cudaError_t launch_compact(const Work &w, const Layout &L, int min_pts,
                           int32_t *labels, uint8_t *is_core, cudaStream_t s);
cudaError_t launch_union(const Work &w, const Layout &L, cudaStream_t s);
cudaError_t launch_flatten(const Work &w, const Layout &L, int32_t *labels, cudaStream_t s);
cudaError_t launch_border(const Work &w, const Layout &L, int32_t *labels, cudaStream_t s);
cudaError_t launch_finalize(const Work &w, const Layout &L, int32_t *labels, cudaStream_t s);
// Sharding: unite every core position with every rank's union-find parent of
// it (gathered: world arrays of stride ints).
cudaError_t launch_merge_forests(const Work &w, const Layout &L, const int *gathered, int64_t stride,
                                 int world, cudaStream_t s);

cudaError_t launch_count_tc(const Work &w, const Layout &L, cudaStream_t s);
// Tensor-core union over the tile pairs (rb, t) of the upper triangle with
// blo <= t - rb < bhi (bhi < 0: no upper limit), one work unit per row block.
cudaError_t launch_union_tc_band(const Work &w, const Layout &L, int band, int blo, int bhi,
                                 cudaStream_t s);
cudaError_t launch_border_tc(const Work &w, const Layout &L, int32_t *labels, cudaStream_t s);

int persistent_ctas(const void *kernel, int threads, size_t smem);

// Fused single-launch pipeline (fused.cu): every stage in one cooperative
// kernel, for problems small enough that launches dominate the multi-kernel
// path.  cnt_out != NULL: counts only.  The control block and the statistics
// arrays after it must be zero, and the counts array too.  Size limits from
// GB300 measurements (the fused call against the multi-kernel call, both
// replayed from graphs): faster up to ~5k points at d <= 4 and ~8k at d = 16.
constexpr int64_t FUSED_MAX_N_LOW_D = 4096;   // d <= 4
constexpr int64_t FUSED_MAX_N = 8192;         // 4 < d <= FUSED_MAX_D
constexpr int FUSED_MAX_D = 32;
bool fused_eligible(int64_t n, int d);
cudaError_t launch_fused(const void *points, int dtype, int64_t n, int d, float eps, int min_pts,
                         int32_t *labels, uint8_t *is_core, int32_t *cnt_out, const Work &w,
                         const Layout &L, cudaStream_t s);

// dbscan_fit_ex with a caller workspace, its kernels always launched directly
// (no graph capture or instantiation): the body of dbscan_fit_noalloc.
int fit_direct(const void *points, int32_t dtype, int64_t n, int32_t d, float eps, int32_t min_pts,
               int32_t *labels, uint8_t *is_core, void *workspace, size_t workspace_bytes,
               void *stream);

// Label compaction (labels.cu): scratch bytes for n labels; the ranking passes
// (*k_err points at the cluster count and the error flag in the scratch); the
// mapping pass.
size_t compact_labels_scratch(int64_t n);
cudaError_t launch_compact_labels_rank(const int32_t *labels, int64_t n, void *scratch, int **k_err,
                                       cudaStream_t s);
cudaError_t launch_compact_labels_map(const int32_t *labels, int64_t n, const void *scratch,
                                      int32_t *out, cudaStream_t s);

// ---- device helpers --------------------------------------------------------
__device__ __forceinline__ void set_error(Ctrl *c, int code) {
    atomicCAS(&c->err, 0, code);
}

// Element e of the caller's row-major point array.
__device__ __forceinline__ float load_point(const void *p, int dtype, size_t e) {
    if (dtype == DBSCAN_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[e]);
    return reinterpret_cast<const float *>(p)[e];
}

// Monotone map float -> int so that integer min/max order equals float order.
__device__ __forceinline__ int float_key(float f) {
    int b = __float_as_int(f);
    return b >= 0 ? b : (b ^ 0x7fffffff);
}
__device__ __forceinline__ float key_float(int k) {
    return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff));
}

}  // namespace dbscan
