/*
 * dbscan.h -- C ABI of the GB300 DBSCAN library (libdbscan_gb300.so).
 *
 * What it computes ("Design and optimization of DBSCAN Algorithm based on
 * CUDA", Wang et al.):
 *   - §II "Background": the eps-neighbourhood of a point is every point within
 *     distance eps of it (the point itself included); a point is a core point
 *     when at least MinPts points are in its eps-neighbourhood; clusters are
 *     maximal sets connected by reachability, which only passes through core
 *     points.
 *   - §IV-A: distances are compared squared, against eps^2; §IV-B: a pair is a
 *     neighbour pair when distance <= eps^2 (inclusive).
 *   - §IV-B1/§IV-B2: neighbour counting is fused with the distance evaluation
 *     (no distance matrix is stored) and uses the expanded form
 *     T + P[n] - (X p_x + Y p_y + Z p_z) with per-point terms hoisted.
 *   - §IV-C: clusters are merged; here by a lock-free union-find over core
 *     pairs instead of the page's cluster matrix.
 *
 * Results (defined exactly):
 *   eps2         = (float)eps * (float)eps            (single-precision product)
 *   neighbour    : sum_k (x_ik - x_jk)^2 <= eps2, i == j included
 *   is_core[i]   = |neighbours(i)| >= min_pts
 *   labels[i]    = for a core point: the smallest core index of its cluster
 *                  (clusters = connected components of core points under the
 *                  neighbour relation);
 *                  for a non-core point with at least one core neighbour
 *                  (border point): the smallest label among the clusters of
 *                  its core neighbours;
 *                  otherwise (noise): -1.
 * The page leaves open whether a point counts itself, whether "core" is
 * ">= MinPts" or "> MinPts", and which cluster a border point shared by two
 * clusters joins; the answers above are the readings this library takes.
 *
 * Arithmetic: float32 throughout -- fp32 FMAs on CUDA cores, or tensor-core
 * MMAs (tf32, bf16 or f16 operands) with a float32 accumulator.
 * Exactness: when every coordinate is an integer and sum_k (max_k - min_k)^2
 * over the data's per-dimension ranges is below 2^24, every product and
 * partial sum the kernels form is an integer below 2^24, which float32 holds
 * exactly, and the results are exact (identical to a double-precision
 * evaluation).  Other data run on CUDA cores with the test in the direct
 * form sum_k (x_ik - x_jk)^2, uncentred: accurate to a few float32 roundings
 * of the squared distance itself and symmetric in i and j, so every pass and
 * every call decides a pair the same way; only pairs whose squared distance
 * lies within that rounding (about 1e-6 relative) of eps2 may be classified
 * either way.  (The opt-in DBSCAN_PATH_F16_ACC16 path is the one exception to
 * float32 accumulation; see dbscan_set_options.)
 *
 * Memory: every pointer argument is a DEVICE pointer unless the entry point's
 * name ends in _host.  The caller owns all buffers; the library never frees
 * or retains them.  points is row-major [n, d] and contiguous.
 *
 * Streams: a stream argument is a cudaStream_t passed as void* (NULL = the
 * legacy default stream).
 *
 * Errors: every entry point returns a dbscan_status.  On error the outputs
 * are undefined.  Errors found on the device (non-finite input, an internal
 * iteration cap) are recorded in the workspace and returned by the
 * synchronous entry points, or by dbscan_workspace_status().
 */
#ifndef DBSCAN_GB300_H
#define DBSCAN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DBSCAN_OK = 0,
    DBSCAN_ERR_INVALID_ARG = -1,  /* bad size, null pointer, eps, min_pts, workspace too small, non-finite input */
    DBSCAN_ERR_UNSUPPORTED = -2,  /* n > 2^31 - 1, d > 256, bf16 with d not a multiple of 16 */
    DBSCAN_ERR_ALLOC = -3,        /* the library could not allocate its own workspace */
    DBSCAN_ERR_CUDA = -4,         /* a CUDA runtime call failed (launch, copy, sync) */
    DBSCAN_ERR_INTERNAL = -5      /* a device-side iteration cap was hit */
} dbscan_status;

typedef enum {
    DBSCAN_F32 = 0,   /* float32 points */
    DBSCAN_BF16 = 1   /* bfloat16 points (d a multiple of 16) */
} dbscan_dtype;

/* Largest supported dimension. */
#define DBSCAN_MAX_D 256

/*
 * Process-wide tuning switches.  They change how the kernels run, never what
 * they compute; every call takes a snapshot when it starts.
 *   paths   tensor-core paths the device may choose among (DBSCAN_PATH_* bits);
 *           the device takes the first one the data allow, in the order
 *           F16_ACC16 (only when set), BF16, F16, TF32, else fp32 FMAs on CUDA
 *           cores (always allowed; paths = 0 forces them).  A path is taken
 *           only when its operands hold the data exactly (integer coordinates,
 *           ranges within the element type, sums below 2^24).
 *   rows    row blocks per work unit of the tensor-core count, union and
 *           border sweeps: 0 automatic, 1 or 2
 *   graphs  1: replay repeated calls from CUDA graphs (see dbscan_fit_ex);
 *           0: launch every kernel directly
 *   fused   1: small problems -- at most 4,096 points with d <= 4, or 8,192
 *           points with 4 < d <= 32 -- run as one fused, cooperative launch
 *           whose grid-wide phases do every stage (CUDA cores, input order);
 *           0: always the multi-kernel path
 *   cull    1: the union and border sweeps (and dbscan_fit_culled's count)
 *           skip tile pairs whose bounding boxes prove that they hold no
 *           pair the sweep would accept; 0: every sweep visits every tile
 *           pair (for checking that the tile test changes nothing)
 * DBSCAN_PATH_F16_ACC16 is an opt-in: f16 operands with an f16 accumulator
 * (one K = 16 MMA per tile pair, d <= 10).  Its integer sum is rounded to f16
 * once, which keeps the sign the sweep reads -- provided the tensor core forms
 * the K = 16 sum exactly before that rounding.  NVIDIA does not document the
 * internal width of that sum; the library's tests observe it on GB300 only.
 * Defaults: paths = DBSCAN_PATHS_DEFAULT, rows automatic, graphs on, fused
 * on, cull on; the environment variables DBSCAN_FORCE_PATH (fp32, tf32, bf16,
 * f16, f16acc16), DBSCAN_TC_ROWS (one digit, or three for count, union,
 * border), DBSCAN_GRAPHS, DBSCAN_FUSED and DBSCAN_CULL (0 = off) override the defaults,
 * read once per process at the first call into the library.  Start from
 * dbscan_get_options when changing one switch.
 */
#define DBSCAN_PATH_TF32 1u
#define DBSCAN_PATH_BF16 2u
#define DBSCAN_PATH_F16 4u        /* f16 operands, f32 accumulator */
#define DBSCAN_PATH_F16_ACC16 8u  /* f16 operands, f16 accumulator (opt-in) */
#define DBSCAN_PATHS_DEFAULT (DBSCAN_PATH_TF32 | DBSCAN_PATH_BF16 | DBSCAN_PATH_F16)
typedef struct {
    uint32_t paths;
    int32_t rows[3];
    int32_t graphs;
    int32_t fused;
    int32_t cull;
} dbscan_options;

/* Replace the switches (NULL restores the defaults above, environment
 * included).  DBSCAN_ERR_INVALID_ARG for unknown path bits, a rows entry
 * outside 0..2, or graphs, fused or cull outside 0..1. */
int dbscan_set_options(const dbscan_options *opt);
/* The switches in force (host pointer). */
int dbscan_get_options(dbscan_options *opt);

/*
 * Full DBSCAN on float32 device points; synchronous on the legacy default
 * stream.  Allocates and frees its own workspace (stream-ordered).
 *   points      [n, d] float32, device, read only
 *   labels_out  [n] int32, device, written
 *   is_core_out [n] uint8 (0/1), device, written
 * n == 0 is a no-op returning DBSCAN_OK.
 * Cites: §II definitions, §IV-A/§IV-B neighbour test, §IV-C merge step.
 */
int dbscan_fit(const float *points, int64_t n, int32_t d, float eps,
               int32_t min_pts, int32_t *labels_out, uint8_t *is_core_out);

/*
 * Full DBSCAN, asynchronous on `stream` when a workspace is supplied.
 *   points      [n, d] of `dtype` (dbscan_dtype), device
 *   workspace   device buffer of at least dbscan_workspace_size(n, d, dtype)
 *               bytes (256-byte aligned), owned by the caller, reused freely
 *               between calls that do not overlap on the GPU; or NULL, in
 *               which case the library allocates one stream-ordered, frees
 *               it, and synchronises `stream` before returning so that
 *               device-side errors can be reported.
 * With a caller workspace nothing waits for the GPU: host-side argument
 * errors and launch errors are returned, device-side errors are read later
 * with dbscan_workspace_status().
 * Graph replay: with a caller workspace on a stream other than the legacy
 * default stream, the first call with a given set of arguments (pointers,
 * sizes, eps, min_pts, device) is captured into a CUDA graph, and later calls
 * with the same arguments replay it; the graph reads whatever the buffers
 * hold at replay, so results are those of a direct call.  The same holds for
 * dbscan_fit_culled and dbscan_neighbor_counts.  Not while the stream is
 * being captured by the caller or stage profiling is on, nor with the
 * graphs switch off (dbscan_set_options).  At most 16 graphs are kept; the
 * least recently used one is destroyed to make room (an instance still
 * running is freed when it completes).
 * Cites: §II, §IV-A, §IV-B, §IV-B1, §IV-B2, §IV-C.
 */
int dbscan_fit_ex(const void *points, int32_t dtype, int64_t n, int32_t d,
                  float eps, int32_t min_pts, int32_t *labels_out,
                  uint8_t *is_core_out, void *workspace,
                  size_t workspace_bytes, void *stream);

/*
 * dbscan_fit_ex with tile culling: the same arguments, workspace and error
 * behaviour, and the same labels and core flags.  The sweeps skip every pair
 * of 128-point tiles whose bounding boxes (of the points in the library's
 * locality order) are eps or more apart: no pair in such tiles can be a
 * neighbour, so for integer data within the exactness bound the result is
 * identical to dbscan_fit_ex.  This is not an all-pairs evaluation (pairs in
 * skipped tiles are never evaluated), which is why it is a separate entry
 * point.  Culling applies for d <= 64 with the cull switch on, otherwise the
 * call runs exactly as dbscan_fit_ex.  For integer data within the exactness
 * bound the box test is exact; for other data (CUDA-core path) it keeps every
 * tile pair within eps plus a bound on the float test's rounding, so it never
 * drops a pair that the unculled sweep would accept.  (dbscan_fit_ex itself
 * applies the same test in its union and border passes, which act only on
 * neighbour pairs; its count pass evaluates every pair.)  The pages evaluate all
 * pairs ("Design and optimization of DBSCAN Algorithm based on CUDA", §IV-A);
 * pruning by spatial bounds is not on them.
 */
int dbscan_fit_culled(const void *points, int32_t dtype, int64_t n, int32_t d,
                      float eps, int32_t min_pts, int32_t *labels_out,
                      uint8_t *is_core_out, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * Full DBSCAN on HOST buffers: copies points in, runs, copies the results
 * out and synchronises `stream`.  Device memory is allocated stream-ordered
 * for the call and freed before returning.  Host buffers may be pageable or
 * pinned (pinned copies are faster).
 *   points_host      [n, d] of `dtype`, host
 *   labels_host      [n] int32, host
 *   is_core_host     [n] uint8, host
 */
int dbscan_fit_host(const void *points_host, int32_t dtype, int64_t n,
                    int32_t d, float eps, int32_t min_pts,
                    int32_t *labels_host, uint8_t *is_core_host,
                    void *stream);

/*
 * Cluster labels renumbered 0..k-1 in increasing order of label (the order of
 * each cluster's smallest core index); noise stays -1.  An optional output:
 * the pages name clusters by the columns of their cluster matrix
 * ("Design and optimization of DBSCAN Algorithm based on CUDA", §IV-B) and
 * fix no numbering.
 *   labels           [n] int32, device: labels as dbscan_fit* writes them --
 *                    -1, or the index of a point whose own label is that index
 *   labels_out       [n] int32, device; may equal labels (in place)
 *   n_clusters       host int32: k, written on success
 * Synchronises `stream`; scratch memory is allocated stream-ordered for the
 * call.  Labels that dbscan_fit* cannot have produced (a label that is not -1
 * and not the index of a point labelled with itself) give
 * DBSCAN_ERR_INVALID_ARG, and labels_out is then left untouched.  n = 0 sets
 * k = 0; n > 2^31 - 1 gives DBSCAN_ERR_UNSUPPORTED.
 */
int dbscan_compact_labels(const int32_t *labels, int64_t n, int32_t *labels_out,
                          int32_t *n_clusters, void *stream);

/*
 * Neighbour counts only (the fused distance + count step, §IV-B1/§IV-B2):
 *   cnt_out[i] = |{ j : sum_k (x_ik - x_jk)^2 <= eps2 }|  (i itself included)
 * cnt_out is [n] int32, device.  Workspace rules as for dbscan_fit_ex
 * (the same size suffices).
 */
int dbscan_neighbor_counts(const void *points, int32_t dtype, int64_t n,
                           int32_t d, float eps, int32_t *cnt_out,
                           void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * Full DBSCAN without any device allocation.  The paper has no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc -- code
 * embedded in a host framework whose own allocator has reserved the device
 * memory (an allocation of ours could fail or fragment its pool), or serving
 * paths that must not allocate after start-up because an allocation can
 * synchronise the device.  It runs exactly what dbscan_fit_ex runs, with the
 * workspace taken from a static device array of DBSCAN_NOALLOC_SCRATCH_BYTES
 * (64 MiB) that every GPU which loads this library holds until the process
 * exits.
 *   points, labels_out, is_core_out: as for dbscan_fit_ex (device pointers).
 *   stream: cudaStream_t as void*, NULL = legacy default stream; asynchronous.
 * Limits and rules:
 *   - problems whose dbscan_workspace_size(n, d, dtype) exceeds
 *     DBSCAN_NOALLOC_SCRATCH_BYTES are rejected with DBSCAN_ERR_UNSUPPORTED
 *     (about 285,000 points at d = 3, 57,000 at d = 64);
 *   - the first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any
 *     stream capture;
 *   - every call shares the one array and each call clears the parts that
 *     must start at zero, so calls that overlap on the GPU (different streams,
 *     different host threads) race and must be serialised by the caller;
 *   - device-side errors are not reported (there is no workspace handle to
 *     read them from); host-side argument errors are returned as usual;
 *   - it never captures or instantiates a CUDA graph (graph instantiation
 *     takes device resources): its kernels are always launched directly.
 */
#define DBSCAN_NOALLOC_SCRATCH_BYTES (64u << 20)
int dbscan_fit_noalloc(const void *points, int32_t dtype, int64_t n, int32_t d,
                       float eps, int32_t min_pts, int32_t *labels_out,
                       uint8_t *is_core_out, void *stream);

/*
 * Sharded DBSCAN across `world` processes, one GPU each (rank = this
 * process's index).  The pages run one GPU; the split follows the row-block
 * partition of the upper triangle: every rank holds all points and stages
 * them in one locality order, while the count, union and border sweeps take
 * only the work units u with u % world == rank.  The caller runs five stages
 * on the same workspace and, between them, four collectives over all ranks
 * (NCCL, say):
 *   stage 0  statistics and the locality order              (points)
 *            -> broadcast from rank 0 the int32 array DBSCAN_SHARD_ORDER
 *               (the order's counting sort places points within a bin in
 *               atomic order, so ranks must share one order)
 *   stage 1  staging + this rank's share of the count        (points)
 *            -> all-reduce SUM over the int32 array DBSCAN_SHARD_COUNTS
 *   stage 2  core flags (is_core_out written) + this rank's share of the
 *            union-find over core pairs                      (labels_out, is_core_out)
 *            -> all-gather the int32 array DBSCAN_SHARD_PARENTS of every rank
 *               into a device array [world, n] (rank order)
 *   stage 3  merge of all ranks' forests, core labels, this rank's share of
 *            the border assignment                           (gathered_parents, labels_out)
 *            -> all-reduce MIN over labels_out (n int32)
 *   stage 4  finalize                                        (labels_out)
 * Arguments not used by a stage may be NULL; n, d, dtype, eps, min_pts, rank
 * and world must be the same at every stage and on every rank (points too).
 * The workspace (dbscan_workspace_size bytes, required) carries the state
 * between stages.  Every stage is asynchronous on `stream` and launches its
 * kernels directly; device-side errors: dbscan_workspace_status.  With
 * world = 1 and no collectives the stages give dbscan_fit_ex's results.
 * The tuning switches in force must not change between stages (the fused
 * small-problem pipeline is never used here).
 */
#define DBSCAN_SHARD_COUNTS 0
#define DBSCAN_SHARD_PARENTS 1
#define DBSCAN_SHARD_ORDER 2
int dbscan_fit_shard(int32_t stage, const void *points, int32_t dtype, int64_t n, int32_t d,
                     float eps, int32_t min_pts, int32_t rank, int32_t world,
                     const int32_t *gathered_parents, int32_t *labels_out,
                     uint8_t *is_core_out, void *workspace, size_t workspace_bytes,
                     void *stream);
/* Device address and length (ints) of a workspace array the caller combines
 * across ranks between stages (which: DBSCAN_SHARD_ORDER, DBSCAN_SHARD_COUNTS
 * or DBSCAN_SHARD_PARENTS); n and d as for the stages.  Pure host
 * computation. */
int dbscan_shard_buffer(void *workspace, int64_t n, int32_t d, int32_t which, void **ptr,
                        int64_t *count);

/* Bytes of workspace dbscan_fit_ex needs for this problem shape; 0 when the
 * shape is invalid or unsupported.  Pure host computation. */
size_t dbscan_workspace_size(int64_t n, int32_t d, int32_t dtype);

/* Synchronises `stream`, then returns the first device-side error recorded in
 * `workspace` by the last call that used it (DBSCAN_OK if none). */
int dbscan_workspace_status(const void *workspace, void *stream);

/*
 * Facts about the last call that used `workspace` (synchronises `stream`
 * first).  Fills up to n of, in this order:
 *   0  arithmetic path of the sweeps: 0 CUDA-core fp32, 1 tf32 tensor cores,
 *      2 bf16 tensor cores, 3 f16 tensor cores (f32 accumulator), 4 f16
 *      tensor cores with the opt-in f16 accumulator (all others accumulate
 *      in float32)
 *   1  number of core points
 *   2  number of border candidates (non-core points with a neighbour
 *      besides themselves)
 *   3  1 when every coordinate was an integer and sum_k (max_k - min_k)^2 <
 *      2^24, i.e. the results are exact (see "Exactness" above), else 0
 *   4  padded operand width K of the tensor-core path (0 on CUDA cores)
 *   5  1 when the call ran as the fused single-launch pipeline (fp32 FMAs
 *      on CUDA cores), else 0
 * info is a host pointer to n int64 values.  Returns DBSCAN_OK,
 * DBSCAN_ERR_INVALID_ARG for a NULL pointer or n < 1, or DBSCAN_ERR_CUDA.
 */
int dbscan_workspace_info(const void *workspace, void *stream, int64_t *info, int32_t n);

/*
 * Stage timing (measurement support, not part of the computation).
 * Between dbscan_profile_begin() and dbscan_profile_end(), every call made
 * on the same host thread records CUDA events on its own stream around its
 * stages.  dbscan_profile_end() waits for those events and returns, summed
 * over the calls, the milliseconds of each stage in the order
 *   0 prep, 1 count, 2 compact, 3 union, 4 flatten, 5 border, 6 finalize
 * (stage_ms has room for max_stages floats; a stage a call did not run adds
 * 0), the number of calls and the number of kernels they launched.
 * Pointers are host pointers and may be NULL.  Returns DBSCAN_OK, or
 * DBSCAN_ERR_CUDA if an event could not be created or read.
 */
#define DBSCAN_NUM_STAGES 7
int dbscan_profile_begin(void);
int dbscan_profile_end(float *stage_ms, int32_t max_stages, int64_t *calls,
                       int64_t *kernel_launches);

/* Static, human-readable name of a status code. */
const char *dbscan_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* DBSCAN_GB300_H */
