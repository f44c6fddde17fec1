// C ABI of the DBSCAN library: argument validation, workspace layout and the
// order of the kernel stages.
//
// Stage order ("Design and optimization of DBSCAN Algorithm based on CUDA",
// §I lists the three GPU steps: all-pair distances, core points + primitive
// clusters, merging):
//   prep     ranges, centring, norms, thresholds, tiled staging      O(N d)
//   count    fused distance + neighbour count over the upper
//            triangle of tiles (§IV-B1, §IV-B2)                      O(N^2 d)
//   compact  core flags, stable compaction of cores and candidates   O(N)
//   union    core-core sweep hooking a lock-free union-find          O(Nc^2 d)
//   flatten  labels of core points                                   O(Nc)
//   border   candidates x cores, smallest neighbouring label         O(Nb Nc d)
//   finalize candidates without a core neighbour become noise        O(Nb)
// Nothing of size N x N is ever stored.
#include "dbscan_internal.cuh"
#include "tc_schedule.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <list>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <tuple>
#include <vector>

namespace dbscan {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Layout make_layout(int64_t n, int32_t d) {
    Layout L{};
    L.n = n;
    L.d = d;
    L.rank = 0;
    L.world = 1;
    L.ntiles = (n + BT - 1) / BT;
    L.tile_floats = (size_t)(d + 1) * BT;
    const size_t staged = (size_t)L.ntiles * L.tile_floats * sizeof(float);
    const size_t per_pt = (size_t)L.ntiles * BT * sizeof(float);
    L.nscan_blocks = (n + SCAN_BLOCK - 1) / SCAN_BLOCK;
    size_t off = 0;
    L.off_ctrl = off;        off += align256(sizeof(Ctrl));
    L.off_stats = off;       off += align256((size_t)3 * DBSCAN_MAX_D * sizeof(int));
    L.off_staged_all = off;  off += align256(staged);
    L.off_staged_core = off; off += align256(staged);
    L.off_staged_cand = off; off += align256(staged);
    L.off_T_all = off;       off += align256(per_pt);
    L.off_T_core = off;      off += align256(per_pt);
    L.off_T_cand = off;      off += align256(per_pt);
    L.off_cnt = off;         off += align256(per_pt);
    L.off_cidx = off;        off += align256(per_pt);
    L.off_candidx = off;     off += align256(per_pt);
    L.off_parent = off;      off += align256(per_pt);
    L.off_clabel = off;      off += align256(per_pt);
    L.off_bsum = off;        off += align256((size_t)2 * (L.nscan_blocks + 1) * sizeof(int));
    // tensor-core operand tiles, sized for the largest path this shape allows
    size_t kb = 0;
    for (int kind = TC_TF32; kind <= TC_NKINDS; ++kind) {
        const int nt = tc_is_f16(kind) ? 2 : 3;   // the most threshold digits a kind takes
        const int b = tc_kbytes(kind, d, nt);
        if (tc_fits(kind, d, nt) && (size_t)b > kb) kb = (size_t)b;
    }
    L.umma_tile_bytes = (size_t)BT * kb;
    const size_t umma = (size_t)L.ntiles * L.umma_tile_bytes;
    // Row and column operand arrays.  The all-point operands die with the
    // count sweep, the core row operands with the union sweep, so the core
    // operands reuse the all-point arrays and the candidate rows (staged after
    // the union) reuse the row array.
    L.off_ua_all = off;      off += align256(umma);
    L.off_ub_all = off;      off += align256(umma);
    L.off_ua_core = L.off_ua_all;
    L.off_ub_core = L.off_ub_all;
    L.off_ua_cand = L.off_ua_all;
    // locality order
    L.order_bits = order_bits(n);
    const size_t nbins = (size_t)1 << L.order_bits;
    L.off_bin = off;         off += align256((size_t)n * sizeof(int));
    L.off_perm = off;        off += align256(per_pt);
    L.off_hist = off;        off += align256(nbins * sizeof(int));
    L.off_bstart = off;      off += align256(nbins * sizeof(int));
    L.off_btot = off;        off += align256((nbins / 1024 + 1) * sizeof(int));
    L.off_rootmin = off;     off += align256(per_pt);
    // tile bounding boxes for culling (three arrays: all, core, candidates)
    L.box_floats = d <= CULL_MAX_D ? (size_t)L.ntiles * 2 * d : 0;
    L.gbox_floats = d <= CULL_MAX_D ? (size_t)((L.ntiles + CULL_GROUP - 1) / CULL_GROUP) * 2 * d : 0;
    L.off_box_all = off;     off += align256(L.box_floats * sizeof(float));
    L.off_box_core = off;    off += align256(L.box_floats * sizeof(float));
    L.off_box_cand = off;    off += align256(L.box_floats * sizeof(float));
    L.off_gbox_all = off;    off += align256(L.gbox_floats * sizeof(float));
    L.off_gbox_core = off;   off += align256(L.gbox_floats * sizeof(float));
    L.off_troot = off;       off += align256((size_t)L.ntiles * sizeof(int));
    L.off_pivrank = off;     off += align256(512 * sizeof(int));
    L.total = off;
    return L;
}

// ---- tuning switches -----------------------------------------------------
// Process-wide, read from the environment once (at the first call) and
// replaced with dbscan_set_options; every call works on a snapshot.
static std::mutex g_opt_mu;
static bool g_opt_init = false;
static dbscan_options g_opt;

static dbscan_options options_from_env() {
    dbscan_options o{};
    o.paths = DBSCAN_PATHS_DEFAULT;
    o.graphs = 1;
    const char *f = getenv("DBSCAN_FORCE_PATH");
    if (f && *f) {
        if (!strcmp(f, "fp32")) o.paths = 0;
        else if (!strcmp(f, "tf32")) o.paths = DBSCAN_PATH_TF32;
        else if (!strcmp(f, "bf16")) o.paths = DBSCAN_PATH_BF16;
        else if (!strcmp(f, "f16")) o.paths = DBSCAN_PATH_F16;
        else if (!strcmp(f, "f16acc16")) o.paths = DBSCAN_PATH_F16_ACC16;
    }
    if (const char *r = getenv("DBSCAN_TC_ROWS")) {
        const size_t len = strlen(r);
        for (int m = 0; m < 3; ++m) {
            const char c = len == 1 ? r[0] : (len == 3 ? r[m] : '0');
            o.rows[m] = (c == '1' || c == '2') ? c - '0' : 0;
        }
    }
    const char *g = getenv("DBSCAN_GRAPHS");
    if (g && g[0] == '0') o.graphs = 0;
    o.fused = 1;
    const char *fu = getenv("DBSCAN_FUSED");
    if (fu && fu[0] == '0') o.fused = 0;
    o.cull = 1;
    const char *cu = getenv("DBSCAN_CULL");
    if (cu && cu[0] == '0') o.cull = 0;
    return o;
}

static dbscan_options options_snapshot() {
    std::lock_guard<std::mutex> lock(g_opt_mu);
    if (!g_opt_init) {
        g_opt = options_from_env();
        g_opt_init = true;
    }
    return g_opt;
}

// Tensor-core kinds a call may take: the allowed paths whose operand rows fit
// dimension d with the threshold digits eps allows.
static unsigned allowed_tc(int d, float eps2, unsigned paths) {
    unsigned allow = 0;
    for (int kind = TC_TF32; kind <= TC_NKINDS; ++kind)
        if ((paths & tc_allow_bit(kind)) && tc_fits(kind, d, tc_nt_bound(kind, eps2)))
            allow |= tc_allow_bit(kind);
    return allow;
}

// The layout of one call: sizes plus eps, the culling switches and the
// tuning switches in force.  Union and border act only on neighbour pairs,
// all of which the count sweep has evaluated; they skip tile pairs that the
// box test proves hold none (exact data only, checked on the device).  The
// count sweep itself evaluates every pair unless the caller asked for culling.
static Layout call_layout(int64_t n, int32_t d, float eps, int cull, const dbscan_options &o) {
    Layout L = make_layout(n, d);
    L.eps2 = eps * eps;
    L.allow = L.umma_tile_bytes ? allowed_tc(d, L.eps2, o.paths) : 0u;
    for (int m = 0; m < 3; ++m) L.rows[m] = o.rows[m];
    L.fused = o.fused && fused_eligible(n, d);
    L.cull_nbr = L.box_floats > 0 && L.umma_tile_bytes > 0 && o.cull;
    L.cull = cull && L.cull_nbr;
    return L;
}

Work carve(void *base, const Layout &L) {
    char *b = static_cast<char *>(base);
    Work w{};
    w.ctrl = reinterpret_cast<Ctrl *>(b + L.off_ctrl);
    w.stat_min = reinterpret_cast<int *>(b + L.off_stats);
    w.stat_max = w.stat_min + DBSCAN_MAX_D;
    w.centre = reinterpret_cast<float *>(w.stat_max + DBSCAN_MAX_D);
    w.staged_all = reinterpret_cast<float *>(b + L.off_staged_all);
    w.staged_core = reinterpret_cast<float *>(b + L.off_staged_core);
    w.staged_cand = reinterpret_cast<float *>(b + L.off_staged_cand);
    w.T_all = reinterpret_cast<float *>(b + L.off_T_all);
    w.T_core = reinterpret_cast<float *>(b + L.off_T_core);
    w.T_cand = reinterpret_cast<float *>(b + L.off_T_cand);
    w.cnt = reinterpret_cast<int *>(b + L.off_cnt);
    w.cidx = reinterpret_cast<int *>(b + L.off_cidx);
    w.candidx = reinterpret_cast<int *>(b + L.off_candidx);
    w.parent = reinterpret_cast<int *>(b + L.off_parent);
    w.clabel = reinterpret_cast<int *>(b + L.off_clabel);
    w.bsum = reinterpret_cast<int *>(b + L.off_bsum);
    w.ua_all = reinterpret_cast<uint8_t *>(b + L.off_ua_all);
    w.ub_all = reinterpret_cast<uint8_t *>(b + L.off_ub_all);
    w.ua_core = reinterpret_cast<uint8_t *>(b + L.off_ua_core);
    w.ub_core = reinterpret_cast<uint8_t *>(b + L.off_ub_core);
    w.ua_cand = reinterpret_cast<uint8_t *>(b + L.off_ua_cand);
    w.bin = reinterpret_cast<int *>(b + L.off_bin);
    w.perm = reinterpret_cast<int *>(b + L.off_perm);
    w.hist = reinterpret_cast<int *>(b + L.off_hist);
    w.bstart = reinterpret_cast<int *>(b + L.off_bstart);
    w.btot = reinterpret_cast<int *>(b + L.off_btot);
    w.rootmin = reinterpret_cast<int *>(b + L.off_rootmin);
    w.troot = reinterpret_cast<int *>(b + L.off_troot);
    w.pivrank = reinterpret_cast<int *>(b + L.off_pivrank);
    w.box_all = reinterpret_cast<float *>(b + L.off_box_all);
    w.box_core = reinterpret_cast<float *>(b + L.off_box_core);
    w.box_cand = reinterpret_cast<float *>(b + L.off_box_cand);
    w.gbox_all = reinterpret_cast<float *>(b + L.off_gbox_all);
    w.gbox_core = reinterpret_cast<float *>(b + L.off_gbox_core);
    return w;
}

// Host-side checks that need no GPU.
static int check_shape(int64_t n, int32_t d, int32_t dtype) {
    if (n < 0 || d < 1) return DBSCAN_ERR_INVALID_ARG;
    if (dtype != DBSCAN_F32 && dtype != DBSCAN_BF16) return DBSCAN_ERR_INVALID_ARG;
    if (n > 0x7fffffffLL) return DBSCAN_ERR_UNSUPPORTED;
    if (d > DBSCAN_MAX_D) return DBSCAN_ERR_UNSUPPORTED;
    if (dtype == DBSCAN_BF16 && (d % 16) != 0) return DBSCAN_ERR_UNSUPPORTED;
    return DBSCAN_OK;
}

static int check_scalars(float eps, int32_t min_pts) {
    if (!(eps >= 0.f) || isinf(eps)) return DBSCAN_ERR_INVALID_ARG;
    if (min_pts < 1) return DBSCAN_ERR_INVALID_ARG;
    return DBSCAN_OK;
}

// A kernel given a host pointer would fault; reject anything the device
// cannot address as device or managed memory.
static int check_device_ptr(const void *p) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return DBSCAN_ERR_INVALID_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return DBSCAN_ERR_INVALID_ARG;
    return DBSCAN_OK;
}

// Keep freed stream-ordered allocations in the device's pool between calls
// (once per device, for this process only).
static void keep_pool(void) {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(dev)) return;
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
        uint64_t thr = 8ull << 30;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    }
    done.insert(dev);
}

// ---- stage timing ------------------------------------------------------------
// Kernels each stage launches.  Every sweep launches its two CUDA-core
// kernels (one per form of the neighbour test) and one kernel per
// tensor-core kind the call allows (ntc: the allowed paths whose operand rows
// fit the shape); all but the one the data select on the device return at
// once.  The per-stage counts are in the switch below.
int union_band_count(int64_t ntiles);   // sweep.cu

static int stage_launches(unsigned allow, int d, int64_t ntiles, int stage) {
    const int ntc = __builtin_popcount(allow);
    const int nb = union_band_count(ntiles);
    const int umma = ntc > 0 ? 1 : 0;
    switch (stage) {
    // (+2: pivot renumbering and assignment of the order for 3 < d <= 64)
    case 0: return 9 + umma + (d > 3 && d <= 64 ? 2 : 0);
    // (each CUDA-core sweep: one launch per form of the neighbour test)
    case 1: return 2 + ntc;
    case 2: return 4 + umma;
    // tile-local union, then per band on CUDA cores (three): the sweep (two
    // forms), a tile-root snapshot and (after the first) a compression, and
    // per tensor-core band (nb): a launch per kind, a tile-root snapshot and
    // (after the first) a compression
    case 3: return 1 + UNION_BANDS * 3 + (UNION_BANDS - 1) + nb * (ntc + 1) + (nb - 1);
    case 4: return 2;
    case 5: return umma + 2 + ntc;
    default: return 1;
    }
}

struct ProfCall {
    cudaEvent_t ev[DBSCAN_NUM_STAGES + 1];
    int stages;       // number of stages the call ran
    unsigned allow;   // tensor-core kinds launched by the call's sweeps
    int d;            // dimension (the order's pivot kernels run for 3 < d <= 64)
    int64_t ntiles;   // tiles of the call (the union's band count)
    int cull;         // 1: culled count, 2: culled union and border (box kernels)
    int fused;        // 1: the fused single-launch pipeline (one kernel)
};
struct ProfState {
    bool on = false;
    bool failed = false;
    std::vector<ProfCall> calls;
};
static thread_local ProfState g_prof;

struct StageMarks {
    ProfCall call{};
    bool on = false;
    int next = 0;
    StageMarks(cudaStream_t s, unsigned allow, int d, int64_t ntiles, int cull, int fused) {
        call.allow = allow;
        call.d = d;
        call.ntiles = ntiles;
        call.cull = cull;
        call.fused = fused;
        if (!g_prof.on) return;
        for (int i = 0; i <= DBSCAN_NUM_STAGES; ++i) {
            if (cudaEventCreate(&call.ev[i]) != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaEventDestroy(call.ev[j]);
                g_prof.failed = true;
                return;
            }
        }
        on = true;
        mark(s);
    }
    void mark(cudaStream_t s) {
        if (on && next <= DBSCAN_NUM_STAGES) cudaEventRecord(call.ev[next++], s);
    }
    void done() {
        if (!on) return;
        call.stages = next - 1;
        for (int i = next; i <= DBSCAN_NUM_STAGES; ++i) cudaEventDestroy(call.ev[i]);
        g_prof.calls.push_back(call);
        on = false;
    }
    ~StageMarks() { done(); }
};

// Launch every stage; cnt_out != NULL stops after the count and copies it out.
static int run(const void *points, int dtype, int64_t n, int d, float eps, int min_pts,
               int32_t *labels, uint8_t *is_core, int32_t *cnt_out, void *ws, const Layout &L,
               cudaStream_t s) {
    Work w = carve(ws, L);
    StageMarks marks(s, L.allow, d, L.ntiles, L.cull + 2 * L.cull_nbr, L.fused);
    if (L.fused) {
        // one launch does every stage; its time is reported under "count"
        const size_t zero = L.off_stats + 2 * DBSCAN_MAX_D * sizeof(int);   // Ctrl + min/max
        if (cudaMemsetAsync(w.ctrl, 0, zero, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
        if (cudaMemsetAsync(w.cnt, 0, (size_t)L.ntiles * BT * sizeof(int), s) != cudaSuccess)
            return DBSCAN_ERR_CUDA;
        marks.mark(s);
        if (launch_fused(points, dtype, n, d, eps, min_pts, labels, is_core, cnt_out, w, L, s) !=
            cudaSuccess)
            return DBSCAN_ERR_CUDA;
        for (int i = 0; i < DBSCAN_NUM_STAGES - 1; ++i) marks.mark(s);
        return DBSCAN_OK;
    }
    if (cudaMemsetAsync(w.ctrl, 0, sizeof(Ctrl), s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    if (cudaMemsetAsync(w.cnt, 0, (size_t)n * sizeof(int), s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    if (launch_prep(points, dtype, n, d, eps, L.allow, w, L, s) != cudaSuccess)
        return DBSCAN_ERR_CUDA;
    if (L.cull && launch_tile_boxes(w, L, 0, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    marks.mark(s);
    if (launch_count(w, L, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    marks.mark(s);
    if (cnt_out) {
        if (launch_unpermute_counts(w, L, cnt_out, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
        return DBSCAN_OK;
    }
    if (launch_compact(w, L, min_pts, labels, is_core, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    if (L.cull_nbr && (launch_tile_boxes(w, L, 1, s) != cudaSuccess ||
                       launch_tile_boxes(w, L, 2, s) != cudaSuccess))
        return DBSCAN_ERR_CUDA;
    marks.mark(s);
    if (launch_union(w, L, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    marks.mark(s);
    if (launch_flatten(w, L, labels, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    marks.mark(s);
    if (launch_stage_umma(w, L, 2, s) != cudaSuccess) return DBSCAN_ERR_CUDA;   // candidate rows
    if (launch_border(w, L, labels, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    marks.mark(s);
    if (launch_finalize(w, L, labels, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    marks.mark(s);
    return DBSCAN_OK;
}

static int read_status(const void *ws, cudaStream_t s) {
    int err = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DBSCAN_ERR_CUDA;
    if (cudaMemcpy(&err, &static_cast<const Ctrl *>(ws)->err, sizeof(int), cudaMemcpyDeviceToHost) !=
        cudaSuccess)
        return DBSCAN_ERR_CUDA;
    return err;
}

// ---- graph replay ----------------------------------------------------------
// A call is some sixty launches whose every decision is taken on the device,
// so a call on a caller's stream and workspace is captured once into a CUDA
// graph and replayed while its arguments repeat (the graph reads whatever the
// buffers hold at replay).  Keys: every argument, the device, and the tuning
// switches of the call.  Not on the legacy default stream (it cannot be
// captured), not while the stream is already capturing (the caller's own
// capture then takes the launches), not while stage profiling records
// events, not with the graphs switch off.  At most kGraphCap graphs are kept,
// the least recently used one destroyed to make room (an instance still
// running is freed when it completes).
using GraphKey = std::tuple<int, const void *, int, int64_t, int, uint32_t, int, void *, void *, void *,
                            void *, int, unsigned, int, int, int, int>;
struct GraphEntry {
    GraphKey key;
    cudaGraphExec_t exec;
};
static std::mutex g_graph_mu;
static std::list<GraphEntry> g_graph_lru;   // most recently used first
static std::map<GraphKey, std::list<GraphEntry>::iterator> g_graphs;
static std::set<GraphKey> g_graph_failed;   // keys whose capture failed: launched directly
constexpr size_t kGraphCap = 16;

static bool graphs_enabled(cudaStream_t s, const dbscan_options &o) {
    if (!o.graphs) return false;
    if (s == nullptr || s == cudaStreamLegacy || g_prof.on) return false;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cs == cudaStreamCaptureStatusNone;
}

// run() through a cached graph; -1 when the graph path does not apply.
static int run_graph(const void *points, int dtype, int64_t n, int d, float eps, int min_pts,
                     int32_t *labels, uint8_t *is_core, int32_t *cnt_out, void *ws, const Layout &L,
                     const dbscan_options &o, cudaStream_t s) {
    if (!graphs_enabled(s, o)) return -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    uint32_t eb;
    memcpy(&eb, &eps, sizeof(eb));
    const GraphKey key(dev, points, dtype, n, d, eb, min_pts, labels, is_core, cnt_out, ws,
                       L.cull + 2 * L.cull_nbr, L.allow, L.rows[0], L.rows[1], L.rows[2], L.fused);
    std::lock_guard<std::mutex> lock(g_graph_mu);
    auto it = g_graphs.find(key);
    if (it != g_graphs.end()) {
        g_graph_lru.splice(g_graph_lru.begin(), g_graph_lru, it->second);
    } else {
        if (g_graph_failed.count(key)) return -1;
        if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
            cudaGetLastError();
            if (g_graph_failed.size() < 64) g_graph_failed.insert(key);
            return -1;
        }
        const int st = run(points, dtype, n, d, eps, min_pts, labels, is_core, cnt_out, ws, L, s);
        cudaGraph_t g = nullptr;
        const cudaError_t ec = cudaStreamEndCapture(s, &g);
        cudaGraphExec_t ex = nullptr;
        const bool ok = st == DBSCAN_OK && ec == cudaSuccess && g != nullptr &&
                        cudaGraphInstantiate(&ex, g, 0) == cudaSuccess;
        if (g) cudaGraphDestroy(g);
        if (!ok) {
            cudaGetLastError();
            if (g_graph_failed.size() < 64) g_graph_failed.insert(key);
            return -1;   // launched directly instead
        }
        if (g_graphs.size() >= kGraphCap) {   // make room: drop the least recently used
            cudaGraphExecDestroy(g_graph_lru.back().exec);
            g_graphs.erase(g_graph_lru.back().key);
            g_graph_lru.pop_back();
        }
        g_graph_lru.push_front(GraphEntry{key, ex});
        it = g_graphs.emplace(key, g_graph_lru.begin()).first;
    }
    return cudaGraphLaunch(it->second->exec, s) == cudaSuccess ? DBSCAN_OK : DBSCAN_ERR_CUDA;
}

// Shared body of dbscan_fit_ex and dbscan_neighbor_counts.
// use_graph = false: launch directly, never capture (dbscan_fit_noalloc).
static int fit_common(const void *points, int32_t dtype, int64_t n, int32_t d, float eps,
                      int32_t min_pts, int32_t *labels, uint8_t *is_core, int32_t *cnt_out,
                      void *workspace, size_t workspace_bytes, void *stream, int cull = 0,
                      bool use_graph = true) {
    int st = check_shape(n, d, dtype);
    if (st != DBSCAN_OK) return st;
    if ((st = check_scalars(eps, min_pts)) != DBSCAN_OK) return st;
    if (n == 0) return DBSCAN_OK;
    if (!points) return DBSCAN_ERR_INVALID_ARG;
    if (!cnt_out && (!labels || !is_core)) return DBSCAN_ERR_INVALID_ARG;
    const dbscan_options opt = options_snapshot();
    const Layout L = call_layout(n, d, eps, cull, opt);
    if (workspace) {
        if (workspace_bytes < L.total) return DBSCAN_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(workspace) & 255) return DBSCAN_ERR_INVALID_ARG;
    }
    if (check_device_ptr(points) != DBSCAN_OK) return DBSCAN_ERR_INVALID_ARG;
    if (cnt_out) {
        if (check_device_ptr(cnt_out) != DBSCAN_OK) return DBSCAN_ERR_INVALID_ARG;
    } else {
        if (check_device_ptr(labels) != DBSCAN_OK || check_device_ptr(is_core) != DBSCAN_OK)
            return DBSCAN_ERR_INVALID_ARG;
    }
    if (workspace && check_device_ptr(workspace) != DBSCAN_OK) return DBSCAN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (workspace) {
        const int gst = use_graph ? run_graph(points, dtype, n, d, eps, min_pts, labels, is_core,
                                              cnt_out, workspace, L, opt, s)
                                  : -1;
        if (gst >= 0) return gst;
        return run(points, dtype, n, d, eps, min_pts, labels, is_core, cnt_out, workspace, L, s);
    }

    keep_pool();
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, L.total, s) != cudaSuccess) {
        cudaGetLastError();
        return DBSCAN_ERR_ALLOC;
    }
    st = run(points, dtype, n, d, eps, min_pts, labels, is_core, cnt_out, ws, L, s);
    int dev_st = read_status(ws, s);
    cudaFreeAsync(ws, s);
    if (cudaStreamSynchronize(s) != cudaSuccess && st == DBSCAN_OK) st = DBSCAN_ERR_CUDA;
    return st != DBSCAN_OK ? st : dev_st;
}

// ---- sharding across processes ----------------------------------------------
// One stage of the sharded pipeline.  Every rank stages the points in rank
// 0's locality order (the caller broadcasts it after stage 0: the order's
// counting sort places points within a bin in atomic order, so it can differ
// between ranks), and staging, compaction, flatten and finalize are then
// deterministic, so every position means the same point on every rank; the
// count, union and border sweeps take only this rank's work units.  Between
// stages the caller combines the ranks' buffers with collectives (dbscan.h,
// dbscan_fit_shard).
static int run_shard_stage(int stage, const void *points, int dtype, int64_t n, int d, float eps,
                           int min_pts, const int32_t *gathered, int32_t *labels, uint8_t *is_core,
                           void *ws, const Layout &L, cudaStream_t s) {
    Work w = carve(ws, L);
    switch (stage) {
    case 0:
        if (cudaMemsetAsync(w.ctrl, 0, sizeof(Ctrl), s) != cudaSuccess ||
            cudaMemsetAsync(w.cnt, 0, (size_t)n * sizeof(int), s) != cudaSuccess)
            return DBSCAN_ERR_CUDA;
        return launch_prep_order(points, dtype, n, d, eps, L.allow, w, L, s) == cudaSuccess
                   ? DBSCAN_OK
                   : DBSCAN_ERR_CUDA;
    case 1:
        if (launch_prep_stage(points, dtype, n, d, w, L, s) != cudaSuccess ||
            launch_count(w, L, s) != cudaSuccess)
            return DBSCAN_ERR_CUDA;
        return DBSCAN_OK;
    case 2:
        if (launch_compact(w, L, min_pts, labels, is_core, s) != cudaSuccess) return DBSCAN_ERR_CUDA;
        if (L.cull_nbr && (launch_tile_boxes(w, L, 1, s) != cudaSuccess ||
                           launch_tile_boxes(w, L, 2, s) != cudaSuccess))
            return DBSCAN_ERR_CUDA;
        return launch_union(w, L, s) == cudaSuccess ? DBSCAN_OK : DBSCAN_ERR_CUDA;
    case 3:
        if (launch_merge_forests(w, L, gathered, n, L.world, s) != cudaSuccess ||
            launch_flatten(w, L, labels, s) != cudaSuccess ||
            launch_stage_umma(w, L, 2, s) != cudaSuccess || launch_border(w, L, labels, s) != cudaSuccess)
            return DBSCAN_ERR_CUDA;
        return DBSCAN_OK;
    default:
        return launch_finalize(w, L, labels, s) == cudaSuccess ? DBSCAN_OK : DBSCAN_ERR_CUDA;
    }
}

int fit_direct(const void *points, int32_t dtype, int64_t n, int32_t d, float eps, int32_t min_pts,
               int32_t *labels, uint8_t *is_core, void *workspace, size_t workspace_bytes,
               void *stream) {
    return fit_common(points, dtype, n, d, eps, min_pts, labels, is_core, nullptr, workspace,
                      workspace_bytes, stream, 0, false);
}

}  // namespace dbscan

using namespace dbscan;

extern "C" {

size_t dbscan_workspace_size(int64_t n, int32_t d, int32_t dtype) {
    if (check_shape(n, d, dtype) != DBSCAN_OK) return 0;
    if (n == 0) return 256;
    return make_layout(n, d).total;
}

const char *dbscan_strerror(int status) {
    switch (status) {
    case DBSCAN_OK: return "DBSCAN_OK";
    case DBSCAN_ERR_INVALID_ARG: return "DBSCAN_ERR_INVALID_ARG: invalid argument";
    case DBSCAN_ERR_UNSUPPORTED: return "DBSCAN_ERR_UNSUPPORTED: unsupported shape or type";
    case DBSCAN_ERR_ALLOC: return "DBSCAN_ERR_ALLOC: workspace allocation failed";
    case DBSCAN_ERR_CUDA: return "DBSCAN_ERR_CUDA: CUDA runtime error";
    case DBSCAN_ERR_INTERNAL: return "DBSCAN_ERR_INTERNAL: device iteration cap reached";
    default: return "DBSCAN: unknown status";
    }
}

int dbscan_fit_ex(const void *points, int32_t dtype, int64_t n, int32_t d, float eps,
                  int32_t min_pts, int32_t *labels_out, uint8_t *is_core_out, void *workspace,
                  size_t workspace_bytes, void *stream) {
    return fit_common(points, dtype, n, d, eps, min_pts, labels_out, is_core_out, nullptr,
                      workspace, workspace_bytes, stream);
}

int dbscan_fit_culled(const void *points, int32_t dtype, int64_t n, int32_t d, float eps,
                      int32_t min_pts, int32_t *labels_out, uint8_t *is_core_out, void *workspace,
                      size_t workspace_bytes, void *stream) {
    return fit_common(points, dtype, n, d, eps, min_pts, labels_out, is_core_out, nullptr,
                      workspace, workspace_bytes, stream, 1);
}

int dbscan_fit(const float *points, int64_t n, int32_t d, float eps, int32_t min_pts,
               int32_t *labels_out, uint8_t *is_core_out) {
    return fit_common(points, DBSCAN_F32, n, d, eps, min_pts, labels_out, is_core_out, nullptr,
                      nullptr, 0, nullptr);
}

int dbscan_neighbor_counts(const void *points, int32_t dtype, int64_t n, int32_t d, float eps,
                           int32_t *cnt_out, void *workspace, size_t workspace_bytes,
                           void *stream) {
    return fit_common(points, dtype, n, d, eps, 1, nullptr, nullptr, cnt_out, workspace,
                      workspace_bytes, stream);
}

int dbscan_fit_shard(int32_t stage, const void *points, int32_t dtype, int64_t n, int32_t d, float eps,
                     int32_t min_pts, int32_t rank, int32_t world, const int32_t *gathered_parents,
                     int32_t *labels_out, uint8_t *is_core_out, void *workspace,
                     size_t workspace_bytes, void *stream) {
    int st = check_shape(n, d, dtype);
    if (st != DBSCAN_OK) return st;
    if ((st = check_scalars(eps, min_pts)) != DBSCAN_OK) return st;
    if (stage < 0 || stage > 4 || world < 1 || rank < 0 || rank >= world) return DBSCAN_ERR_INVALID_ARG;
    if (n == 0) return DBSCAN_OK;
    if (!workspace) return DBSCAN_ERR_INVALID_ARG;   // the stages share the workspace's state
    Layout L = call_layout(n, d, eps, 0, options_snapshot());
    L.fused = 0;   // the fused pipeline does not split its work
    L.rank = rank;
    L.world = world;
    if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return DBSCAN_ERR_INVALID_ARG;
    if (check_device_ptr(workspace) != DBSCAN_OK) return DBSCAN_ERR_INVALID_ARG;
    if (stage <= 1 && (!points || check_device_ptr(points) != DBSCAN_OK)) return DBSCAN_ERR_INVALID_ARG;
    if (stage == 2 && (!labels_out || !is_core_out || check_device_ptr(labels_out) != DBSCAN_OK ||
                       check_device_ptr(is_core_out) != DBSCAN_OK))
        return DBSCAN_ERR_INVALID_ARG;
    if (stage >= 3 && (!labels_out || check_device_ptr(labels_out) != DBSCAN_OK)) return DBSCAN_ERR_INVALID_ARG;
    if (stage == 3 && (!gathered_parents || check_device_ptr(gathered_parents) != DBSCAN_OK))
        return DBSCAN_ERR_INVALID_ARG;
    return run_shard_stage(stage, points, dtype, n, d, eps, min_pts, gathered_parents, labels_out,
                           is_core_out, workspace, L, static_cast<cudaStream_t>(stream));
}

int dbscan_shard_buffer(void *workspace, int64_t n, int32_t d, int32_t which, void **ptr,
                        int64_t *count) {
    if (!workspace || !ptr || !count || n < 0 || d < 1 || d > DBSCAN_MAX_D) return DBSCAN_ERR_INVALID_ARG;
    if (which != DBSCAN_SHARD_COUNTS && which != DBSCAN_SHARD_PARENTS && which != DBSCAN_SHARD_ORDER)
        return DBSCAN_ERR_INVALID_ARG;
    const Layout L = make_layout(n, d);
    char *b = static_cast<char *>(workspace);
    *ptr = b + (which == DBSCAN_SHARD_COUNTS ? L.off_cnt
                                             : (which == DBSCAN_SHARD_PARENTS ? L.off_parent : L.off_perm));
    *count = n;
    return DBSCAN_OK;
}

int dbscan_set_options(const dbscan_options *opt) {
    dbscan_options o;
    if (opt) {
        const unsigned known = DBSCAN_PATH_TF32 | DBSCAN_PATH_BF16 | DBSCAN_PATH_F16 |
                               DBSCAN_PATH_F16_ACC16;
        if (opt->paths & ~known) return DBSCAN_ERR_INVALID_ARG;
        for (int m = 0; m < 3; ++m)
            if (opt->rows[m] < 0 || opt->rows[m] > 2) return DBSCAN_ERR_INVALID_ARG;
        if (opt->graphs < 0 || opt->graphs > 1) return DBSCAN_ERR_INVALID_ARG;
        if (opt->fused < 0 || opt->fused > 1) return DBSCAN_ERR_INVALID_ARG;
        if (opt->cull < 0 || opt->cull > 1) return DBSCAN_ERR_INVALID_ARG;
        o = *opt;
    } else {
        o = options_from_env();
    }
    std::lock_guard<std::mutex> lock(g_opt_mu);
    g_opt = o;
    g_opt_init = true;
    return DBSCAN_OK;
}

int dbscan_get_options(dbscan_options *opt) {
    if (!opt) return DBSCAN_ERR_INVALID_ARG;
    *opt = options_snapshot();
    return DBSCAN_OK;
}

int dbscan_workspace_info(const void *workspace, void *stream, int64_t *info, int32_t n) {
    if (!workspace || !info || n < 1) return DBSCAN_ERR_INVALID_ARG;
    Ctrl c;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DBSCAN_ERR_CUDA;
    if (cudaMemcpy(&c, workspace, sizeof(Ctrl), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DBSCAN_ERR_CUDA;
    const int64_t v[6] = {c.tc_kind, c.n_core, c.n_cand, c.exact, c.tc_kpad, c.fused};
    for (int i = 0; i < n && i < 6; ++i) info[i] = v[i];
    return DBSCAN_OK;
}

int dbscan_profile_begin(void) {
    for (auto &c : g_prof.calls)
        for (int i = 0; i <= c.stages; ++i) cudaEventDestroy(c.ev[i]);
    g_prof.calls.clear();
    g_prof.failed = false;
    g_prof.on = true;
    return DBSCAN_OK;
}

int dbscan_profile_end(float *stage_ms, int32_t max_stages, int64_t *calls,
                       int64_t *kernel_launches) {
    float acc[DBSCAN_NUM_STAGES] = {0};
    int64_t launches = 0;
    int st = g_prof.failed ? DBSCAN_ERR_CUDA : DBSCAN_OK;
    for (auto &c : g_prof.calls) {
        for (int i = 0; i < c.stages; ++i) {
            float ms = 0.f;
            if (cudaEventSynchronize(c.ev[i + 1]) != cudaSuccess ||
                cudaEventElapsedTime(&ms, c.ev[i], c.ev[i + 1]) != cudaSuccess)
                st = DBSCAN_ERR_CUDA;
            acc[i] += ms;
            // box kernels: all points in prep (culled count), core and
            // candidate arrays after compaction (union and border)
            if (c.fused)
                launches += i == 1 ? 1 : 0;   // the one fused kernel, in the count stage
            else
                launches += stage_launches(c.allow, c.d, c.ntiles, i) + ((c.cull & 1) && i == 0 ? 2 : 0) +
                            ((c.cull & 2) && i == 2 ? 3 : 0);
        }
        for (int i = 0; i <= c.stages; ++i) cudaEventDestroy(c.ev[i]);
    }
    if (calls) *calls = (int64_t)g_prof.calls.size();
    if (kernel_launches) *kernel_launches = launches;
    if (stage_ms)
        for (int i = 0; i < max_stages && i < DBSCAN_NUM_STAGES; ++i) stage_ms[i] = acc[i];
    g_prof.calls.clear();
    g_prof.on = false;
    return st;
}

int dbscan_workspace_status(const void *workspace, void *stream) {
    if (!workspace) return DBSCAN_ERR_INVALID_ARG;
    return read_status(workspace, static_cast<cudaStream_t>(stream));
}

int dbscan_compact_labels(const int32_t *labels, int64_t n, int32_t *labels_out, int32_t *n_clusters,
                          void *stream) {
    if (n < 0 || !n_clusters) return DBSCAN_ERR_INVALID_ARG;
    if (n > (int64_t)INT32_MAX) return DBSCAN_ERR_UNSUPPORTED;
    if (n == 0) {
        *n_clusters = 0;
        return DBSCAN_OK;
    }
    if (!labels || !labels_out) return DBSCAN_ERR_INVALID_ARG;
    if (check_device_ptr(labels) != DBSCAN_OK || check_device_ptr(labels_out) != DBSCAN_OK)
        return DBSCAN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    keep_pool();
    void *scratch = nullptr;
    if (cudaMallocAsync(&scratch, compact_labels_scratch(n), s) != cudaSuccess) {
        cudaGetLastError();
        return DBSCAN_ERR_ALLOC;
    }
    int st = DBSCAN_OK;
    int *k_err = nullptr;
    int host[2] = {0, 0};
    if (launch_compact_labels_rank(labels, n, scratch, &k_err, s) != cudaSuccess ||
        cudaMemcpyAsync(host, k_err, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        st = DBSCAN_ERR_CUDA;
    else if (host[1])
        st = DBSCAN_ERR_INVALID_ARG;   // not labels of dbscan_fit*: nothing is written
    else if (launch_compact_labels_map(labels, n, scratch, labels_out, s) != cudaSuccess)
        st = DBSCAN_ERR_CUDA;
    cudaFreeAsync(scratch, s);
    if (cudaStreamSynchronize(s) != cudaSuccess && st == DBSCAN_OK) st = DBSCAN_ERR_CUDA;
    if (st == DBSCAN_OK) *n_clusters = host[0];
    return st;
}

int dbscan_fit_host(const void *points_host, int32_t dtype, int64_t n, int32_t d, float eps,
                    int32_t min_pts, int32_t *labels_host, uint8_t *is_core_host, void *stream) {
    int st = check_shape(n, d, dtype);
    if (st != DBSCAN_OK) return st;
    if ((st = check_scalars(eps, min_pts)) != DBSCAN_OK) return st;
    if (n == 0) return DBSCAN_OK;
    if (!points_host || !labels_host || !is_core_host) return DBSCAN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Layout L = call_layout(n, d, eps, 0, options_snapshot());
    const size_t esz = dtype == DBSCAN_BF16 ? 2 : 4;
    const size_t pbytes = align256((size_t)n * d * esz);
    const size_t lbytes = align256((size_t)n * sizeof(int32_t));
    const size_t cbytes = align256((size_t)n);
    keep_pool();
    char *buf = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&buf), pbytes + lbytes + cbytes + L.total, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return DBSCAN_ERR_ALLOC;
    }
    void *dp = buf;
    int32_t *dl = reinterpret_cast<int32_t *>(buf + pbytes);
    uint8_t *dc = reinterpret_cast<uint8_t *>(buf + pbytes + lbytes);
    void *ws = buf + pbytes + lbytes + cbytes;
    st = DBSCAN_OK;
    if (cudaMemcpyAsync(dp, points_host, (size_t)n * d * esz, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        st = DBSCAN_ERR_CUDA;
    if (st == DBSCAN_OK)
        st = run(dp, dtype, n, d, eps, min_pts, dl, dc, nullptr, ws, L, s);
    if (st == DBSCAN_OK &&
        (cudaMemcpyAsync(labels_host, dl, (size_t)n * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
             cudaSuccess ||
         cudaMemcpyAsync(is_core_host, dc, (size_t)n, cudaMemcpyDeviceToHost, s) != cudaSuccess))
        st = DBSCAN_ERR_CUDA;
    int dev_st = read_status(ws, s);
    cudaFreeAsync(buf, s);
    if (cudaStreamSynchronize(s) != cudaSuccess && st == DBSCAN_OK) st = DBSCAN_ERR_CUDA;
    return st != DBSCAN_OK ? st : dev_st;
}

}  // extern "C"
