// Tensor-core sweeps (tcgen05): the same three passes as sweep.cu -- count,
// union, border -- with the pair quantity produced by the MMA unit.
//
// The squared distance is a dense contraction once the point-only terms are
// hoisted ("Design and optimization of DBSCAN Algorithm based on CUDA",
// §IV-B2).  prep.cu writes each point as a tf32, bf16 or f16 operand row whose
// dot product with another point's row is exactly w_ij = |c_i - c_j|^2 - thrx,
// so one 128 x 256 x K MMA evaluates two tiles and a pair is a neighbour iff
// w_ij < 0.  The CUDA cores only read the accumulator and test signs.
//
// CTA = 18 warps, one per SM (the CTA owns all 512 TMEM columns):
//   warp 16     producer: pulls work units (a row unit of one or two row
//               blocks and a run of column tiles; for the union, one per band
//               of tile distances) and bulk-copies (cp.async.bulk) the unit's
//               row operand tiles and groups of up to 32 consecutive column
//               tiles (plus their aux ints) into a ring of shared-memory
//               stages, each stage in parts from rotating lanes, since the bulk
//               copies of one thread complete one after another.  With tile
//               culling it streams only the column tiles whose bounding boxes
//               are within eps of the unit's;
//   warp 17     MMA: one thread issues a 128 x 256 x K MMA per pair of column
//               tiles and row block into one of two 256-column TMEM
//               accumulators and commits completion to mbarriers; its loop
//               is the critical path of the sweep and keeps everything it
//               needs in registers;
//   warps 0-15  epilogue: every warp reads every tile pair, 32 rows x 64
//               columns (two reducing tcgen05.ld.red.min, or one packed load
//               of an f16 accumulator), and frees the accumulator before it
//               tests anything -- TMEM read bandwidth grows with the number of
//               warps loading.  The reducing loads return each row's minimum
//               with the values, so the common case (no neighbour among the
//               64 columns) costs one sign test instead of an OR over 64
//               registers on the ALU pipe, which the MMA thread's SMSP shares;
//               only where a 32 x 32 block holds a neighbour does a warp build
//               exact per-row bit masks.  Counting credits the row with a popcount and the
//               columns by atomics (few neighbours) or a warp bit transpose
//               (many); union and border act on each neighbour pair as on CUDA
//               cores.
// The MMA thread polls its barriers without suspending: each MMA issue lies
// on the critical path of the accumulator round trip, and a suspended thread
// resumes hundreds of cycles after the phase completes.  The epilogue warps
// (accumulator and stage waits) and the producer (free stages) wait suspended
// (try_wait): spinning, they took issue slots from the MMA thread (1M x 3
// count 27.8 -> 27.2 ms, 500k x 64 14.9 -> 14.1 ms).
// Every wait on an mbarrier is bounded; on timeout the CTA records
// DBSCAN_ERR_INTERNAL, stops issuing work, waits (bounded) for its own copies
// and MMAs in flight, frees its TMEM and returns.
#include "dbscan_internal.cuh"
#include "tc_schedule.h"

#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>

namespace dbscan {
namespace {

constexpr int EPI_WARPS = 16;                       // two groups of two warpgroups
constexpr int TC_THREADS = (EPI_WARPS + 2) * 32;
constexpr int PRODUCER_WARP = EPI_WARPS, MMA_WARP = EPI_WARPS + 1;
constexpr int NACC = 2;                 // TMEM accumulators of 256 columns
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int TC_MAX_STAGES = 8;
constexpr int TC_MAX_GROUP = 32;        // column tiles per stage (one bulk copy)
// Producer lanes: the bulk copies of one thread complete one after another,
// each taking some 600 cycles up to about 48 KB, so a stage is copied in parts
// of about PART_BYTES issued by different lanes (B_LANES of them, in turn) and
// the row tiles by the other A_LANES.
constexpr int B_LANES = 24, A_LANES = 8;
constexpr int PART_BYTES = 16384;
constexpr long long WAIT_LIMIT = 8000000000LL;   // clock cycles (about 4 s)
constexpr int UF_CAP = 1 << 22;

// Stage flags: the unit's first stage (its row tiles are loaded with it); the
// end of a unit (no tiles: with one row buffer the MMA thread frees it here);
// the end of the sweep.
constexpr int F_FIRST = 1, F_UEND = 2, F_TERM = 8;

struct TcArgs {
    const uint8_t *ua, *ub;   // row / column operand tiles, packed 128 x kbytes each
    const int *n_rows, *n_cols;
    const int *aux;           // per-column int staged with the tiles (parent or label), or null
    int tri;
    int band, blo, bhi;       // band != 0: one unit per row block, tiles rb+blo .. rb+bhi-1
    const float *rbox, *cbox; // per-tile bounding boxes of rows / columns (d x (min, max))
    const float *cgbox;       // boxes of groups of CULL_GROUP column tiles
    const int *troot;         // union: common root of each tile's points, or -1 (else null)
    int cull, d;              // cull != 0: skip column tiles whose box is eps or more away
    unsigned *ctr;
    Ctrl *ctrl;
    int *cnt, *parent;
    const int *candidx;
    int32_t *labels;
    int stages;               // ring depth
    int group;                // column tiles per stage
    int stage_bytes;          // bytes reserved per stage (group tiles + group x BT ints)
    int tile_bytes_max;       // bytes reserved per operand tile
    int nabuf;                // row-tile buffers: 2 (double-buffered units), or 1 for wide rows
    int srank, sworld;        // sharding: this rank takes units k * sworld + srank
};

struct Meta {
    int rb, nrow, t_first, ntiles, flags, abuf;
};

// ---- PTX wrappers ------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// try_wait with a suspend-time hint: a waiting thread sleeps until the phase
// completes (or about 100 us pass) instead of spinning on the issue slots.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(100000u)
        : "memory");
    return ok != 0;
}
// Non-blocking probe of a phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait that polls without suspending; false on timeout or when
// another role aborted.  Out of line: only the slow path of mbar_spin.
__device__ __noinline__ bool mbar_spin_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                            Ctrl *ctrl) {
    long long start = 0;
    for (unsigned it = 0;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 1023) == 1023) {
            if (*abort_flag) return false;
            const long long now = clock64();
            if (start == 0) start = now;
            else if (now - start > WAIT_LIMIT) {
                set_error(ctrl, DBSCAN_ERR_INTERNAL);
                *abort_flag = 1;
                return false;
            }
        }
    }
}
// A phase that has already completed is the common case on the critical
// path; testing it inline avoids a call (which saves and restores the live
// registers of the caller) on every tile pair.
__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          Ctrl *ctrl) {
    return mbar_test(bar, parity) || mbar_spin_slow(bar, parity, abort_flag, ctrl);
}
// Bounded wait that ignores the abort flag (draining copies in flight).
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    const long long start = clock64();
    while (!mbar_try(bar, parity))
        if (clock64() - start > WAIT_LIMIT) return;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)(128u >> 4) << 16;                   // leading (K) core-matrix stride
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;         // 8-row group stride
    d |= (uint64_t)1 << 46;                             // tcgen05 descriptor version
    return d;                                           // no swizzle, base offset 0
}
// D f32 (or f16), A and B of format fmt, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t umma_idesc(int fmt, int n, bool f32acc) {
    return ((f32acc ? 1u : 0u) << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) |
           (((uint32_t)n >> 3) << 17) | ((128u >> 4) << 24);
}
// kind::f16 serves the bf16, f16 and f16-accumulator kinds (the instruction
// descriptor carries the element and accumulator types), kind::tf32 the tf32 one.
template <int KIND>
__device__ __forceinline__ void umma(uint32_t tmem, uint64_t da, uint64_t db, uint32_t idesc,
                                     uint32_t accumulate) {
    if (KIND == TC_TF32)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n"
            ::"r"(tmem), "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
            ::"r"(tmem), "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 lanes x 32 columns of an f32 accumulator (one register per column), and
// per lane the minimum of the 32 values as an f32: the reduction runs in the
// TMEM load path, not on the ALU pipe.
__device__ __forceinline__ void tmem_ld32min(uint32_t taddr, uint32_t (&r)[32], uint32_t &mn) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.min.f32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31]), "=r"(mn)
        : "r"(taddr));
}
// 32 lanes x 64 columns of an f16 accumulator, two columns per register:
// column 2j in bits 0-15 of r[j], column 2j + 1 in bits 16-31.
__device__ __forceinline__ void tmem_ld32p(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.pack::16b.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- union-find (same invariants as the CUDA-core sweep) ---------------------
__device__ __noinline__ int tc_find(int *parent, int x, Ctrl *ctrl) {
    for (int it = 0; it < UF_CAP; ++it) {
        int p = __ldcg(parent + x);
        if (p == x) return x;
        int gp = __ldcg(parent + p);
        if (gp != p) __stcg(parent + x, gp);
        x = gp;
    }
    set_error(ctrl, DBSCAN_ERR_INTERNAL);
    return x;
}
__device__ __noinline__ int tc_unite(int *parent, int a, int b, Ctrl *ctrl) {
    for (int it = 0; it < UF_CAP; ++it) {
        a = tc_find(parent, a, ctrl);
        b = tc_find(parent, b, ctrl);
        if (a == b) return a;
        if (a < b) { int t = a; a = b; b = t; }
        if (atomicCAS(parent + a, a, b) == a) return b;
    }
    set_error(ctrl, DBSCAN_ERR_INTERNAL);
    return min(a, b);
}

// OR of 32 words as a shallow tree of three-input ORs.
__device__ __forceinline__ uint32_t or32(const uint32_t (&a)[32]) {
    uint32_t t[11];
#pragma unroll
    for (int g = 0; g < 10; ++g) t[g] = a[3 * g] | a[3 * g + 1] | a[3 * g + 2];
    t[10] = a[30] | a[31];
    return (t[0] | t[1] | t[2]) | (t[3] | t[4] | t[5]) | (t[6] | t[7] | t[8]) | (t[9] | t[10]);
}

// 32 x 32 bit transpose across a warp: lane i bit j -> lane j bit i.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
    const uint32_t masks[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int st = 0; st < 5; ++st) {
        const int s = 16 >> st;
        const uint32_t m = masks[st];
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, s);
        x = (lane & s) ? ((x & ~m) | ((y >> s) & m)) : ((x & m) | ((y & m) << s));
    }
    return x;
}

// ---- unit schedule: tc_schedule.h ----
static_assert(TC_TILE == BT, "the schedule counts tiles of BT points");

// ---- the kernel --------------------------------------------------------------------
template <int MODE, int KIND, int RT>
__global__ void __launch_bounds__(TC_THREADS, 1) k_sweep_tc(TcArgs a) {
    Ctrl *ctrl = a.ctrl;
    if (ctrl->tc_kind != KIND) return;     // another path was selected for this data
    const int n_rows = *a.n_rows, n_cols = *a.n_cols;
    if (n_rows <= 0 || n_cols <= 0) return;
    constexpr bool AUX = MODE != SWEEP_COUNT;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ __align__(1024) uint8_t smem[];
    const int S = a.stages, G = a.group;
    // layout: [A0 | A1 | stage 0 .. stage S-1 | barriers | meta | misc]; an A
    // buffer holds the RT row tiles of a unit, a stage up to G column tiles back
    // to back, then G x BT ints of aux data
    const size_t abuf_bytes = (size_t)RT * a.tile_bytes_max;
    uint8_t *sA = smem;
    const int NA = a.nabuf;
    uint8_t *sStage = smem + (size_t)NA * abuf_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sStage + (size_t)S * a.stage_bytes);
    uint64_t *b_full = bars, *b_empty = bars + TC_MAX_STAGES;
    uint64_t *a_full = bars + 2 * TC_MAX_STAGES, *a_empty = a_full + 2;
    uint64_t *acc_full = a_empty + 2, *acc_empty = acc_full + NACC;
    uint64_t *drain_bar = acc_empty + NACC;
    Meta *meta = reinterpret_cast<Meta *>(drain_bar + 1);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(meta + TC_MAX_STAGES);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kbytes = ctrl->tc_kbytes;
    const uint32_t tile_bytes = 128u * (uint32_t)kbytes;   // one packed 128-point tile
    const uint32_t sbo = (uint32_t)(kbytes >> 4) * 128u;
    const int ksteps = kbytes / 32;        // 8 tf32 or 16 f16/bf16 elements per MMA
    if (tile_bytes > (uint32_t)a.tile_bytes_max) {   // the host sized the tiles for less
        if (tid == 0) set_error(ctrl, DBSCAN_ERR_INTERNAL);
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_addr(&b_full[i]), 1);
            // every epilogue warp; a warp arrives only after it has seen the
            // accumulator commit of the stage's last tile pair, which implies that
            // every MMA reading the stage has completed
            mbar_init(smem_addr(&b_empty[i]), EPI_WARPS);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&a_full[i]), 1);
            mbar_init(smem_addr(&a_empty[i]), 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(smem_addr(&acc_full[i]), 1);
            mbar_init(smem_addr(&acc_empty[i]), EPI_WARPS);   // every epilogue warp
        }
        mbar_init(smem_addr(drain_bar), 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr(s_tmem)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int lo = a.band ? a.blo : 0, hi = a.band ? a.bhi : -1;
    const TcSched sc = tc_sched(n_rows, n_cols, a.tri, lo, hi, RT, tc_chunk(MODE == SWEEP_UNION && a.band, hi, n_cols));

    if (warp == PRODUCER_WARP) {
        // The whole warp walks the schedule; the copies of consecutive stages
        // are issued by different lanes, since one thread's bulk copies
        // complete one after another.
        int k = 0, ua = 0, a_issued = 0;
        unsigned lane_turn = 0;   // next lane to issue a stage part
        // column tiles per copy: about PART_BYTES, and at most B_LANES copies a
        // stage, the aux ints included
        const int maxp = B_LANES - (AUX ? 1 : 0);
        const int tpp = max(max(1, PART_BYTES / (int)tile_bytes), (G + maxp - 1) / maxp);
        bool ok = true;
        // Culling by tile boxes is exact for integer data within the exactness
        // bound: box gaps are integers, their squared sum is exact, and every
        // pair of a culled tile pair has d^2 >= that sum >= thrx (not a neighbour).
        const bool cull = a.cull && ctrl->exact && a.rbox && a.cbox && a.cgbox;
        const float cthr = ctrl->thrx;
        for (;;) {
            unsigned u = 0;
            if (lane == 0) u = atomicAdd(a.ctr, 1u) * (unsigned)a.sworld + (unsigned)a.srank;
            u = __shfl_sync(FULL, u, 0);
            if (u >= sc.units) break;
            int rb, nrow, t0, t1;
            if (!tc_unit(sc, u, a.tri, lo, hi, rb, nrow, t0, t1)) continue;
            const int ab = NA == 2 ? (ua & 1) : 0;
            const int a_use = NA == 2 ? (ua >> 1) : ua;   // earlier uses of buffer ab
            bool started = false;   // this unit's row tile has been loaded
            // Stages of up to G consecutive tiles over [ts, te); the unit's row
            // tile is loaded before its first stage, so a unit whose column
            // tiles are all culled costs nothing.
            auto emit = [&](int ts, int te) -> bool {
                for (int tf = ts; tf < te; tf += G) {
                    bool first = false;
                    if (!started) {
                        if (!__all_sync(FULL, mbar_spin(smem_addr(&a_empty[ab]), (a_use & 1) ^ 1,
                                                        s_abort, ctrl)))
                            return false;
                        if (lane == B_LANES + (ua % A_LANES)) {
                            // the unit's row tiles are consecutive in the operand array
                            mbar_expect_tx(smem_addr(&a_full[ab]), (uint32_t)nrow * tile_bytes);
                            bulk_g2s(smem_addr(sA + (size_t)ab * abuf_bytes), a.ua + (size_t)rb * tile_bytes,
                                     (uint32_t)nrow * tile_bytes, smem_addr(&a_full[ab]));
                        }
                        a_issued = ua + 1;
                        started = first = true;
                    }
                    const int s = k % S;
                    const int nt = min(G, te - tf);
                    // a stage still in use: wait suspended (the producer runs ahead
                    // of the MMA thread and shares its SMSP with epilogue warps)
                    const uint32_t be = smem_addr(&b_empty[s]), bep = (uint32_t)((k / S) & 1) ^ 1u;
                    if (!__all_sync(FULL, mbar_test(be, bep) || mbar_try(be, bep) ||
                                              mbar_spin_slow(be, bep, s_abort, ctrl)))
                        return false;
                    if (lane == 0) {
                        Meta m;
                        m.rb = rb;
                        m.nrow = nrow;
                        m.t_first = tf;
                        m.ntiles = nt;
                        m.flags = first ? F_FIRST : 0;
                        m.abuf = ab;
                        meta[s] = m;
                    }
                    // one arrival with the stage's bytes, then the parts from
                    // consecutive lanes (the arrival is ordered before them)
                    if (lane == 0)
                        mbar_expect_tx(smem_addr(&b_full[s]),
                                       (uint32_t)nt * tile_bytes + (AUX ? (uint32_t)nt * BT * 4u : 0u));
                    __syncwarp();
                    const int parts = (nt + tpp - 1) / tpp + (AUX ? 1 : 0);
                    const int j = (lane - (int)(lane_turn % B_LANES) + B_LANES) % B_LANES;
                    if (lane < B_LANES && j < parts) {
                        uint8_t *dst = sStage + (size_t)s * a.stage_bytes;
                        const int ntp = (nt + tpp - 1) / tpp;
                        if (j < ntp) {
                            const int t_lo = j * tpp, t_n = min(tpp, nt - t_lo);
                            bulk_g2s(smem_addr(dst + (size_t)t_lo * tile_bytes),
                                     a.ub + (size_t)(tf + t_lo) * tile_bytes, (uint32_t)t_n * tile_bytes,
                                     smem_addr(&b_full[s]));
                        } else {
                            bulk_g2s(smem_addr(dst + (size_t)G * a.tile_bytes_max), a.aux + (size_t)tf * BT,
                                     (uint32_t)nt * BT * 4u, smem_addr(&b_full[s]));
                        }
                    }
                    lane_turn += (unsigned)parts;
                    ++k;
                }
                return true;
            };
            if (!cull) {
                ok = emit(t0, t1);
            } else {
                // Column tiles go by groups of CULL_GROUP (8) tiles: the boxes of
                // 32 groups are tested at once, and only the tiles of the kept
                // groups are tested, 32 at a time (four groups); runs of kept
                // tiles become stages.  Gaps are integers, so every sum below
                // is exact in any order.
                static_assert(CULL_GROUP == 8, "32 tile slots hold four groups");
                // The unit's box is the union of its row tiles' boxes.
                const float *rbx0 = a.rbox + (size_t)rb * 2 * a.d;
                const float *rbx1 = a.rbox + (size_t)(rb + nrow - 1) * 2 * a.d;
                auto rlo = [&](int kk) { return fminf(rbx0[2 * kk], rbx1[2 * kk]); };
                auto rhi = [&](int kk) { return fmaxf(rbx0[2 * kk + 1], rbx1[2 * kk + 1]); };
                // d > 4: the lanes split the dimensions (lane and lane + 32), each
                // keeping its share of the unit's box in registers; d <= 4: every
                // lane keeps the whole box and tests a box of its own
                const bool split = a.d > 4;
                float rl0 = 0.f, rh0 = 0.f, rl1 = 0.f, rh1 = 0.f;
                float rl[4] = {0.f, 0.f, 0.f, 0.f}, rh[4] = {0.f, 0.f, 0.f, 0.f};
                if (split) {
                    if (lane < a.d) { rl0 = rlo(lane); rh0 = rhi(lane); }
                    if (lane + 32 < a.d) { rl1 = rlo(lane + 32); rh1 = rhi(lane + 32); }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        if (kk < a.d) { rl[kk] = rlo(kk); rh[kk] = rhi(kk); }
                }
                // this lane's part of the squared gap between the unit's box and box bx
                auto part = [&](const float *bx) -> float {
                    float g2 = 0.f;
                    if (lane < a.d) {
                        const float2 v = *reinterpret_cast<const float2 *>(bx + 2 * lane);
                        const float gp = fmaxf(0.f, fmaxf(v.x - rh0, rl0 - v.y));
                        g2 = gp * gp;
                    }
                    if (lane + 32 < a.d) {
                        const float2 v = *reinterpret_cast<const float2 *>(bx + 2 * (lane + 32));
                        const float gp = fmaxf(0.f, fmaxf(v.x - rh1, rl1 - v.y));
                        g2 = fmaf(gp, gp, g2);
                    }
                    return g2;
                };
                // Bit j: the box at bx0 + ix(j) (every ix(j) in range) is closer
                // than eps to the unit's box.  Split: every lane's parts for all
                // 32 boxes, then a butterfly reduce-scatter -- after the round of
                // offset o a lane keeps the half of the boxes whose index bit o
                // matches its own, so lane j ends with box j's sum.
                auto test32 = [&](const float *bx0, auto ix) -> unsigned {
                    float g2 = 0.f;
                    if (split) {
                        float pv[32];
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) pv[jj] = part(bx0 + (size_t)ix(jj) * 2 * a.d);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const bool up = (lane & o) != 0;
#pragma unroll
                            for (int jj = 0; jj < o; ++jj) {
                                const float send = up ? pv[jj] : pv[jj + o];
                                const float mine = up ? pv[jj + o] : pv[jj];
                                pv[jj] = mine + __shfl_xor_sync(FULL, send, o);
                            }
                        }
                        g2 = pv[0];
                    } else {
                        const float *bx = bx0 + (size_t)ix(lane) * 2 * a.d;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            if (kk < a.d) {
                                const float gp = fmaxf(0.f, fmaxf(bx[2 * kk] - rh[kk], rl[kk] - bx[2 * kk + 1]));
                                g2 = fmaf(gp, gp, g2);
                            }
                    }
                    return __ballot_sync(FULL, g2 < cthr);
                };
                // union: the common root of the unit's row tiles, or -1; a column
                // tile with the same common root holds no pair left to join
                int uroot = -1;
                if (MODE == SWEEP_UNION && a.troot) {
                    uroot = a.troot[rb];
                    if (nrow > 1 && a.troot[rb + 1] != uroot) uroot = -1;
                }
                const int gend = (t1 + CULL_GROUP - 1) / CULL_GROUP;
                for (int gb = t0 / CULL_GROUP; gb < gend && ok; gb += 32) {
                    unsigned gk = test32(a.cgbox, [&](int jj) { return min(gb + jj, gend - 1); });
                    if (gend - gb < 32) gk &= (1u << (gend - gb)) - 1u;
                    while (gk && ok) {
                        // up to four kept groups (5-bit offsets from gb in sel); slot
                        // s holds tile s & 7 of the (s >> 3)-th of them
                        uint32_t sel = 0;
                        int ns = 0;
                        while (gk && ns < 4) {
                            sel |= (uint32_t)(__ffs(gk) - 1) << (5 * ns);
                            gk &= gk - 1;
                            ++ns;
                        }
                        auto slot_tile = [&](int sl) {
                            return (gb + (int)((sel >> (5 * (sl >> 3))) & 31u)) * CULL_GROUP + (sl & 7);
                        };
                        const int my = slot_tile(lane);
                        const bool inr = (lane >> 3) < ns && my >= t0 && my < t1;
                        const bool joined = inr && uroot >= 0 && a.troot[my] == uroot;
                        const unsigned valid = __ballot_sync(FULL, inr && !joined);
                        unsigned km = valid & test32(a.cbox, [&](int sl) {
                                          return min(max(slot_tile(sl), t0), t1 - 1);
                                      });
                        // a run breaks where the next group does not follow on
                        unsigned brk = 0;
                        for (int q = 1; q < ns; ++q)
                            if (((sel >> (5 * q)) & 31u) != ((sel >> (5 * (q - 1))) & 31u) + 1u) brk |= 1u << (8 * q);
                        while (km && ok) {
                            const int s0 = __ffs(km) - 1;
                            int e = s0 + 1;
                            while (e < 32 && ((km >> e) & 1u) && !((brk >> e) & 1u)) ++e;
                            km = e >= 32 ? 0u : (km & (0xffffffffu << e));
                            const int ts = slot_tile(s0);
                            ok = emit(ts, ts + (e - s0));
                        }
                    }
                }
            }
            if (started && ok && NA == 1) {
                // end of the unit: the MMA thread frees the one row buffer here
                const int s = k % S;
                ok = __all_sync(FULL, mbar_spin(smem_addr(&b_empty[s]), ((k / S) & 1) ^ 1, s_abort, ctrl));
                if (ok && lane == 0) {
                    Meta m;
                    m.rb = rb;
                    m.nrow = nrow;
                    m.t_first = t0;
                    m.ntiles = 0;
                    m.flags = F_UEND;
                    m.abuf = 0;
                    meta[s] = m;
                    mbar_arrive(smem_addr(&b_full[s]));
                }
                ++k;
            }
            if (started) ++ua;
            if (!ok) break;
        }
        if (ok) {   // terminate marker (every consumer reads every stage)
            const int s = k % S;
            ok = __all_sync(FULL, mbar_spin(smem_addr(&b_empty[s]), ((k / S) & 1) ^ 1, s_abort, ctrl));
            if (ok && lane == 0) {
                meta[s].flags = F_TERM;
                mbar_arrive(smem_addr(&b_full[s]));
            }
        }
        if (!ok && lane == 0) {   // let the copies already issued land before the CTA exits
            for (int j = max(0, k - S); j < k; ++j) mbar_drain(smem_addr(&b_full[j % S]), (j / S) & 1);
            for (int j = max(0, a_issued - NA); j < a_issued; ++j)
                mbar_drain(smem_addr(&a_full[j % NA]), (j / NA) & 1);
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            // One thread issues every MMA, and its loop is a dependent chain
            // on the critical path of the accumulator round trip: everything
            // it needs is kept in registers -- barrier addresses, descriptors
            // (a descriptor is a constant plus address >> 4 in bits 0-13, and
            // every shared-memory address is below 2^18), stage index and
            // phase -- and nothing is divided.
            const int fmt = KIND == TC_TF32 ? 2 : (KIND == TC_BF16 ? 1 : 0);
            const bool f32acc = KIND != TC_F16H;
            const uint32_t idesc256 = umma_idesc(fmt, 256, f32acc), idesc128 = umma_idesc(fmt, 128, f32acc);
            const uint64_t dbase = umma_desc(0, sbo);
            const uint32_t bar_bf = smem_addr(b_full), bar_af = smem_addr(a_full), bar_ae = smem_addr(a_empty);
            const uint32_t bar_accf = smem_addr(acc_full), bar_acce = smem_addr(acc_empty);
            const uint64_t dA0 = dbase + (smem_addr(sA) >> 4), dA1 = dbase + (smem_addr(sA + abuf_bytes) >> 4);
            const uint64_t dS0 = dbase + (smem_addr(sStage) >> 4);
            const uint32_t dstage = (uint32_t)a.stage_bytes >> 4, dpair = (2u * tile_bytes) >> 4,
                           drow = tile_bytes >> 4;
            int s = 0, ua = 0;
            uint32_t sph = 0;           // phase of the current use of stage s
            uint32_t b = 0, eph = 1;    // accumulator of the next item, and the phase of its release
            bool issued = false, ok = true;
            for (;;) {
                if (!mbar_spin(bar_bf + 8u * s, sph, s_abort, ctrl)) break;
                const Meta m = meta[s];
                if (m.flags & F_TERM) break;
                if (m.flags & F_FIRST) {
                    // the previous unit's row tiles have been read by every MMA
                    // issued so far (one buffer: freed at the unit's end marker)
                    if (ua > 0 && NA == 2) umma_commit(bar_ae + 8u * ((ua - 1) & 1));
                    if (!mbar_spin(bar_af + 8u * m.abuf, (NA == 2 ? (ua >> 1) : ua) & 1, s_abort, ctrl)) break;
                    ++ua;
                }
                if (m.flags & F_UEND) umma_commit(bar_ae);   // one buffer: free it (no tiles follow)
                const uint64_t da0 = m.abuf ? dA1 : dA0;
                // item (i, r): row tile r of the unit against column tiles 2i, 2i + 1;
                // a pair of consecutive column tiles is one 256-row B operand, and
                // a K step is 256 bytes further (16 in the address field)
                uint64_t db = dS0 + (uint64_t)((uint32_t)s * dstage);
                if (RT == 1 && ksteps == 1) {
                    // one row block and one K step (d <= 10 on f16): a slimmer
                    // loop -- no K loop, accumulate flag or row index, and the
                    // two accumulators' addresses selected, not computed (this
                    // loop bounds the sweep: 29.2 -> 27.9 ms at 1M x 3)
                    const int npair = m.ntiles >> 1;
                    const uint32_t td0 = tmem, td1 = tmem + (uint32_t)ACC_COLS;
                    const uint32_t ae0 = bar_acce, ae1 = bar_acce + 8u, af0 = bar_accf, af1 = bar_accf + 8u;
                    for (int i = 0; i < npair; ++i, db += dpair) {
                        if (!(ok = mbar_spin(b ? ae1 : ae0, eph, s_abort, ctrl))) break;
                        tc_fence_after();
                        umma<KIND>(b ? td1 : td0, da0, db, idesc256, 0u);
                        umma_commit(b ? af1 : af0);
                        eph ^= b;
                        b ^= 1u;
                    }
                    if (ok && (m.ntiles & 1)) {   // an odd last column tile: N = 128
                        if ((ok = mbar_spin(b ? ae1 : ae0, eph, s_abort, ctrl))) {
                            tc_fence_after();
                            umma<KIND>(b ? td1 : td0, da0, db, idesc128, 0u);
                            umma_commit(b ? af1 : af0);
                            eph ^= b;
                            b ^= 1u;
                        }
                    }
                    issued = issued || m.ntiles > 0;
                } else if (RT == 1) {
                    // one row block, K steps in a loop: the same slimming (the
                    // first MMA overwrites, the rest accumulate; 200k x 16 count
                    // 1.75 -> 1.44 ms, 500k x 64 15.5 -> 14.9 ms)
                    const uint32_t td0 = tmem, td1 = tmem + (uint32_t)ACC_COLS;
                    const uint32_t ae0 = bar_acce, ae1 = bar_acce + 8u, af0 = bar_accf, af1 = bar_accf + 8u;
                    for (int i = 0; 2 * i < m.ntiles; ++i, db += dpair) {
                        const uint32_t idesc = 2 * i + 1 < m.ntiles ? idesc256 : idesc128;
                        if (!(ok = mbar_spin(b ? ae1 : ae0, eph, s_abort, ctrl))) break;
                        tc_fence_after();
                        const uint32_t td = b ? td1 : td0;
                        umma<KIND>(td, da0, db, idesc, 0u);
                        for (int ks = 1; ks < ksteps; ++ks)
                            umma<KIND>(td, da0 + (uint64_t)(16 * ks), db + (uint64_t)(16 * ks), idesc, 1u);
                        umma_commit(b ? af1 : af0);
                        eph ^= b;
                        b ^= 1u;
                    }
                    issued = issued || m.ntiles > 0;
                } else {
                    // two row blocks: row tile 0, then row tile 1 (when the unit
                    // has one), against each pair of column tiles
                    const uint32_t td0 = tmem, td1 = tmem + (uint32_t)ACC_COLS;
                    const uint32_t ae0 = bar_acce, ae1 = bar_acce + 8u, af0 = bar_accf, af1 = bar_accf + 8u;
                    const uint64_t da1 = da0 + (uint64_t)drow;
                    for (int i = 0; 2 * i < m.ntiles; ++i, db += dpair) {
                        const uint32_t idesc = 2 * i + 1 < m.ntiles ? idesc256 : idesc128;
                        if (!(ok = mbar_spin(b ? ae1 : ae0, eph, s_abort, ctrl))) break;
                        tc_fence_after();
                        uint32_t td = b ? td1 : td0;
                        umma<KIND>(td, da0, db, idesc, 0u);
                        for (int ks = 1; ks < ksteps; ++ks)
                            umma<KIND>(td, da0 + (uint64_t)(16 * ks), db + (uint64_t)(16 * ks), idesc, 1u);
                        umma_commit(b ? af1 : af0);
                        eph ^= b;
                        b ^= 1u;
                        if (m.nrow > 1) {
                            if (!(ok = mbar_spin(b ? ae1 : ae0, eph, s_abort, ctrl))) break;
                            tc_fence_after();
                            td = b ? td1 : td0;
                            umma<KIND>(td, da1, db, idesc, 0u);
                            for (int ks = 1; ks < ksteps; ++ks)
                                umma<KIND>(td, da1 + (uint64_t)(16 * ks), db + (uint64_t)(16 * ks), idesc, 1u);
                            umma_commit(b ? af1 : af0);
                            eph ^= b;
                            b ^= 1u;
                        }
                    }
                    issued = issued || m.ntiles > 0;
                }
                if (!ok) break;
                if (++s == S) {
                    s = 0;
                    sph ^= 1u;
                }
            }
            if (issued) {   // no MMA may be in flight when TMEM is freed
                umma_commit(smem_addr(drain_bar));
                mbar_drain(smem_addr(drain_bar), 0);
            }
        }
    } else {
        // ---------------- epilogue: all 16 warps read every item ----------------
        // Warp w reads TMEM lanes 32*(w % 4).. (the lanes its position in a
        // warpgroup may access) and the 64 columns 64*(w / 4).. of the
        // 256-column item, releases the accumulator as soon as its two loads
        // have landed, and only then tests the values: the accumulator round
        // trip is bounded by how fast TMEM is drained, which takes every warp.
        const int wq = warp & 3, cq = warp >> 2;
        const int row = wq * 32 + lane;
        // per row tile r of the unit (at most two): UNION keeps a known ancestor
        // of this row's point and the last staged parent joined to it
        int last_rb = -1, acc0 = -1, acc1 = -1, lastq0 = -1, lastq1 = -1;
        int s = 0, it = 0;
        uint32_t sph = 0;   // phase of the current use of stage s
        for (;;) {
            // every lane waits (suspended, like the accumulator waits); the warp
            // goes on only if all lanes saw the phase
            const uint32_t bf = smem_addr(&b_full[s]);
            if (!__all_sync(FULL, mbar_test(bf, sph) || mbar_try(bf, sph) || mbar_spin_slow(bf, sph, s_abort, ctrl)))
                break;
            const Meta m = meta[s];
            if (m.flags & F_TERM) break;
            const int p0 = m.rb * BT + row, p1 = p0 + BT;
            const bool valid0 = p0 < n_rows, valid1 = RT > 1 && m.nrow > 1 && p1 < n_rows;
            if (MODE == SWEEP_UNION && m.rb != last_rb) {
                acc0 = valid0 ? tc_find(a.parent, p0, ctrl) : -1;
                if (RT > 1) acc1 = valid1 ? tc_find(a.parent, p1, ctrl) : -1;
                last_rb = m.rb;
                lastq0 = lastq1 = -1;
            }
            const int *saux = reinterpret_cast<const int *>(sStage + (size_t)s * a.stage_bytes +
                                                            (size_t)G * a.tile_bytes_max);
            int rowadd0 = 0, rowadd1 = 0, rowmin0 = 0x7fffffff, rowmin1 = 0x7fffffff;
            bool ok = true;
            for (int i = 0; 2 * i < m.ntiles && ok; ++i) {
                for (int r = 0; r < (RT == 1 ? 1 : m.nrow); ++r, ++it) {
                    const int b = it % NACC;
                    // a phase not yet complete: wait suspended (mbarrier.try_wait), so
                    // that the 16 waiting warps leave their SMSPs' issue slots to the
                    // MMA thread and the producer (count 1M x 3 27.8 -> 27.4 ms,
                    // 500k x 64 14.9 -> 14.2 ms); bounded by the spin behind it
                    const uint32_t af = smem_addr(&acc_full[b]), afp = (uint32_t)(it / NACC) & 1u;
                    const bool got = mbar_test(af, afp) || mbar_try(af, afp) || mbar_spin_slow(af, afp, s_abort, ctrl);
                    if (!(ok = __all_sync(FULL, got))) break;
                    tc_fence_after();
                    const int ti = 2 * i + (cq >> 1);     // tile within the stage
                    const int tile = m.t_first + ti;
                    const int rt = m.rb + r;              // row tile of this item
                    // warp-uniform: the tile exists and, in the triangle, is not
                    // below this row tile (that pair belongs to the other order);
                    // the union also skips the diagonal tile, whose pairs the
                    // tile-local union has already joined
                    const bool have = ti < m.ntiles &&
                                      !(a.tri && (MODE == SWEEP_UNION ? tile <= rt : (RT > 1 && tile < rt)));
                    const bool diag = a.tri && tile == rt;
                    // f32 accumulator: v0, v1 = columns 0-31, 32-63 of the warp's 64,
                    // and mn0, mn1 the minimum of each half (from the loads);
                    // f16 accumulator (F16H): v0 = all 64 columns, two per register
                    uint32_t v0[32], v1[32], mn0 = 0, mn1 = 0;
                    if (have) {
                        const uint32_t taddr = tmem + ((uint32_t)(wq * 32) << 16) +
                                               (uint32_t)(b * ACC_COLS + cq * 64);
                        if (KIND == TC_F16H) {
                            tmem_ld32p(taddr, v0);
                        } else {
                            tmem_ld32min(taddr, v0, mn0);
                            tmem_ld32min(taddr + 32, v1, mn1);
                        }
                        tmem_ld_wait();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&acc_empty[b]));
                    if (!have) continue;
                    const int p = r ? p1 : p0;
                    const bool rowvalid = r ? valid1 : valid0;
                    // a negative minimum has its sign bit set (an exact zero is +0)
                    const uint32_t neg = KIND == TC_F16H ? (or32(v0) & 0x80008000u) : ((mn0 | mn1) >> 31);
                    if (!__any_sync(FULL, rowvalid && neg)) continue;
                    int rowadd = 0, rowmin = 0x7fffffff;
                    int acc = r ? acc1 : acc0, lastq = r ? lastq1 : lastq0;
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        const int cb = (cq & 1) * 64 + blk * 32;   // column offset in the tile
                        const int qbase = tile * BT + cb;
                        // bit c of mask = (w_c < 0) for the block's 32 columns
                        uint32_t mask;
                        if (KIND == TC_F16H) {
                            uint32_t o = 0;
#pragma unroll
                            for (int c = 0; c < 16; c += 2) o |= v0[16 * blk + c] | v0[16 * blk + c + 1];
                            if (!__any_sync(FULL, rowvalid && (o & 0x80008000u))) continue;
                            // two 16-column chains; register j holds columns 2j (bit 15)
                            // and 2j + 1 (bit 31)
                            uint32_t m16[2] = {0u, 0u};
#pragma unroll
                            for (int j = 7; j >= 0; --j)
#pragma unroll
                                for (int g = 0; g < 2; ++g) {
                                    const uint32_t rr = v0[16 * blk + 8 * g + j];
                                    m16[g] = __funnelshift_l(rr, m16[g], 1);
                                    m16[g] = __funnelshift_l(rr << 16, m16[g], 1);
                                }
                            mask = m16[0] | (m16[1] << 16);
                        } else {
                            uint32_t (&v)[32] = blk ? v1 : v0;
                            uint32_t o = 0;
#pragma unroll
                            for (int c = 0; c < 32; c += 2) o |= v[c] | v[c + 1];
                            if (!__any_sync(FULL, rowvalid && (o >> 31))) continue;
                            // four independent 8-column chains
                            uint32_t m8[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                            for (int c = 7; c >= 0; --c)
#pragma unroll
                                for (int g = 0; g < 4; ++g) m8[g] = __funnelshift_l(v[8 * g + c], m8[g], 1);
                            mask = m8[0] | (m8[1] << 8) | (m8[2] << 16) | (m8[3] << 24);
                        }
                        const int nv = n_cols - qbase;
                        mask &= nv >= 32 ? 0xffffffffu : (nv <= 0 ? 0u : ((1u << nv) - 1u));
                        if (!rowvalid) mask = 0;
                        if (MODE == SWEEP_COUNT) {
                            const int nh = __popc(mask);
                            rowadd += nh;
                            if (!diag) {   // the diagonal tile is counted from both sides already
                                if (__any_sync(FULL, nh > 2)) {
                                    // many neighbours: per-column sums through a bit transpose
                                    const int cc = __popc(warp_transpose32(mask, lane));
                                    if (cc) atomicAdd(a.cnt + qbase + lane, cc);
                                } else {
                                    // few: credit each neighbour's column directly
                                    while (mask) {
                                        const int cq2 = __ffs(mask) - 1;
                                        mask &= mask - 1;
                                        atomicAdd(a.cnt + qbase + cq2, 1);
                                    }
                                }
                            }
                        } else {
                            while (mask) {
                                const int cq2 = __ffs(mask) - 1;
                                mask &= mask - 1;
                                const int q = qbase + cq2;
                                const int aq = saux[ti * BT + cb + cq2];
                                if (MODE == SWEEP_UNION) {
                                    if (diag && q <= p) continue;
                                    if (aq == acc || aq == lastq) continue;
                                    lastq = aq;   // aq joins this row's set for good
                                    acc = tc_unite(a.parent, acc, aq, ctrl);
                                } else {
                                    rowmin = min(rowmin, aq);
                                }
                            }
                        }
                    }
                    if (r) {
                        rowadd1 += rowadd;
                        rowmin1 = min(rowmin1, rowmin);
                        acc1 = acc;
                        lastq1 = lastq;
                    } else {
                        rowadd0 += rowadd;
                        rowmin0 = min(rowmin0, rowmin);
                        acc0 = acc;
                        lastq0 = lastq;
                    }
                }
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&b_empty[s]));
            if (MODE == SWEEP_COUNT) {
                if (rowadd0) atomicAdd(a.cnt + p0, rowadd0);
                if (RT > 1 && rowadd1) atomicAdd(a.cnt + p1, rowadd1);
            }
            if (MODE == SWEEP_BORDER) {
                if (rowmin0 != 0x7fffffff) atomicMin(a.labels + a.candidx[p0], rowmin0);
                if (RT > 1 && rowmin1 != 0x7fffffff) atomicMin(a.labels + a.candidx[p1], rowmin1);
            }
            if (++s == S) {
                s = 0;
                sph ^= 1u;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                     : "memory");
}

// Bytes of shared memory the kernel needs.
size_t tc_smem_bytes(int tile_bytes, int rows, int nabuf, int stage_bytes, int stages) {
    return (size_t)nabuf * rows * tile_bytes + (size_t)stages * stage_bytes +
           (2 * TC_MAX_STAGES + 4 + 2 * NACC + 1) * sizeof(uint64_t) + TC_MAX_STAGES * sizeof(Meta) +
           16;
}

// Row blocks per unit.  A unit costs a row-tile load and the fill of its first
// stage before its first MMA; when tile culling leaves a unit a few short runs
// of column tiles, that cost dominates, and two row blocks per unit halve the
// number of units and copy every kept column tile once for both (the culling
// box is then the union of the two row tiles' boxes).  A full-length unit gains
// nothing from it and pays for the second row's bookkeeping in the epilogue.
// The border sweep keeps one row block: its candidate tiles are sparse.
// The rows tuning switch (dbscan_set_options) overrides per sweep.
int tc_rows(const Layout &L, int mode, int cull) {
    const int r = L.rows[mode];
    if (r == 1 || r == 2) return r;
    return cull && mode != SWEEP_BORDER ? 2 : 1;
}

template <int MODE, int KIND>
cudaError_t run_tc(TcArgs a, const Layout &L, cudaStream_t s) {
    // largest operand row this path can need for this eps (the device's choice
    // of threshold digits never exceeds the host's bound)
    const int ntb = tc_nt_bound(KIND, L.eps2);
    const int kb = tc_kbytes(KIND, L.d, ntb);
    // never selected: not allowed for this call, or the operand rows do not fit
    if (L.umma_tile_bytes == 0 || !(L.allow & tc_allow_bit(KIND)) || !tc_fits(KIND, L.d, ntb))
        return cudaSuccess;
    const int tile = 128 * kb;
    const int aux = MODE != SWEEP_COUNT ? BT * 4 : 0;
    const size_t budget = 224 * 1024;
    int rows = tc_rows(L, MODE, a.cull);
    // two row blocks need room for four row tiles next to two stages of two
    // column tiles; wide operand rows keep one
    if (rows == 2 && 4 * (size_t)tile + 4 * (size_t)(tile + aux) > budget) rows = 1;
    // Few, large stages: every stage costs a round of barrier handshakes
    // between the producer, the MMA thread and all epilogue warps, so the
    // group is the largest even number of tiles (<= 32) for which two stages
    // and the row buffers fit; what is left takes further stages.  Rows too
    // wide for two row buffers next to two stages of two tiles (d = 256 on
    // bf16 or f16: 544-byte rows, 68 KB tiles) take one row buffer, freed at
    // the end of each unit, and stages of one tile.
    int nabuf = 2;
    if (2 * (size_t)rows * tile + 2 * 2 * (size_t)(tile + aux) > budget) {
        nabuf = 1;
        rows = 1;
    }
    auto kernel = rows == 2 ? k_sweep_tc<MODE, KIND, 2> : k_sweep_tc<MODE, KIND, 1>;
    const size_t abufs = (size_t)nabuf * rows * tile;   // buffers of a unit's row tiles
    int group = TC_MAX_GROUP;
    while (group > 2 && abufs + 2 * (size_t)group * (tile + aux) > budget) group -= 2;
    if (nabuf == 1 && abufs + 2 * (size_t)group * (tile + aux) > budget) group = 1;
    if (abufs + 2 * (size_t)group * (tile + aux) > budget) return cudaErrorInvalidValue;
    const int stage_bytes = group * (tile + aux);
    int stages = (int)((budget - abufs) / stage_bytes);
    if (stages > TC_MAX_STAGES) stages = TC_MAX_STAGES;
    if (stages < 2) stages = 2;
    size_t smem = tc_smem_bytes(tile, rows, nabuf, stage_bytes, stages);
    if (smem < 120 * 1024) smem = 120 * 1024;   // one CTA per SM: it owns all of TMEM
    cudaError_t e = cudaFuncSetAttribute((const void *)kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    a.stages = stages;
    a.nabuf = nabuf;
    a.group = group;
    a.stage_bytes = stage_bytes;
    a.tile_bytes_max = tile;
    kernel<<<sms, TC_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t run_tc_both(const TcArgs &a, const Layout &L, cudaStream_t s) {
    cudaError_t e = run_tc<MODE, TC_TF32>(a, L, s);
    if (e != cudaSuccess) return e;
    if ((e = run_tc<MODE, TC_BF16>(a, L, s)) != cudaSuccess) return e;
    if ((e = run_tc<MODE, TC_F16>(a, L, s)) != cudaSuccess) return e;
    return run_tc<MODE, TC_F16H>(a, L, s);
}

}  // namespace

cudaError_t launch_count_tc(const Work &w, const Layout &L, cudaStream_t s) {
    TcArgs a{};
    a.srank = L.rank; a.sworld = L.world;
    a.ua = w.ua_all; a.ub = w.ub_all;
    a.n_rows = &w.ctrl->n_all; a.n_cols = &w.ctrl->n_all;
    a.tri = 1;
    a.ctr = &w.ctrl->unit_ctr[0]; a.ctrl = w.ctrl; a.cnt = w.cnt;
    a.rbox = w.box_all; a.cbox = w.box_all; a.cgbox = w.gbox_all; a.cull = L.cull; a.d = L.d;
    return run_tc_both<SWEEP_COUNT>(a, L, s);
}

cudaError_t launch_union_tc_band(const Work &w, const Layout &L, int band, int blo, int bhi,
                                 cudaStream_t s) {
    TcArgs a{};
    a.srank = L.rank; a.sworld = L.world;
    a.ua = w.ua_core; a.ub = w.ub_core;
    a.n_rows = &w.ctrl->n_core; a.n_cols = &w.ctrl->n_core; a.aux = w.parent;
    a.tri = 1;
    a.band = 1; a.blo = blo; a.bhi = bhi;
    a.ctr = &w.ctrl->band_ctr[band]; a.ctrl = w.ctrl; a.parent = w.parent;
    a.rbox = w.box_core; a.cbox = w.box_core; a.cgbox = w.gbox_core; a.cull = L.cull_nbr; a.d = L.d;
    a.troot = w.troot;
    return run_tc_both<SWEEP_UNION>(a, L, s);
}

cudaError_t launch_border_tc(const Work &w, const Layout &L, int32_t *labels, cudaStream_t s) {
    TcArgs a{};
    a.srank = L.rank; a.sworld = L.world;
    a.ua = w.ua_cand; a.ub = w.ub_core;
    a.n_rows = &w.ctrl->n_cand; a.n_cols = &w.ctrl->n_core; a.aux = w.clabel;
    a.tri = 0;
    a.ctr = &w.ctrl->unit_ctr[5]; a.ctrl = w.ctrl;
    a.candidx = w.candidx; a.labels = labels;
    a.rbox = w.box_cand; a.cbox = w.box_core; a.cgbox = w.gbox_core; a.cull = L.cull_nbr; a.d = L.d;
    return run_tc_both<SWEEP_BORDER>(a, L, s);
}

}  // namespace dbscan
