// Block-scaled grouped GEMM for routed MoE experts on sm_103a tensor cores (tcgen05).
//
// Definition [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本":
// section "方案 1：端到端 MXFP8 强化学习" (forward, weight-gradient and data-gradient GEMMs run in
// MXFP8, microscaling blocks along the reduction dimension); section "结果：在 8x B200 上对
// Qwen3-30B-A3B 配方进行消融实验" (the per-token NVFP4 GEMM applies the FP32 per-token scaling in the
// kernel epilogue instead of a separate op); NVFP4-ru = page "NVIDIA верифицировала 4-битный формат
// NVFP4 ..." (FP4 GEMMs run natively on Blackwell tensor cores)]:
//   GROUP_M: D[i, j] = s_a[i] s_b[e] sum_k deq(A)[i, k] deq(B[e])[j, k]   (rows i of group e)
//   GROUP_K: D[e][i, j] = sum_{k in group e} deq(A)[i, k] deq(B)[j, k]
//
// Design (one CTA per SM, persistent, warp-specialised; 256 threads for MXFP8, 384 for NVFP4 and
// BF16 operands). A CTA computes 128 x 256
// output tiles (tcgen05 M = 128, N = 256) from a ring of stages (MXFP8: 4 x 50 KB, NVFP4: 3 x 58 KB),
// each holding a 128x128-byte A tile, a 256x128-byte B tile (128B swizzle) and their 512-byte
// scale tiles. Roles:
//   warp 0 lane 0  TMA producer: A and B tiles (tensor copies) and the scale tiles (bulk copies).
//   warp 6         A-scale transposer: a GROUP_M tile starts at its group's row offset (any row),
//                  so its 128 rows of A scales straddle two 128-row scale tiles; the producer loads
//                  both into the stage and the warp rebuilds the tile's own 512-byte scale tile (each
//                  16-byte line a 4-word window of one line of the two loaded tiles).
//   warp 7 lane 0  scale warp: copies each stage's scale tiles smem -> TMEM (tcgen05.cp
//                  32x128b.warpx4) into one of two TMEM scale sets, so that the copies of the next
//                  stage are queued while the MMAs of this one run.
//   warp 1 lane 0  MMA issuer: four tcgen05.mma block_scale instructions per stage (K = 32 for
//                  MXFP8 E4M3 x UE8M0/32, K = 64 for NVFP4 E2M1 x UE4M3/16) into a 256-column fp32
//                  TMEM accumulator; commits free stages and scale sets and signal the epilogue.
//                  Warp 1 also allocates and frees TMEM.
//   warps 2-5      epilogue (and warps 8-11 for NVFP4 and BF16 operands, so that two warps share
//   (8-11)         each TMEM lane quarter, one per 128-column half, and the accumulator goes back
//                  to the MMA warp in about half the time; MXFP8's four stages leave no shared
//                  memory for their staging buffers): tcgen05.ld 32 columns at a time (the next load
//                  in flight while the current chunk converts), multiply by s_a[row] s_b[e], round to
//                  bf16 into registers (the thread's row within the warp's columns), hand TMEM back
//                  to the MMA warp, then store while the next tile's MMAs run: for grouped row-offset GEMMs
//                  each warp whose 32 rows all belong to the tile's group stages 32 x 32 chunks in
//                  shared memory (64-byte swizzle) and sends them with TMA box stores; otherwise each
//                  thread stores its own row with 256-bit stores (fp32 output: chunk by chunk).
// GROUP_K tiles iterate the group's reduction range in 32-element MMA steps (k-steps outside the
// group inside a 128-element stage are skipped).
//
// Every wait on an mbarrier is bounded; a wait that runs out sets the caller's status word to
// NVQ_DEV_TIMEOUT and a CTA-wide abort flag, and every role then leaves its loop, waits (bounded)
// for the asynchronous work it issued, and the CTA frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/nvq.h"
#include "nvq_device.cuh"
#include "nvq_internal.h"

namespace nvq {

// Warps 0-7 have fixed roles; warps 8-11 (when a format has 8 epilogue warps) are the second
// epilogue warp of each TMEM lane quarter.
constexpr int W_PRODUCER = 0, W_MMA = 1, W_EPI0 = 2, W_TRANSPOSER = 6, W_SCALE = 7, W_EPI1 = 8;
constexpr int BM = 128, BN = 256, BKB = 128;       // tile rows, tile columns, K bytes per stage
constexpr int MAX_GROUPS = 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;    // 2 s: far beyond any legitimate wait (default)

enum { F_MXFP8 = 0, F_NVFP4 = 1, F_BF16 = 2 };       // operand formats (the kernel's template argument)

template <int FMT>
struct GemmCfg {
    static constexpr bool FP4 = FMT == F_NVFP4;
    static constexpr bool SCALED = FMT != F_BF16;      // block-scaled MMA (scale tiles staged to TMEM)
    static constexpr int STAGES = FP4 ? 3 : 4;
    static constexpr int KGS = FP4 ? 4 : 1;            // 4-scale-column groups per stage
    static constexpr int EPS = FP4 ? 256 : (SCALED ? 128 : 64);   // reduction elements per stage (128 B)
    static constexpr int MMA_K = FP4 ? 64 : (SCALED ? 32 : 16);   // reduction elements per MMA (32 B)
    static constexpr int A_BYTES = BM * BKB;
    static constexpr int B_BYTES = BN * BKB;
    static constexpr int SFA_BYTES = SCALED ? KGS * 512 : 0;        // the tile's own 128 row scales
    static constexpr int SFB_BYTES = SCALED ? 2 * KGS * 512 : 0;    // two 128-row scale tiles (N = 256)
    static constexpr int SFA_RAW_BYTES = SCALED ? 2 * KGS * 512 : 0;  // the two row tiles a 32-aligned tile spans
    static constexpr int STAGE_BYTES =
        (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES + SFA_RAW_BYTES + 1023) / 1024 * 1024;
    static constexpr uint32_t SF_SETS = SCALED ? 2 : 0;             // TMEM scale sets
    static constexpr uint32_t SF_SETS_NZ = SCALED ? SF_SETS : 1;    // divisor for set arithmetic
    static constexpr uint32_t SFA_COLS = KGS * 4;      // TMEM columns of A's scales
    static constexpr uint32_t SFB_COLS = KGS * 8;      // TMEM columns of B's scales
    static constexpr uint32_t SF_SET_COLS = SFA_COLS + SFB_COLS;
    static constexpr uint32_t IDESC =
        (SCALED ? ((FP4 ? ((1u << 7) | (1u << 10)) : 0u)   // A, B format: E2M1 (mxf4nvf4) or E4M3
                   | (FP4 ? 0u : (1u << 23)))               // scale type: UE4M3 (0) / UE8M0 (1)
                : ((1u << 4) | (1u << 7) | (1u << 10)))     // kind::f16: D F32, A and B BF16
        | ((uint32_t)(BN >> 3) << 17)                  // N >> 3
        | ((uint32_t)(BM >> 4) << 24);                 // M >> 4
    static constexpr int BAR_BYTES = 256;
    // Epilogue warps: one per TMEM lane quarter draining all BN columns of its 32 rows, or two per
    // quarter draining BN / 2 columns each (the accumulator goes back to the MMA warp in about half
    // the time). MXFP8's four stages leave no shared memory for the second set's staging buffers.
    static constexpr int EPI_WARPS = (FMT == F_MXFP8) ? 4 : 8;
    static constexpr int EPI_COLS = BN * 4 / EPI_WARPS;         // accumulator columns per epilogue warp
    static constexpr int THREADS = 32 * (4 + EPI_WARPS);
    // bf16 output staging for the TMA stores: per epilogue warp, STG_BUFS buffers of 32 rows x 32
    // columns (2 KB, 64-byte swizzle), 1024-aligned after the stages, barriers and group tables
    static constexpr size_t STG_OFFSET =
        ((size_t)STAGES * STAGE_BYTES + BAR_BYTES + 8 * (MAX_GROUPS + 1) + 1023) / 1024 * 1024;
    static constexpr int STG_BUFS = (1024 + STG_OFFSET + (size_t)EPI_WARPS * 2 * 2048 <= 232448) ? 2 : 1;
    static constexpr size_t STG_BYTES = (size_t)EPI_WARPS * STG_BUFS * 2048;
    static constexpr size_t SMEM_BYTES = 1024 + STG_OFFSET + STG_BYTES;
    static_assert(BN + SF_SETS * SF_SET_COLS <= TMEM_COLS, "TMEM columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

struct GemmParams {
    int mode;
    int out_f32;
    int groups;
    int64_t m, n, k;
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* s_a;
    const float* s_b;
    const int64_t* offsets;
    void* d;
    int64_t ldd;
    int d_aligned32;        // d and every row of it start on 32 bytes: 256-bit stores
    int tma_store;          // bf16 output leaves through staged TMA box stores (else per-thread rows)
    int32_t* status;
    uint64_t wait_limit_ns; // bound of every pipeline wait (teardown drains keep WAIT_LIMIT_NS)
    int inject_stage;       // > 0: CTA 0's producer stops before its inject_stage-th stage (watchdog test)
    int64_t a_rowtiles;     // 128-row scale tiles of A
    int64_t b_rowtiles;     // 128-row scale tiles of B (stacked rows)
    int64_t sf_tiles_per_row;   // 4-column scale tiles per row (same for A and B)
};

// ------------------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait; returns false (and raises the abort flag / status) when `limit_ns` of wall-clock
// time pass without the phase completing, or when another role has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* status,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) break;
        }
    }
    *abort_flag = 1;
    if (status) atomicExch(status, NVQ_DEV_TIMEOUT);
    return false;
}

// Bounded drain used at teardown: wait for a phase without raising anything.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Shared -> global tensor copy of one box (bulk-group completion); x, y: element coordinates
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N bulk groups of this thread still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrives on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start >> 4, LBO >> 4, SBO >> 4, version 1, swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46) | ((uint64_t)swizzle << 61);
}

template <int FMT>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    if constexpr (FMT == F_NVFP4) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
    } else if constexpr (FMT == F_MXFP8) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Start a 32-lane x 32-column TMEM load into r; the registers are valid after tmem_wait_ld(r).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Wait for every outstanding TMEM load of this thread; r is threaded through so that no use of the
// loaded registers can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// 32 bytes to a 32-byte aligned global address in one 256-bit store.
__device__ __forceinline__ void st_v8(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t e,
                                      uint32_t f, uint32_t g, uint32_t h) {
    asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
                 : "memory");
}

__device__ __forceinline__ void pack_scaled(const uint32_t (&r)[32], float scale, uint32_t (&pk)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
        pk[j] = cvt_bf16x2(__uint_as_float(r[2 * j]) * scale, __uint_as_float(r[2 * j + 1]) * scale);
}

// ------------------------------------------------------------------------------------------------
// Tile schedule (identical in every role)
// ------------------------------------------------------------------------------------------------
struct Tile {
    int e;
    int64_t a_row0;     // first A row of the tile (GROUP_M: inside group e; GROUP_K: output row)
    int64_t b_row0;     // first B row of the tile (stacked rows)
    int64_t row_end;    // GROUP_M: end of group e's rows (exclusive); GROUP_K: m
    int64_t n0;         // first output column
    int64_t k_begin, k_end;   // reduction range (elements)
    int64_t d_row0;     // first output row in D's row space
};

struct Schedule {
    const int32_t* off;        // group offsets (smem, int32)
    const int32_t* tile_start; // GROUP_M: prefix of tiles per group (smem)
    int mode, groups;
    int64_t m, n, k;
    int n_tiles, m_tiles;      // GROUP_K: per-group tile grid
    int64_t total;

    __device__ Tile get(int64_t t) const {
        Tile tl;
        if (mode == NVQ_GEMM_GROUP_M) {
            int lo = 0, hi = groups - 1;           // largest e with tile_start[e] <= t
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
            }
            const int e = lo;
            const int64_t local = t - tile_start[e];
            const int64_t mt = local / n_tiles, nt = local - mt * n_tiles;
            tl.e = e;
            tl.a_row0 = off[e] + mt * BM;
            tl.row_end = min((int64_t)off[e + 1], m);
            tl.n0 = nt * BN;
            tl.b_row0 = (int64_t)e * n + tl.n0;
            tl.k_begin = 0;
            tl.k_end = k;
            tl.d_row0 = tl.a_row0;
        } else {
            const int64_t per = (int64_t)m_tiles * n_tiles;
            const int e = (int)(t / per);
            const int64_t local = t - (int64_t)e * per;
            const int64_t mt = local / n_tiles, nt = local - mt * n_tiles;
            tl.e = e;
            tl.a_row0 = mt * BM;
            tl.row_end = m;
            tl.n0 = nt * BN;
            tl.b_row0 = tl.n0;
            tl.k_begin = off[e];
            tl.k_end = off[e + 1];
            tl.d_row0 = (int64_t)e * m + tl.a_row0;
        }
        return tl;
    }
};

// Walks the stages (k-steps of non-empty tiles) of one CTA in schedule order, for roles that run
// ahead of the stage they are working on.
template <int EPS>
struct StageCursor {
    const Schedule* sched;
    int64_t t, step, ks, ks1;
    Tile tl;
    bool valid;

    __device__ void seek(int64_t from) {
        for (t = from; t < sched->total; t += step) {
            tl = sched->get(t);
            if (tl.k_end > tl.k_begin) {
                ks = tl.k_begin / EPS;
                ks1 = (tl.k_end + EPS - 1) / EPS;
                valid = true;
                return;
            }
        }
        valid = false;
    }
    __device__ void begin(const Schedule* s, int64_t first, int64_t stride) {
        sched = s;
        step = stride;
        seek(first);
    }
    __device__ void next() {
        if (++ks < ks1) return;
        seek(t + step);
    }
};

// ------------------------------------------------------------------------------------------------
// Kernel
// ------------------------------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(GemmCfg<FMT>::THREADS, 1)
block_scaled_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_d, const GemmParams p) {
    griddep_begin();
    using C = GemmCfg<FMT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_base = smem;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty_bar = full_bar + C::STAGES;
    uint64_t* sfa_bar = empty_bar + C::STAGES;         // [STAGES] raw A scales of a shifted tile landed
    uint64_t* sf_ready = sfa_bar + C::STAGES;          // [SF_SETS] scale set copied into TMEM
    uint64_t* sf_free = sf_ready + C::SF_SETS;         // [SF_SETS] MMAs reading the set are done
    uint64_t* tmem_full = sf_free + C::SF_SETS;
    uint64_t* tmem_empty = tmem_full + 1;
    uint64_t* mma_done = tmem_empty + 1;
    uint64_t* cp_done = mma_done + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(cp_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* bad_flag = reinterpret_cast<int*>(tmem_holder + 2);
    int32_t* off32 = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(full_bar) + C::BAR_BYTES);
    int32_t* tile_start = off32 + (MAX_GROUPS + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.groups;
    const int n_tiles = (int)((p.n + BN - 1) / BN);

    // ---- validate offsets and build the schedule (all threads see the same smem) ----
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        *bad_flag = 0;
    }
    __syncthreads();
    const int64_t limit = (p.mode == NVQ_GEMM_GROUP_M) ? p.m : p.k;
    for (int e = threadIdx.x; e <= G; e += blockDim.x) {
        const int64_t o = p.offsets[e];
        // weight gradients: a 32-element reduction block never straddles two groups
        const bool ok = (o >= 0) && (o <= limit) && (p.mode == NVQ_GEMM_GROUP_M || (o & 31) == 0) &&
                        (e > 0 || o == 0) && (e == 0 || p.offsets[e - 1] <= o);
        if (!ok) *bad_flag = 1;
        off32[e] = (int32_t)o;
    }
    __syncthreads();
    if (*bad_flag) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && p.status) atomicExch(p.status, NVQ_DEV_BAD_OFFSETS);
        return;
    }
    Schedule sched;
    sched.off = off32;
    sched.tile_start = tile_start;
    sched.mode = p.mode;
    sched.groups = G;
    sched.m = p.m;
    sched.n = p.n;
    sched.k = p.k;
    sched.n_tiles = n_tiles;
    sched.m_tiles = (int)((p.m + BM - 1) / BM);
    if (p.mode == NVQ_GEMM_GROUP_M) {
        if (threadIdx.x == 0) {
            int32_t acc = 0;
            for (int e = 0; e < G; ++e) {
                tile_start[e] = acc;
                acc += (int32_t)(((off32[e + 1] - off32[e]) + BM - 1) / BM) * n_tiles;
            }
            tile_start[G] = acc;
        }
        __syncthreads();
        sched.total = tile_start[G];
    } else {
        sched.total = (int64_t)G * sched.m_tiles * n_tiles;
    }
    const int64_t total = sched.total;

    // ---- barriers and TMEM ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            // the producer's expect_tx arrival + its second arrival or the scale transposer's
            mbar_init(&full_bar[s], 2);
            mbar_init(&empty_bar[s], 1);
            mbar_init(&sfa_bar[s], 1);
        }
        if constexpr (C::SCALED) {
            for (uint32_t k = 0; k < C::SF_SETS; ++k) {
                mbar_init(&sf_ready[k], 1);
                mbar_init(&sf_free[k], 1);
            }
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, C::EPI_WARPS);   // one arrival per epilogue warp
        mbar_init(mma_done, 1);
        mbar_init(cp_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_holder)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint32_t tmem_acc = tmem_base;
    // scale set k: A's scales at tmem_sfa(k) (k-group j at +4j), B's at tmem_sfb(k) (+8j)
    auto tmem_sfa = [&](uint32_t k) { return tmem_base + BN + k * C::SF_SET_COLS; };
    auto tmem_sfb = [&](uint32_t k) { return tmem_base + BN + k * C::SF_SET_COLS + C::SFA_COLS; };
    const int64_t first = blockIdx.x, stride = gridDim.x;

    if (warp == W_PRODUCER && lane == 0) {
        // =========================== TMA producer ===========================
        int slot = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        uint32_t sfa_fills[C::STAGES];          // shifted-tile fills of each slot's sfa_bar
        for (int i = 0; i < C::STAGES; ++i) sfa_fills[i] = 0;
        StageCursor<C::EPS> cur;
        for (cur.begin(&sched, first, stride); cur.valid; cur.next()) {
            // watchdog test: stop before this stage, arming nothing, so its consumers' waits run out
            if (p.inject_stage > 0 && blockIdx.x == 0 && issued + 1 == p.inject_stage) break;
            if (!mbar_wait(&empty_bar[slot], phase ^ 1u, abort_flag, p.status, p.wait_limit_ns)) break;
            const Tile& tl = cur.tl;
            const int64_t rb_a = tl.a_row0 / BM;
            const bool shifted = C::SCALED && (tl.a_row0 % BM) != 0;
            const bool need_a2 = shifted && rb_a + 1 < p.a_rowtiles;
            const int64_t rb_b = tl.b_row0 / BM;
            const bool need_b2 = rb_b + 1 < p.b_rowtiles;
            uint8_t* st = stage_base + (size_t)slot * C::STAGE_BYTES;
            uint8_t* ssfa = st + C::A_BYTES + C::B_BYTES;
            uint8_t* ssfb = ssfa + C::SFA_BYTES;
            uint8_t* ssfa_raw = ssfb + C::SFB_BYTES;
            const int64_t kg0 = cur.ks * C::KGS;
            const int64_t kgn = min((int64_t)C::KGS, p.sf_tiles_per_row - kg0);
            const uint32_t sf_bytes = (uint32_t)kgn * 512u;
            // full_bar completes after two arrivals and all bytes: the producer's expect_tx arrival
            // (A, B, B scales, and the A scales of an aligned tile) plus either the producer's second
            // arrival (aligned tile) or the transposer's (tile starting inside a scale tile)
            const uint32_t tx = C::A_BYTES + C::B_BYTES +
                                (C::SCALED ? sf_bytes * (1u + (need_b2 ? 1u : 0u)) + (shifted ? 0u : sf_bytes) : 0u);
            mbar_arrive_expect_tx(&full_bar[slot], tx);
            if (!C::SCALED) {
                // no scales to stage
            } else if (shifted) {
                mbar_arrive_expect_tx(&sfa_bar[slot], sf_bytes * (1u + (need_a2 ? 1u : 0u)));
                ++sfa_fills[slot];
                bulk_load(ssfa_raw, p.sfa + ((rb_a * p.sf_tiles_per_row + kg0) << 9), sf_bytes, &sfa_bar[slot]);
                if (need_a2)
                    bulk_load(ssfa_raw + C::KGS * 512, p.sfa + (((rb_a + 1) * p.sf_tiles_per_row + kg0) << 9),
                              sf_bytes, &sfa_bar[slot]);
            } else {
                bulk_load(ssfa, p.sfa + ((rb_a * p.sf_tiles_per_row + kg0) << 9), sf_bytes, &full_bar[slot]);
            }
            tma_load_2d(st, &tmap_a, (int32_t)(cur.ks * BKB), (int32_t)tl.a_row0, &full_bar[slot]);
            tma_load_2d(st + C::A_BYTES, &tmap_b, (int32_t)(cur.ks * BKB), (int32_t)tl.b_row0, &full_bar[slot]);
            if (C::SCALED) {
                bulk_load(ssfb, p.sfb + ((rb_b * p.sf_tiles_per_row + kg0) << 9), sf_bytes, &full_bar[slot]);
                if (need_b2)
                    bulk_load(ssfb + C::KGS * 512, p.sfb + (((rb_b + 1) * p.sf_tiles_per_row + kg0) << 9), sf_bytes,
                              &full_bar[slot]);
            }
            if (!shifted) mbar_arrive(&full_bar[slot]);
            ++issued;
            if (++slot == C::STAGES) { slot = 0; phase ^= 1u; }
        }
        // wait (bounded) until the copies of the last fill of every slot have landed
        const int64_t n_last = issued < C::STAGES ? issued : C::STAGES;
        for (int64_t i = 0; i < n_last; ++i) {
            int s2 = slot - 1 - (int)i;
            uint32_t ph = phase;
            if (s2 < 0) { s2 += C::STAGES; ph ^= 1u; }
            mbar_drain(&full_bar[s2], ph);
        }
        for (int s2 = 0; s2 < C::STAGES; ++s2)
            if (sfa_fills[s2]) mbar_drain(&sfa_bar[s2], (sfa_fills[s2] - 1u) & 1u);
    } else if (C::SCALED && warp == W_SCALE && lane == 0) {
        // =========================== scale warp ===========================
        // Copies stage `fill`'s scale tiles into scale set fill % SF_SETS (A's k-group j at columns
        // [4j, 4j+4) of the set, B's at [8j, 8j+8): two 128-row tiles) once the stage has landed and
        // the MMAs of the set's previous use are done.
        int slot = 0;
        uint32_t phase = 0;
        uint32_t fill = 0;
        const uint32_t stage0 = smem_u32(stage_base);
        StageCursor<C::EPS> cur;
        for (cur.begin(&sched, first, stride); cur.valid; cur.next()) {
            const uint32_t set = fill % C::SF_SETS_NZ;
            if (!mbar_wait(&full_bar[slot], phase, abort_flag, p.status, p.wait_limit_ns) ||
                !mbar_wait(&sf_free[set], ((fill / C::SF_SETS_NZ) & 1u) ^ 1u, abort_flag, p.status, p.wait_limit_ns))
                break;
            tc_fence_after();
            const uint32_t ssfa = stage0 + (uint32_t)slot * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
            const uint32_t ssfb = ssfa + C::SFA_BYTES;
#pragma unroll
            for (int j = 0; j < C::KGS; ++j) {
                tc_cp_sf(tmem_sfa(set) + 4 * j, smem_desc(ssfa + j * 512, 0, 128, 0));
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tc_cp_sf(tmem_sfb(set) + 8 * j + 4 * h, smem_desc(ssfb + (h * C::KGS + j) * 512, 0, 128, 0));
            }
            tc_commit(&sf_ready[set]);
            ++fill;
            if (++slot == C::STAGES) { slot = 0; phase ^= 1u; }
        }
        // wait (bounded) for the copies issued above before TMEM is released
        tc_commit(cp_done);
        mbar_drain(cp_done, 0);
    } else if (warp == W_MMA && lane == 0) {
        // =========================== MMA issuer ===========================
        int slot = 0;
        uint32_t phase = 0;
        uint32_t acc_phase = 0;
        uint32_t fill = 0;                       // stages consumed (selects the scale set)
        bool ok = true;
        const uint32_t stage0 = smem_u32(stage_base);
        for (int64_t t = first; t < total && ok; t += stride) {
            const Tile tl = sched.get(t);
            if (tl.k_end <= tl.k_begin) continue;
            if (!mbar_wait(tmem_empty, acc_phase ^ 1u, abort_flag, p.status, p.wait_limit_ns)) break;
            tc_fence_after();
            const int64_t ks0 = tl.k_begin / C::EPS, ks1 = (tl.k_end + C::EPS - 1) / C::EPS;
            uint32_t accumulate = 0;
            for (int64_t ks = ks0; ks < ks1; ++ks) {
                const uint32_t set = fill % C::SF_SETS_NZ;
                if (!mbar_wait(&full_bar[slot], phase, abort_flag, p.status, p.wait_limit_ns) ||
                    (C::SCALED && !mbar_wait(&sf_ready[set], (fill / C::SF_SETS_NZ) & 1u, abort_flag, p.status, p.wait_limit_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = stage0 + (uint32_t)slot * C::STAGE_BYTES;
                const uint64_t adesc0 = smem_desc(sa, 16, 1024, 2);
                const uint64_t bdesc0 = smem_desc(sa + C::A_BYTES, 16, 1024, 2);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t kel = ks * C::EPS + (int64_t)j * C::MMA_K;
                    if (kel < tl.k_begin || kel >= tl.k_end) continue;
                    const uint32_t kg = C::FP4 ? (uint32_t)j : 0u;
                    const uint32_t sf_id = (C::SCALED && !C::FP4) ? (uint32_t)j : 0u;
                    const uint32_t idesc = C::IDESC | (sf_id << 4) | (sf_id << 29);
                    // K advance inside the 128-byte swizzled row: 32 bytes per MMA (encoded >> 4)
                    tc_mma<FMT>(tmem_acc, adesc0 + (uint64_t)(2 * j), bdesc0 + (uint64_t)(2 * j), idesc,
                                tmem_sfa(set) + 4 * kg, tmem_sfb(set) + 8 * kg, accumulate);
                    accumulate = 1;
                }
                tc_commit(&empty_bar[slot]);
                if (C::SCALED) tc_commit(&sf_free[set]);
                ++fill;
                if (++slot == C::STAGES) { slot = 0; phase ^= 1u; }
            }
            if (!ok) break;
            tc_commit(tmem_full);
            acc_phase ^= 1u;
        }
        // wait (bounded) for every tcgen05 operation issued above before TMEM is released
        tc_commit(mma_done);
        mbar_drain(mma_done, 0);
    } else if (C::SCALED && warp == W_TRANSPOSER) {
        // ======================= A-scale transposer =======================
        // A tile starting g rows into a 128-row scale tile needs rows [g, 128) of that tile followed
        // by rows [0, g) of the next. In the 512-byte tile layout line l holds the scales of rows l,
        // l+32, l+64, l+96 as four 4-byte words (one word = a row's four scale columns). The tile's
        // own line l holds its rows l + 32w, i.e. rows g + l + 32w of the two loaded tiles, which
        // all sit on line L = (g + l) % 32 at words (g + l) / 32 + w of (line L of tile 0 ++ line L
        // of tile 1): lane l copies that 4-word window.
        int slot = 0;
        uint32_t sfa_phase = 0;                 // bit s: parity of the next sfa_bar[s] phase
        bool ok = true;
        const uint32_t stage0 = smem_u32(stage_base);
        for (int64_t t = first; t < total && ok; t += stride) {
            const Tile tl = sched.get(t);
            if (tl.k_end <= tl.k_begin) continue;
            const int64_t ks0 = tl.k_begin / C::EPS, ks1 = (tl.k_end + C::EPS - 1) / C::EPS;
            const int g = (int)(tl.a_row0 % BM);
            const uint32_t src_line = (uint32_t)((g + lane) & 31), shift = (uint32_t)((g + lane) >> 5);   // 0..4
            if (g == 0) {
                // aligned tile: the producer loaded the scales in place; only keep the ring position
                slot = (int)((slot + (ks1 - ks0)) % C::STAGES);
                continue;
            }
            for (int64_t ks = ks0; ks < ks1; ++ks) {
                int good = 1;
                if (lane == 0) good = mbar_wait(&sfa_bar[slot], (sfa_phase >> slot) & 1u, abort_flag, p.status, p.wait_limit_ns) ? 1 : 0;
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) { ok = false; break; }
                const uint32_t dst = stage0 + (uint32_t)slot * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
                const uint32_t raw = dst + C::SFA_BYTES + C::SFB_BYTES;
#pragma unroll
                for (int j = 0; j < C::KGS; ++j) {
                    uint32_t w[8];
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                 : "r"(raw + j * 512 + src_line * 16));
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                                 : "r"(raw + (C::KGS + j) * 512 + src_line * 16));
                    // window of 4 words starting at word `shift` (0..4): barrel shift by 4, 2, 1
                    if (shift & 4u) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) w[i] = w[i + 4];
                    }
                    if (shift & 2u) {
#pragma unroll
                        for (int i = 0; i < 5; ++i) w[i] = w[i + 2];
                    }
                    if (shift & 1u) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) w[i] = w[i + 1];
                    }
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                                 ::"r"(dst + j * 512 + lane * 16), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
                // make the generic-proxy writes visible to tcgen05.cp (async proxy), then hand over
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_bar[slot]);
                sfa_phase ^= 1u << slot;
                if (++slot == C::STAGES) slot = 0;
            }
        }
    } else if ((warp >= W_EPI0 && warp < W_EPI0 + 4) || (warp >= W_EPI1 && warp < 4 + C::EPI_WARPS)) {
        // =========================== epilogue ===========================
        constexpr int NCH = C::EPI_COLS / 32;         // 32-column chunks this warp drains per tile
        const int q = warp & 3;                       // TMEM lane quarter this warp may access
        const int ei = warp < W_EPI1 ? warp - W_EPI0 : warp - 4;   // epilogue warp index 0..EPI_WARPS-1
        const int cbase = warp < W_EPI1 ? 0 : C::EPI_COLS;         // first accumulator column it drains
        const int row_in_tile = q * 32 + lane;
        const uint32_t stg_warp = smem_u32(smem + C::STG_OFFSET) + (uint32_t)(ei * C::STG_BUFS * 2048);
        uint32_t stg_count = 0;                       // chunks this warp has staged
        const uint32_t tbase = tmem_acc + ((uint32_t)(q * 32) << 16) + (uint32_t)cbase;
        uint32_t acc_phase = 0;
        for (int64_t t = first; t < total; t += stride) {
            const Tile tl = sched.get(t);
            const int64_t row = tl.a_row0 + row_in_tile;
            const bool row_ok = row < tl.row_end;
            const int64_t drow = tl.d_row0 + row_in_tile;
            float scale = 1.0f;
            if (row_ok && p.s_a) scale = p.s_a[row];
            if (p.s_b) scale *= p.s_b[tl.e];
            const bool empty = tl.k_end <= tl.k_begin;
            if (!empty) {
                // every lane waits; the warp leaves together if any lane gave up (the TMEM loads
                // below are warp-wide instructions)
                const bool good = mbar_wait(tmem_full, acc_phase, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, good)) break;
                tc_fence_after();
            }
            if (p.out_f32) {
                // fp32 output: store each 32-column chunk as it leaves TMEM
                for (int c = 0; c < NCH; ++c) {
                    const int64_t col = tl.n0 + cbase + c * 32;
                    uint32_t r[32];
                    if (!empty) {
                        tmem_ld32_async(tbase + (uint32_t)(c * 32), r);
                        tmem_wait_ld(r);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;
                    }
                    if (!row_ok || col >= p.n) continue;
                    float* dst = reinterpret_cast<float*>(p.d) + drow * p.ldd + col;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float4 v = make_float4(__uint_as_float(r[4 * j]) * scale, __uint_as_float(r[4 * j + 1]) * scale,
                                               __uint_as_float(r[4 * j + 2]) * scale, __uint_as_float(r[4 * j + 3]) * scale);
                        reinterpret_cast<float4*>(dst)[j] = v;
                    }
                }
                if (!empty) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tmem_empty);
                    acc_phase ^= 1u;
                }
                continue;
            }
            // bf16 output: drain the whole accumulator row into registers as packed bf16 (the next
            // 32-column load in flight while the current one converts) and hand TMEM back to the
            // MMA warp before storing, so the stores overlap the next tile's MMAs
            uint32_t pk[NCH][16];
            if (!empty) {
                uint32_t ra[32], rb[32];
                tmem_ld32_async(tbase, ra);
                tmem_wait_ld(ra);
#pragma unroll
                for (int c = 0; c < NCH; c += 2) {
                    tmem_ld32_async(tbase + (uint32_t)((c + 1) * 32), rb);
                    pack_scaled(ra, scale, pk[c]);
                    tmem_wait_ld(rb);
                    if (c + 2 < NCH) tmem_ld32_async(tbase + (uint32_t)((c + 2) * 32), ra);
                    pack_scaled(rb, scale, pk[c + 1]);
                    if (c + 2 < NCH) tmem_wait_ld(ra);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tmem_empty);
                acc_phase ^= 1u;
            } else {
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int j = 0; j < 16; ++j) pk[c][j] = 0u;
            }
            // box stores need the warp's 32 rows inside the tile's group (a group may end at any row)
            const bool box = p.tma_store && tl.a_row0 + q * 32 + 32 <= tl.row_end;
            if (!box) {
                if (row_ok) {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.d) + drow * p.ldd + tl.n0 + cbase;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        if (tl.n0 + cbase + c * 32 >= p.n) break;
                        if (p.d_aligned32) {
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                st_v8(dst + c * 32 + h * 16, pk[c][8 * h], pk[c][8 * h + 1], pk[c][8 * h + 2],
                                      pk[c][8 * h + 3], pk[c][8 * h + 4], pk[c][8 * h + 5], pk[c][8 * h + 6],
                                      pk[c][8 * h + 7]);
                        } else {
#pragma unroll
                            for (int h = 0; h < 4; ++h)
                                reinterpret_cast<uint4*>(dst + c * 32)[h] =
                                    make_uint4(pk[c][4 * h], pk[c][4 * h + 1], pk[c][4 * h + 2], pk[c][4 * h + 3]);
                        }
                    }
                }
                continue;
            }
            // Stores: each 32-column chunk of the warp's 32 rows goes through a 2 KB staging buffer
            // (row `lane` = 64 bytes, 16-byte pieces placed by the 64-byte swizzle: piece j of row r
            // at j ^ ((r >> 1) & 3)) and leaves as one TMA box store.
            {
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    if (tl.n0 + cbase + c * 32 >= p.n) break;
                    const uint32_t buf = stg_warp + (uint32_t)((stg_count % C::STG_BUFS) * 2048);
                    // the buffer's previous store has finished reading it (groups complete in order)
                    if (lane == 0) bulk_wait_read<C::STG_BUFS - 1>();
                    __syncwarp();
                    const uint32_t rowp = buf + (uint32_t)lane * 64;
                    const uint32_t swz = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                                     ::"r"(rowp + ((j ^ swz) << 4)), "r"(pk[c][4 * j]), "r"(pk[c][4 * j + 1]),
                                       "r"(pk[c][4 * j + 2]), "r"(pk[c][4 * j + 3])
                                     : "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmap_d, buf, (int32_t)(tl.n0 + cbase + c * 32), (int32_t)(tl.d_row0 + q * 32));
                        bulk_commit();
                    }
                    ++stg_count;
                }
            }
        }
        // the staged chunks must be read out before the CTA exits
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }

    // teardown: every role is done (and has drained the asynchronous work it issued)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_MMA) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// ------------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D uint8 tensor map over [rows, row_bytes] with a (box_rows x 128-byte) box, 128B swizzle,
// zero fill out of bounds.
static bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)BKB, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor map over D [rows, n] (row pitch ldd elements) with a 32 x 32 box and 64-byte
// swizzle, for the epilogue's box stores; columns past n are not written.
static bool make_tmap_d(CUtensorMap* map, void* base, int64_t rows, int64_t n, int64_t ldd) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ldd * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <int FMT>
static nvq_status launch_gemm(const nvq_gemm_args* a, cudaStream_t stream) {
    using C = GemmCfg<FMT>;
    const int64_t row_bytes = C::FP4 ? a->k / 2 : (C::SCALED ? a->k : 2 * a->k);
    const int64_t rows_a = a->m;
    const int64_t rows_b = (a->mode == NVQ_GEMM_GROUP_M) ? a->groups * a->n : a->n;
    CUtensorMap ta, tb, td;
    if (!make_tmap(&ta, a->a, rows_a, row_bytes, BM) || !make_tmap(&tb, a->b, rows_b, row_bytes, BN))
        return NVQ_ERR_CUDA;
    if (a->out_type == NVQ_OUT_F32) {
        td = ta;                                   // unused: fp32 rows are stored by the threads
    } else {
        const int64_t rows_d = (a->mode == NVQ_GEMM_GROUP_M) ? a->m : a->groups * a->m;
        if (!make_tmap_d(&td, a->d, rows_d, a->n, a->ldd)) return NVQ_ERR_CUDA;
    }
    GemmParams p;
    p.mode = a->mode;
    p.out_f32 = a->out_type == NVQ_OUT_F32;
    p.groups = (int)a->groups;
    p.m = a->m;
    p.n = a->n;
    p.k = a->k;
    p.sfa = static_cast<const uint8_t*>(a->sfa);
    p.sfb = static_cast<const uint8_t*>(a->sfb);
    p.s_a = a->s_a;
    p.s_b = a->s_b;
    p.offsets = a->offsets;
    p.d = a->d;
    p.ldd = a->ldd;
    p.d_aligned32 = ((reinterpret_cast<uintptr_t>(a->d) & 31u) == 0) && (a->ldd % 16 == 0);
    // Box stores through shared memory for grouped row-offset GEMMs whose groups fill their row
    // tiles (MoE forward and data gradient: measured 5-22% faster); per-thread row stores for one
    // group, for per-expert weight gradients (4-8% faster that way) and for groups of a few rows
    // (decode: most warps of a tile have no rows to store).
    p.tma_store = a->out_type == NVQ_OUT_BF16 && a->mode == NVQ_GEMM_GROUP_M && a->groups > 1 &&
                  a->m >= BM * a->groups;
    p.status = a->status;
    p.wait_limit_ns = a->wait_limit_ns > 0 ? (uint64_t)a->wait_limit_ns : WAIT_LIMIT_NS;
    p.inject_stage = a->inject_timeout_stage;
    p.a_rowtiles = (rows_a + BM - 1) / BM;
    p.b_rowtiles = (rows_b + BM - 1) / BM;
    const int64_t kb = a->k / (C::FP4 ? 16 : 32);
    p.sf_tiles_per_row = (kb + 3) / 4;

    static bool attr_ok = false;
    static std::once_flag once;
    std::call_once(once, [] {
        attr_ok = cudaFuncSetAttribute(block_scaled_gemm_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::SMEM_BYTES) == cudaSuccess;
    });
    if (!attr_ok) return NVQ_ERR_CUDA;
    const int grid = num_sms();
    if (grid <= 0) return NVQ_ERR_CUDA;
    // the staging buffers sit at the end of shared memory: launches that store rows directly leave
    // them out (a larger shared-memory request shrinks L1; measured on the decode shape)
    const size_t smem = p.tma_store ? C::SMEM_BYTES : C::SMEM_BYTES - C::STG_BYTES;
    if (launch_pdl(block_scaled_gemm_kernel<FMT>, dim3(grid), dim3(C::THREADS), smem, stream, ta, tb, td, p) !=
            cudaSuccess ||
        cudaGetLastError() != cudaSuccess)
        return NVQ_ERR_CUDA;
    count_launches(1);
    return NVQ_OK;
}

}  // namespace nvq

namespace {
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

extern "C" nvq_status block_scaled_grouped_gemm(const nvq_gemm_args* a, void* stream) {
    if (a == nullptr) return NVQ_ERR_INVALID_ARG;
    if ((a->fmt != NVQ_MXFP8 && a->fmt != NVQ_NVFP4 && a->fmt != NVQ_BF16) ||
        (a->mode != NVQ_GEMM_GROUP_M && a->mode != NVQ_GEMM_GROUP_K) ||
        (a->out_type != NVQ_OUT_BF16 && a->out_type != NVQ_OUT_F32))
        return NVQ_ERR_INVALID_ARG;
    if (a->groups < 0 || a->m < 0 || a->n < 0 || a->k < 0 || a->wait_limit_ns < 0 || a->inject_timeout_stage < 0)
        return NVQ_ERR_INVALID_ARG;
    if (a->groups == 0 || a->m == 0 || a->n == 0) return NVQ_OK;
    if (a->groups > nvq::MAX_GROUPS) return NVQ_ERR_UNSUPPORTED;
    const bool scaled = a->fmt != NVQ_BF16;
    if (a->a == nullptr || a->b == nullptr || a->offsets == nullptr || a->d == nullptr ||
        (scaled && (a->sfa == nullptr || a->sfb == nullptr)))
        return NVQ_ERR_INVALID_ARG;
    if (a->k == 0 || a->n % 128) return NVQ_ERR_INVALID_ARG;
    if (scaled ? a->k % (a->mode == NVQ_GEMM_GROUP_M ? 128 : 32) : a->k % 16) return NVQ_ERR_INVALID_ARG;
    if (a->ldd < a->n || a->ldd % 8) return NVQ_ERR_INVALID_ARG;
    if (a->m > INT32_MAX || a->k > INT32_MAX || a->groups * a->n > INT32_MAX) return NVQ_ERR_UNSUPPORTED;
    if (a->mode == NVQ_GEMM_GROUP_K) {
        if (a->fmt == NVQ_NVFP4) return NVQ_ERR_UNSUPPORTED;
        if (a->m % 128 || a->s_a != nullptr) return NVQ_ERR_INVALID_ARG;
    }
    if (!aligned16(a->a) || !aligned16(a->b) || (scaled && (!aligned16(a->sfa) || !aligned16(a->sfb))) ||
        !aligned16(a->d) || (reinterpret_cast<uintptr_t>(a->offsets) & 7u))
        return NVQ_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (a->fmt == NVQ_NVFP4) return nvq::launch_gemm<nvq::F_NVFP4>(a, s);
    if (a->fmt == NVQ_MXFP8) return nvq::launch_gemm<nvq::F_MXFP8>(a, s);
    return nvq::launch_gemm<nvq::F_BF16>(a, s);
}
