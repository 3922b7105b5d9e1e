// MXFP8 quantizer: rowwise 1x32 and columnwise 32x1 copies of a bf16 matrix in one pass.
//
// Definition [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本",
// section "为什么需要 Blackwell 原生方案？" (32 E4M3 values share an E8M0 power-of-two scale, rounded up
// so the block maximum is not clipped) and section "方案 1：端到端 MXFP8 强化学习" (rowwise 1x32 and
// columnwise 32x1 copies are numerically different and are both quantized from the original
// full-precision data during quantization)].
//
// Design: one CTA per 128 x 128 bf16 tile (32 KB). With a columnwise copy the tile is copied straight
// into shared memory with cp.async (two 256-byte row segments per warp instruction, no registers
// held while the loads are in flight, 5-6 CTAs per SM); the rowwise-only copy keeps the tile in
// registers (4 CTAs per SM, no barrier). The rowwise copy is produced by the same lanes from 16-byte
// pieces (a 1x32 block is four lanes, amax by two xor-shuffles); the columnwise copy by 256
// threads, each owning a column pair of one 32-row block (conflict-free: a warp reads 128
// contiguous bytes of one tile row per access), amax in one sweep of its 32 words and codes in a
// second. The columnwise codes are written transposed, 32 contiguous bytes per column and block.
// Input bytes are read from HBM exactly once.
#include <mutex>

#include "nvq_device.cuh"
#include "nvq_internal.h"

namespace nvq {

constexpr int MX_TILE = 128;
constexpr int MX_THREADS = 256;

// Resident CTAs per SM of each variant (measured on GB300). STAGED: the tile is copied to shared
// memory by cp.async and both copies are made from there (5-6 CTAs per SM; best when the grid is
// many waves deep); otherwise the tile is loaded into registers, the rowwise copy is made straight
// from them and the tile is parked in shared memory for the columnwise copy (4 CTAs per SM; shorter
// per-CTA latency, best for grids of one or two waves).
template <bool ROW, bool COL, bool STAGED>
struct MxOcc {
    static constexpr int value = STAGED ? (ROW ? 6 : 5) : 4;
};

template <bool ROW, bool COL, bool STAGED>
__global__ void __launch_bounds__(MX_THREADS, (MxOcc<ROW, COL, STAGED>::value))
mxfp8_quant_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ldx,
                   uint8_t* __restrict__ q_row, uint8_t* __restrict__ sf_row,
                   uint8_t* __restrict__ q_colT, uint8_t* __restrict__ sf_colT, int mma_layout) {
    griddep_begin();
    __shared__ __align__(16) uint32_t tile[MX_TILE][MX_TILE / 2];   // bf16 pairs
    __shared__ __align__(4) uint8_t sfT_stage[MX_TILE][4];

    const int64_t r0 = (int64_t)blockIdx.y * MX_TILE;
    const int64_t c0 = (int64_t)blockIdx.x * MX_TILE;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool do_row = ROW, do_col = COL;
    const int64_t kb_row = C >> 5;          // scale columns of the rowwise copy
    const int64_t kb_col = R >> 5;          // scale columns of the columnwise copy

    // ---- load: 8 x 16 bytes per thread (zero outside the matrix), either straight to shared memory
    // (cp.async: no registers held while the loads are in flight) or into registers ----
    const int cc = (lane & 15) * 8;
    uint4 v_reg[STAGED ? 1 : 8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int rr = it * 16 + warp * 2 + (lane >> 4);
        const int64_t r = r0 + rr, c = c0 + cc;
        const bool in = r < R && c < C;
        if (STAGED) {
            const uint16_t* src = in ? x + r * ldx + c : x;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                         ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(&tile[rr][cc >> 1]))), "l"(src),
                         "r"(in ? 16 : 0)
                         : "memory");
        } else {
            v_reg[STAGED ? 0 : it] = in ? ld_stream_v4(x + r * ldx + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (STAGED) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
    }

#pragma unroll STAGED ? 2 : 8
    for (int it = 0; it < 8; ++it) {
        const int rr = it * 16 + warp * 2 + (lane >> 4);
        const int64_t r = r0 + rr, c = c0 + cc;
        if (!STAGED && do_col) *reinterpret_cast<uint4*>(&tile[rr][cc >> 1]) = v_reg[STAGED ? 0 : it];
        if (do_row) {
            const uint4 v = STAGED ? *reinterpret_cast<const uint4*>(&tile[rr][cc >> 1]) : v_reg[STAGED ? 0 : it];
            uint32_t m = absmax_bits_8(v);
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const uint32_t sf = e8m0_byte(m << 16);
            const float inv = e8m0_inv_scale(sf);
            const uint32_t w0 = v.x, w1 = v.y, w2 = v.z, w3 = v.w;
            uint32_t o0 = cvt_e4m3x2(bf16_lo(w0) * inv, bf16_hi(w0) * inv) |
                          (cvt_e4m3x2(bf16_lo(w1) * inv, bf16_hi(w1) * inv) << 16);
            uint32_t o1 = cvt_e4m3x2(bf16_lo(w2) * inv, bf16_hi(w2) * inv) |
                          (cvt_e4m3x2(bf16_lo(w3) * inv, bf16_hi(w3) * inv) << 16);
            if (r < R && c < C) *reinterpret_cast<uint2*>(q_row + r * C + c) = make_uint2(o0, o1);
            // gather the four block scales of this 128-column row segment into the segment's lane 0
            const uint32_t s4 = __shfl_down_sync(0xffffffffu, sf, 4);
            const uint32_t s8 = __shfl_down_sync(0xffffffffu, sf, 8);
            const uint32_t s12 = __shfl_down_sync(0xffffffffu, sf, 12);
            if ((lane & 15) == 0) {
                const int64_t kb0 = c0 >> 5;
                if (mma_layout) {
                    if (r < ((R + 127) & ~int64_t(127))) {
                        uint32_t word = sf | (s4 << 8) | (s8 << 16) | (s12 << 24);
                        *reinterpret_cast<uint32_t*>(sf_row + mma_sf_offset(r, kb0, kb_row)) = word;
                    }
                } else if (r < R) {
                    const uint32_t s[4] = {sf, s4, s8, s12};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (kb0 + j < kb_row) sf_row[r * kb_row + kb0 + j] = (uint8_t)s[j];
                }
            }
        }
    }
    if (!do_col) return;
    if (!STAGED) __syncthreads();

    // ---- columnwise: thread = (column pair cp, 32-row block rb). Staged: the block's amax in a
    // first sweep of its 32 words and the codes in a second (few registers); otherwise the 32 words
    // are read once into registers. ----
    const int cp = threadIdx.x & 63, rb = threadIdx.x >> 6;
    uint32_t w[STAGED ? 1 : 32];
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t wi = tile[rb * 32 + i][cp];
        if (!STAGED) w[STAGED ? 0 : i] = wi;
        m2 = __vmaxu2(m2, wi & 0x7FFF7FFFu);
    }
    const uint32_t sf_lo = e8m0_byte((m2 & 0xFFFFu) << 16);
    const uint32_t sf_hi = e8m0_byte(m2 & 0xFFFF0000u);
    const float inv_lo = e8m0_inv_scale(sf_lo), inv_hi = e8m0_inv_scale(sf_hi);
    const int64_t c = c0 + 2 * cp;
    const int64_t rs = r0 + rb * 32;
    if (c < C && rs < R) {
        uint32_t olo[8], ohi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t a[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) a[j] = STAGED ? tile[rb * 32 + 4 * i + j][cp] : w[STAGED ? 0 : 4 * i + j];
            olo[i] = cvt_e4m3x2(bf16_lo(a[0]) * inv_lo, bf16_lo(a[1]) * inv_lo) |
                     (cvt_e4m3x2(bf16_lo(a[2]) * inv_lo, bf16_lo(a[3]) * inv_lo) << 16);
            ohi[i] = cvt_e4m3x2(bf16_hi(a[0]) * inv_hi, bf16_hi(a[1]) * inv_hi) |
                     (cvt_e4m3x2(bf16_hi(a[2]) * inv_hi, bf16_hi(a[3]) * inv_hi) << 16);
        }
        // each column's 32 codes are one 32-byte sector (R % 32 == 0, rs a multiple of 32): one
        // 256-bit store when q_colT is 32-byte aligned, so no store instruction writes half sectors
        uint8_t* plo = q_colT + c * R + rs;
        uint8_t* phi = q_colT + (c + 1) * R + rs;
        if ((reinterpret_cast<uintptr_t>(q_colT) & 31u) == 0) {
            st_sector(plo, make_uint4(olo[0], olo[1], olo[2], olo[3]), make_uint4(olo[4], olo[5], olo[6], olo[7]));
            st_sector(phi, make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]), make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]));
        } else {
            reinterpret_cast<uint4*>(plo)[0] = make_uint4(olo[0], olo[1], olo[2], olo[3]);
            reinterpret_cast<uint4*>(plo)[1] = make_uint4(olo[4], olo[5], olo[6], olo[7]);
            reinterpret_cast<uint4*>(phi)[0] = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
            reinterpret_cast<uint4*>(phi)[1] = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
        }
    }
    sfT_stage[2 * cp][rb] = (uint8_t)sf_lo;
    sfT_stage[2 * cp + 1][rb] = (uint8_t)sf_hi;
    __syncthreads();
    if (threadIdx.x < MX_TILE) {
        const int64_t cr = c0 + threadIdx.x;             // row of the transposed copy
        const int64_t kb0 = r0 >> 5;
        const uint32_t word = *reinterpret_cast<const uint32_t*>(&sfT_stage[threadIdx.x][0]);
        if (mma_layout) {
            if (cr < ((C + 127) & ~int64_t(127)))
                *reinterpret_cast<uint32_t*>(sf_colT + mma_sf_offset(cr, kb0, kb_col)) = word;
        } else if (cr < C) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (kb0 + j < kb_col) sf_colT[cr * kb_col + kb0 + j] = (uint8_t)(word >> (8 * j));
        }
    }
}

cudaError_t launch_mxfp8_quantize(const uint16_t* x, int64_t R, int64_t C, int64_t ldx,
                                  uint8_t* q_row, uint8_t* sf_row, uint8_t* q_colT, uint8_t* sf_colT,
                                  int mma_layout, cudaStream_t stream) {
    // the MMA layout pads rows to 128: cover the padded rows so the padding gets zero scales
    dim3 grid((unsigned)((C + MX_TILE - 1) / MX_TILE), (unsigned)((R + MX_TILE - 1) / MX_TILE));
    static int sms = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            sms = 0;
    });
    // grids deeper than two waves of the register variant are staged through shared memory, and so
    // are grids just past one register wave that fit one wave of the staged variant (its extra
    // resident CTAs take the whole grid at once instead of leaving a short second round)
    const int64_t tiles = (int64_t)grid.x * grid.y, reg_wave = (int64_t)MxOcc<true, true, false>::value * sms;
    const int64_t staged_wave = (int64_t)(q_row ? MxOcc<true, true, true>::value : MxOcc<false, true, true>::value) * sms;
    const bool staged = tiles > 2 * reg_wave || (tiles > reg_wave && tiles <= staged_wave);
    cudaError_t lerr;
#define NVQ_MX(RW, CL, ST)                                                                                       \
    lerr = launch_pdl(mxfp8_quant_kernel<RW, CL, ST>, grid, dim3(MX_THREADS), 0, stream, x, R, C, ldx, q_row, sf_row, \
                      q_colT, sf_colT, mma_layout)
    if (q_row && q_colT) {
        if (staged) NVQ_MX(true, true, true);
        else NVQ_MX(true, true, false);
    } else if (q_colT) {
        if (staged) NVQ_MX(false, true, true);
        else NVQ_MX(false, true, false);
    } else {
        NVQ_MX(true, false, false);
    }
#undef NVQ_MX
    const cudaError_t err = lerr != cudaSuccess ? lerr : cudaGetLastError();
    if (err == cudaSuccess) count_launches(1);
    return err;
}

}  // namespace nvq
