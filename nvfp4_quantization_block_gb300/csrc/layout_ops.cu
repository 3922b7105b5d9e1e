// Scale-layout conversion and the gather of quantized rows (quantize-once dispatch).
//
// Layout conversion [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本",
// section "重构权重更新接口": backend-specific swizzled layouts must stay explicit and verifiable]: the
// tcgen05 block-scale tile layout is a pure permutation of the canonical [rows, kb] scale bytes
// (128-row x 4-column tiles of 512 bytes, the scale of (r, c) at (r % 32) 16 + (r % 128 / 32) 4 +
// c % 4, tiles row-tile major, zero padding), so one 4-scale word of a row is contiguous in both.
//
// Gather [Miles-zh, section "逐 Token 激活值缩放": one FP32 scale per token, so a token's quantized
// bytes depend on its own row only]: quantizing the tokens once and gathering their packed rows,
// block scales and token scales into expert order gives the same bytes as quantizing the gathered
// bf16 rows, with 1/topk of the quantization work. Index -1 marks a padding row: zero codes, zero
// scales and a zero token scale, which is exactly what quantizing a zero row gives.
#include <cstdint>

#include "../../include/nvq.h"
#include "nvq_device.cuh"
#include "nvq_internal.h"

namespace nvq {

constexpr int LO_ROWS = 8;            // rows per CTA of the conversion kernel (one warp each)

// One warp per row r of the padded tile layout, one lane per 4-scale word.
template <bool TO_MMA>
__global__ void __launch_bounds__(32 * LO_ROWS)
sf_convert_kernel(const uint8_t* __restrict__ src, int64_t rows, int64_t kb, uint8_t* __restrict__ dst,
                  int64_t rows_cover) {
    griddep_begin();
    const int64_t r = (int64_t)blockIdx.x * LO_ROWS + threadIdx.y;
    if (r >= rows_cover) return;
    const int64_t words = (kb + 3) >> 2;
    for (int64_t wd = threadIdx.x; wd < words; wd += 32) {
        const int64_t c0 = wd << 2;
        if (TO_MMA) {
            uint32_t word = 0;
            if (r < rows) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (c0 + j < kb) word |= (uint32_t)src[r * kb + c0 + j] << (8 * j);
            }
            *reinterpret_cast<uint32_t*>(dst + mma_sf_offset(r, c0, kb)) = word;
        } else {
            const uint32_t word = *reinterpret_cast<const uint32_t*>(src + mma_sf_offset(r, c0, kb));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c0 + j < kb) dst[r * kb + c0 + j] = (uint8_t)(word >> (8 * j));
        }
    }
}

cudaError_t launch_sf_layout_convert(const uint8_t* src, int to_mma, int64_t rows, int64_t kb, uint8_t* dst,
                                     cudaStream_t stream) {
    const int64_t cover = to_mma ? ((rows + 127) & ~int64_t(127)) : rows;
    const dim3 block(32, LO_ROWS);
    const unsigned grid = (unsigned)((cover + LO_ROWS - 1) / LO_ROWS);
    const cudaError_t lerr =
        to_mma ? launch_pdl(sf_convert_kernel<true>, dim3(grid), block, 0, stream, src, rows, kb, dst, cover)
               : launch_pdl(sf_convert_kernel<false>, dim3(grid), block, 0, stream, src, rows, kb, dst, cover);
    const cudaError_t err = lerr != cudaSuccess ? lerr : cudaGetLastError();
    if (err == cudaSuccess) count_launches(1);
    return err;
}

// One warp per output row i: source row index[i] (-1: a zero row). The packed codes move in
// 8-byte pieces (a row is a multiple of 8 bytes), the scales as 4-scale words in either layout.
template <bool SRC_MMA, bool DST_MMA>
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf, const float* __restrict__ s,
                   int64_t src_rows, int64_t qbytes, int64_t kb, const int32_t* __restrict__ index, int64_t rows,
                   int64_t rows_cover, uint8_t* __restrict__ q_out, uint8_t* __restrict__ sf_out,
                   float* __restrict__ s_out, int32_t* __restrict__ status) {
    griddep_begin();
    const int lane = threadIdx.x & 31;
    const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (i >= rows_cover) return;
    int64_t src = -1;
    if (i < rows) {
        src = index[i];
        if (src < -1 || src >= src_rows) {
            if (lane == 0 && status) atomicExch(status, NVQ_DEV_BAD_INDEX);
            src = -1;
        }
        uint2* to = reinterpret_cast<uint2*>(q_out + i * qbytes);
        if (src >= 0) {
            const uint2* from = reinterpret_cast<const uint2*>(q + src * qbytes);
            for (int64_t p = lane; p < (qbytes >> 3); p += 32) to[p] = from[p];
        } else {
            for (int64_t p = lane; p < (qbytes >> 3); p += 32) to[p] = make_uint2(0u, 0u);
        }
        if (s_out && lane == 0) s_out[i] = src >= 0 ? s[src] : 0.0f;
    }
    const int64_t words = (kb + 3) >> 2;
    for (int64_t wd = lane; wd < words; wd += 32) {
        const int64_t c0 = wd << 2;
        uint32_t word = 0;
        if (src >= 0) {
            if (SRC_MMA) {
                word = *reinterpret_cast<const uint32_t*>(sf + mma_sf_offset(src, c0, kb));
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (c0 + j < kb) word |= (uint32_t)sf[src * kb + c0 + j] << (8 * j);
            }
        }
        if (DST_MMA) {
            *reinterpret_cast<uint32_t*>(sf_out + mma_sf_offset(i, c0, kb)) = word;
        } else if (i < rows) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c0 + j < kb) sf_out[i * kb + c0 + j] = (uint8_t)(word >> (8 * j));
        }
    }
}

cudaError_t launch_quantized_gather_rows(const uint8_t* q, const uint8_t* sf, const float* s, int64_t src_rows,
                                         int64_t qbytes, int64_t kb, int src_mma, const int32_t* index, int64_t rows,
                                         uint8_t* q_out, uint8_t* sf_out, float* s_out, int dst_mma,
                                         int32_t* status, cudaStream_t stream) {
    const int64_t cover = dst_mma ? ((rows + 127) & ~int64_t(127)) : rows;
    const unsigned grid = (unsigned)((cover + 7) / 8);
    cudaError_t lerr;
#define NVQ_GATHER(SM, DM)                                                                                 \
    lerr = launch_pdl(gather_rows_kernel<SM, DM>, dim3(grid), dim3(256), 0, stream, q, sf, s, src_rows, qbytes, \
                      kb, index, rows, cover, q_out, sf_out, s_out, status)
    if (src_mma && dst_mma) NVQ_GATHER(true, true);
    else if (src_mma) NVQ_GATHER(true, false);
    else if (dst_mma) NVQ_GATHER(false, true);
    else NVQ_GATHER(false, false);
#undef NVQ_GATHER
    const cudaError_t err = lerr != cudaSuccess ? lerr : cudaGetLastError();
    if (err == cudaSuccess) count_launches(1);
    return err;
}

}  // namespace nvq
