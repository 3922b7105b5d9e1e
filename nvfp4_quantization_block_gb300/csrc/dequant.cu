// BF16 dequantization of MXFP8 / NVFP4 operands (the dequantized-backward mode).
//
// Definition [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本", section
// "高精度反向和去量化反向": the backward GEMMs run in BF16 on the dequantization of the exact
// low-precision operands produced by the forward pass]: out = RN_bf16(exact value).
//   MXFP8: E4M3(q) * 2^(sf-127) is an exact fp32 product (4 significant bits times a power of
//          two), so one hardware bf16 conversion rounds it once.
//   NVFP4: E2M1(q) * E4M3(sf) is exact in fp32; its product with the fp32 coarse scale s has up to
//          30 significant bits. It is formed as t = RZ(p * s) plus the exact remainder
//          fma(p, s, -t); the remainder's sign sets the last bit of t (round to odd), after which
//          the bf16 conversion yields the single rounding of the exact product (Boldo & Melquiond,
//          IEEE TC 2008). Tiny products, where the remainder could underflow, use fp64.
// One thread produces one 32-element (MXFP8) block, or four (rows of a multiple of 64 elements) or
// two 16-element NVFP4 blocks, with one scale byte per block, streaming through HBM once. NVFP4
// blocks look their 16 results up in a per-block table of the 8 possible bf16 values (byte
// permutes), so the E2M1 conversion instruction, which issues on a low-throughput pipe, is not
// used per element.
#include "nvq_device.cuh"
#include "nvq_internal.h"

namespace nvq {

__device__ __forceinline__ int64_t sf_index(int64_t row, int64_t kb, int64_t nkb, int mma_layout) {
    return mma_layout ? mma_sf_offset(row, kb, nkb) : row * nkb + kb;
}

// (row, block) of block index blk in a [rows, nkb] block grid; 32-bit division when the grid has
// fewer than 2^32 blocks (a 64-bit division expands to several dozen instructions)
__device__ __forceinline__ void block_coords(int64_t blk, int64_t nkb, bool small, int64_t& row, int64_t& kb) {
    if (small) {
        const uint32_t r = (uint32_t)blk / (uint32_t)nkb;
        row = r;
        kb = (int64_t)((uint32_t)blk - r * (uint32_t)nkb);
    } else {
        row = blk / nkb;
        kb = blk - row * nkb;
    }
}

__global__ void __launch_bounds__(256)
dequant_mxfp8_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf, int64_t rows,
                     int64_t cols, int mma_layout, uint16_t* __restrict__ out) {
    griddep_begin();
    const int64_t nkb = cols >> 5;
    const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nblk = rows * nkb;
    if (blk >= nblk) return;
    int64_t row, kb;
    block_coords(blk, nkb, nblk <= 0xFFFFFFFFll, row, kb);
    const float scale = e8m0_scale(sf[sf_index(row, kb, nkb, mma_layout)]);
    const uint8_t* src = q + row * cols + kb * 32;
    const uint4 a = ld_stream_v4(src), b = ld_stream_v4(src + 16);
    const uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float f0, f1, f2, f3;
        e4m3x2_to_f32(in[i] & 0xFFFFu, f0, f1);
        e4m3x2_to_f32(in[i] >> 16, f2, f3);
        o[2 * i] = cvt_bf16x2(f0 * scale, f1 * scale);
        o[2 * i + 1] = cvt_bf16x2(f2 * scale, f3 * scale);
    }
    // the block's 64 output bytes: two 256-bit stores of whole sectors when out is 32-byte aligned
    uint16_t* dst = out + row * cols + kb * 32;
    if ((reinterpret_cast<uintptr_t>(out) & 31u) == 0) {
        st_sector(dst, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
        st_sector(dst + 16, make_uint4(o[8], o[9], o[10], o[11]), make_uint4(o[12], o[13], o[14], o[15]));
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            reinterpret_cast<uint4*>(dst)[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
}

// RN_bf16(p * s) for exact fp32 p and s (both finite).
__device__ __forceinline__ float round_odd_product(float p, float s) {
    const float t = __fmul_rz(p, s);
    if (fabsf(t) >= 0x1p-96f) {
        const float r = fmaf(p, s, -t);
        return r != 0.0f ? __uint_as_float(__float_as_uint(t) | 1u) : t;
    }
    if (p == 0.0f || s == 0.0f) return t;
    return f64_to_f32_round_odd((double)p * (double)s);
}

// One 16-element block: every element takes one of 8 magnitudes times the block's scale product,
// so the block's 8 possible bf16 results are computed once (round-to-odd products) and the codes
// select them with byte permutes; the sign bit is copied from the code. No per-element conversion.
__device__ __forceinline__ void dequant_nvfp4_block(uint2 packed, float v_sf, float coarse, uint4& d0, uint4& d1) {
    // bf16 results for magnitude codes 0..7 = {0, .5, 1, 1.5, 2, 3, 4, 6} x v_sf x coarse
    const uint32_t p01 = cvt_bf16x2(0.0f, round_odd_product(0.5f * v_sf, coarse));
    const uint32_t p23 = cvt_bf16x2(round_odd_product(v_sf, coarse), round_odd_product(1.5f * v_sf, coarse));
    const uint32_t p45 = cvt_bf16x2(round_odd_product(2.0f * v_sf, coarse), round_odd_product(3.0f * v_sf, coarse));
    const uint32_t p67 = cvt_bf16x2(round_odd_product(4.0f * v_sf, coarse), round_odd_product(6.0f * v_sf, coarse));
    const uint32_t lo_a = __byte_perm(p01, p23, 0x6420), hi_a = __byte_perm(p01, p23, 0x7531);
    const uint32_t lo_b = __byte_perm(p45, p67, 0x6420), hi_b = __byte_perm(p45, p67, 0x7531);
    uint32_t o[8];
    const uint32_t in[2] = {packed.x, packed.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t qq = in[i >> 1] >> (16 * (i & 1));       // codes of elements 4i .. 4i+3
        const uint32_t sel = qq & 0x7777u;
        const uint32_t lo = __byte_perm(lo_a, lo_b, sel), hi = __byte_perm(hi_a, hi_b, sel);
        o[2 * i] = __byte_perm(lo, hi, 0x5140) | ((qq << 12) & 0x8000u) | ((qq << 24) & 0x80000000u);
        o[2 * i + 1] = __byte_perm(lo, hi, 0x7362) | ((qq << 4) & 0x8000u) | ((qq << 16) & 0x80000000u);
    }
    d0 = make_uint4(o[0], o[1], o[2], o[3]);
    d1 = make_uint4(o[4], o[5], o[6], o[7]);
}

// Two blocks per thread: blocks 2t and 2t + 1 of the row-major block grid (the same row unless
// the row has an odd number of blocks).
__global__ void __launch_bounds__(256)
dequant_nvfp4_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                     const float* __restrict__ s, int64_t rows_per_group, int64_t total_rows,
                     int64_t cols, int scope_matrix, int mma_layout, uint16_t* __restrict__ out) {
    griddep_begin();
    const int64_t nkb = cols >> 4;
    const int64_t nblk = total_rows * nkb;
    const int64_t blk0 = 2 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x);
    if (blk0 >= nblk) return;
    const bool small = nblk <= 0xFFFFFFFFll;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int64_t blk = blk0 + h;
        if (blk >= nblk) break;
        int64_t row, kb;
        block_coords(blk, nkb, small, row, kb);
        int64_t scope = row;
        if (scope_matrix) {
            if (small) scope = (int64_t)((uint32_t)row / (uint32_t)rows_per_group);
            else scope = row / rows_per_group;
        }
        const float coarse = s[scope];
        const float v_sf = e4m3_to_f32(sf[sf_index(row, kb, nkb, mma_layout)]);
        const uint2 packed = *reinterpret_cast<const uint2*>(q + row * (cols >> 1) + kb * 8);
        uint4 d0, d1;
        dequant_nvfp4_block(packed, v_sf, coarse, d0, d1);
        uint4* dst = reinterpret_cast<uint4*>(out + row * cols + kb * 16);
        dst[0] = d0;
        dst[1] = d1;
    }
}

// Four blocks per thread (64 elements of one row: blocks 4t .. 4t + 3 of the row-major grid of
// 4-block groups): one 32-byte code load, the four scale bytes as one word (a row's four
// consecutive blocks are adjacent bytes in both scale layouts), and four 256-bit stores that each
// fill one whole 32-byte sector, so a warp's store instruction writes 32 complete sectors. For rows
// of a multiple of 64 elements with q and out 32-byte aligned and sf 4-byte aligned.
__global__ void __launch_bounds__(256)
dequant_nvfp4_x4_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                        const float* __restrict__ s, int64_t rows_per_group, int64_t total_rows,
                        int64_t cols, int scope_matrix, int mma_layout, uint16_t* __restrict__ out) {
    griddep_begin();
    const int64_t nkb = cols >> 4;                             // a multiple of 4
    const int64_t ngrp = total_rows * (nkb >> 2);
    const int64_t grp = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (grp >= ngrp) return;
    const bool small = ngrp <= 0xFFFFFFFFll;
    int64_t row, kq;
    block_coords(grp, nkb >> 2, small, row, kq);
    const int64_t kb = 4 * kq;
    int64_t scope = row;
    if (scope_matrix) {
        if (small) scope = (int64_t)((uint32_t)row / (uint32_t)rows_per_group);
        else scope = row / rows_per_group;
    }
    const float coarse = s[scope];
    const uint32_t sfw = *reinterpret_cast<const uint32_t*>(sf + sf_index(row, kb, nkb, mma_layout));
    uint4 a, b;
    ld_v8(q + row * (cols >> 1) + kb * 8, a, b);
    const uint2 packed[4] = {make_uint2(a.x, a.y), make_uint2(a.z, a.w), make_uint2(b.x, b.y), make_uint2(b.z, b.w)};
    uint16_t* dst = out + row * cols + kb * 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 d0, d1;
        dequant_nvfp4_block(packed[i], e4m3_to_f32((uint8_t)(sfw >> (8 * i))), coarse, d0, d1);
        st_sector(dst + 16 * i, d0, d1);
    }
}

cudaError_t launch_dequantize_bf16(int fmt_nvfp4, const uint8_t* q, const uint8_t* sf, const float* s,
                                   int scope_matrix, int64_t groups, int64_t rows, int64_t cols,
                                   int mma_layout, uint16_t* out, cudaStream_t stream) {
    const int64_t total_rows = groups * rows;
    cudaError_t lerr;
    if (!fmt_nvfp4) {
        const int64_t nblk = total_rows * (cols >> 5);
        lerr = launch_pdl(dequant_mxfp8_kernel, dim3((unsigned)((nblk + 255) / 256)), dim3(256), 0, stream, q, sf,
                          total_rows, cols, mma_layout, out);
    } else if (cols % 64 == 0 && (reinterpret_cast<uintptr_t>(q) & 31u) == 0 &&
               (reinterpret_cast<uintptr_t>(out) & 31u) == 0 && (reinterpret_cast<uintptr_t>(sf) & 3u) == 0) {
        const int64_t threads = total_rows * (cols >> 6);
        lerr = launch_pdl(dequant_nvfp4_x4_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, stream, q,
                          sf, s, rows, total_rows, cols, scope_matrix, mma_layout, out);
    } else {
        const int64_t nblk = total_rows * (cols >> 4);
        const int64_t threads = (nblk + 1) / 2;
        lerr = launch_pdl(dequant_nvfp4_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, stream, q, sf,
                          s, rows, total_rows, cols, scope_matrix, mma_layout, out);
    }
    const cudaError_t err = lerr != cudaSuccess ? lerr : cudaGetLastError();
    if (err == cudaSuccess) count_launches(1);
    return err;
}

}  // namespace nvq
