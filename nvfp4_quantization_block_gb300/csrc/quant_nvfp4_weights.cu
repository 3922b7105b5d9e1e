// NVFP4 expert weights: one FP32 scale per expert matrix, 1x16 blocks along the reduction
// dimension, codes and scales written K-major for the GEMM.
//
// Definition [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本":
// section "为什么需要 Blackwell 原生方案？" (E2M1 values, one E4M3 scale per 16 values rounded to
// nearest, a coarse FP32 scale on top); section "逐 Token 激活值缩放" (gate and up weights feed one
// fused GEMM and share one FP32 scale); section "移除额外的 BF16 权重副本" (1-D 1x16 weight blocks);
// section "比特精确量化器合约" (bit-exact contract)]. Coarse scale s = RN(amax / 2688) over the
// expert matrix; block scale = E4M3 RNE of amax_b / (6 s); code = E2M1 RNE (saturating) of
// x / (E4M3(sf) s). An expert whose table passes the product-path check (nvq_device.cuh) encodes
// its elements by one fp32 multiply and the hardware E2M1 conversion; any other expert compares
// each element with its block's exact boundaries.
#include <algorithm>
#include <mutex>

#include "nvq_device.cuh"
#include "nvq_internal.h"
#include "nvq_nvfp4_encode.cuh"

namespace nvq {

// ------------------------------------------------------------------------------------------------
// Weights: W [E, K, N] -> qT [E, N, K/2], sfT [E, N, K/16], s_w [E]; coarse scope = expert matrix.
// Kernels: amax per expert (atomic max on the fp32 bits, kept in s_w); for more than one expert a
// check kernel (s_w <- coarse scale with a product-path flag, for a cost-weighted split of the
// encode work); encode; finalize (s_w <- RN(amax / 2688), or the flag cleared).
// ------------------------------------------------------------------------------------------------
constexpr int WA_VEC = 4;                // 16-byte vectors in flight per thread in the amax pass

__global__ void __launch_bounds__(256)
nvfp4_weight_amax_kernel(const uint16_t* __restrict__ w, int64_t per_expert, uint32_t* __restrict__ amax_bits) {
    griddep_begin();
    const int64_t e = blockIdx.y;
    const uint16_t* we = w + e * per_expert;
    const int64_t nvec = per_expert >> 3;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t m = 0;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // WA_VEC independent loads issued before any of them is used
    for (; i + (WA_VEC - 1) * stride < nvec; i += WA_VEC * stride) {
        uint4 v[WA_VEC];
#pragma unroll
        for (int j = 0; j < WA_VEC; ++j) v[j] = ld_stream_v4(we + (i + j * stride) * 8);
#pragma unroll
        for (int j = 0; j < WA_VEC; ++j) m = max(m, absmax_bits_8(v[j]));
    }
    for (; i < nvec; i += stride) m = max(m, absmax_bits_8(ld_stream_v4(we + i * 8)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ uint32_t red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = red[0];
        for (int j = 1; j < (int)(blockDim.x >> 5); ++j) t = max(t, red[j]);
        if (t) atomicMax(amax_bits + e, t << 16);    // non-negative floats order like their bits
    }
}

// Encode: the CTA's warps take adjacent 64-column strips of the same 64 rows (a super-tile of
// WE_WARPS x 64 columns, so each row is read as WE_WARPS x 128 contiguous bytes), and CTAs take
// contiguous ranges of the (expert, super-strip, k tile) sequence, k fastest (equal unit counts for
// one expert, equal shares of the expected cost for several: see the check kernel), so a warp
// rebuilds its scope table only when its range enters the next expert. Each warp stages its strip through a ring of WE_STAGES 32-row half tiles in shared
// memory, filled by 16-byte cp.async copies WE_STAGES - 1 half tiles ahead of the one it encodes,
// so loads stay in flight without holding registers (the encode work per byte is high, and a
// register pipeline held the warps to 12 per SM). Lane l owns columns n0 + 2l and n0 + 2l + 1: it
// reads the 4 bytes of its two columns from each staged row (a row's 128 bytes across the warp,
// no bank conflict), so each column's block is the low or high halves of one word per row and no
// transpose is needed. Its outputs are whole per column: the tile's four blocks' 32 code bytes
// (one L2 sector, one store) and their 4 scale bytes (one 4-column group); consecutive tiles of a
// warp continue the same columns' rows. (Half-sector code stores, 16 bytes per tile, made L2 write
// partial sectors back: 3.4x the output bytes in DRAM writes.)
constexpr int WE_K = 64, WE_N = 64, WE_WARPS = 4, WE_THREADS = WE_WARPS * 32, WE_STAGES = 3;
constexpr int WE_HALF_BYTES = (WE_K / 2) * WE_N * 2;           // one staged half tile: 32 rows x 128 B
constexpr int WE_SMEM_BYTES = WE_WARPS * WE_STAGES * WE_HALF_BYTES;

// Pairs (x[2i], x[2i + 1]) of one column of 8 rows, as the bf16x2 words of the table and exact
// paths: the column is the low (HI false) or high half of each row's word.
template <bool HI>
__device__ __forceinline__ uint4 column_pairs(const uint32_t* r) {
    constexpr uint32_t sel = HI ? 0x7632u : 0x5410u;
    return make_uint4(__byte_perm(r[0], r[1], sel), __byte_perm(r[2], r[3], sel), __byte_perm(r[4], r[5], sel),
                      __byte_perm(r[6], r[7], sel));
}

// RN_fp32(a g), RN_fp32(b g): one packed fp32 multiply (two IEEE products, no flush to zero)
__device__ __forceinline__ void mul2_rn(float a, float b, float g, float& ya, float& yb) {
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\t"
        "mul.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(ya), "=f"(yb) : "f"(a), "f"(b), "f"(g));
}

// fp32 values of 8 rows of one column, times g, to 8 E2M1 codes (product path)
template <bool HI>
__device__ __forceinline__ uint32_t column_codes_mul(const uint32_t* r, float g) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2)
        mul2_rn(HI ? bf16_hi(r[i]) : bf16_lo(r[i]), HI ? bf16_hi(r[i + 1]) : bf16_lo(r[i + 1]), g, x[i], x[i + 1]);
    return cvt_e2m1x8(x[0], x[1], x[2], x[3], x[4], x[5], x[6], x[7]);
}

// Running magnitude maximum of two bf16 columns (one per half): max.xorsign.abs keeps the larger
// magnitude of each half, with a sign of no meaning that the caller clears. Finite inputs.
__device__ __forceinline__ uint32_t absmax2_bf16x2(uint32_t m, uint32_t w) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(m), "r"(w));
    return d;
}

struct BlockCodes {
    uint32_t sfc, c0, c1;
};

// Table or exact decisions for one column's 16-row block (the four pair words of each half): kept
// out of line, so the product path's loop stays small.
__device__ __noinline__ BlockCodes column_block_slow(uint4 a, uint4 b, uint32_t mb, int mode, Nvfp4Scope sc,
                                                     const Nvfp4Table* T, const Nvfp4CodeInfo* I) {
    BlockCodes r;
    if (mode == ENC_TABLE) r.sfc = encode_block<ENC_TABLE>(a, b, mb, sc, *T, *I, r.c0, r.c1);
    else r.sfc = encode_block<ENC_EXACT>(a, b, mb, sc, *T, *I, r.c0, r.c1);
    return r;
}

// Scale code and codes of one column's 16-row block (rows r[0..15], the column in the low or high
// halves), magnitude maximum mb
template <bool HI>
__device__ __forceinline__ BlockCodes column_block(const uint32_t* r, uint32_t mb, int mode, const Nvfp4Scope& sc,
                                                   const Nvfp4Table& T, const Nvfp4CodeInfo& I) {
    if (mode == ENC_PRODUCT) {
        BlockCodes o;
        o.sfc = nvfp4_block_scale_t(mb, sc, T);
        const float g = nvfp4_block_g(o.sfc, T, I);
        o.c0 = column_codes_mul<HI>(r, g);
        o.c1 = column_codes_mul<HI>(r + 8, g);
        return o;
    }
    return column_block_slow(column_pairs<HI>(r), column_pairs<HI>(r + 8), mb, mode, sc, &T, &I);
}

// (expert, super-strip, k tile, half) cursor over the half tiles of a CTA's range
struct WeCursor {
    int64_t e, st, kt;
    int half;
    __device__ __forceinline__ void next(int64_t tiles_k, int64_t strips) {
        if (++half < 2) return;
        half = 0;
        if (++kt < tiles_k) return;
        kt = 0;
        if (++st < strips) return;
        st = 0;
        ++e;
    }
};

// Weighted split (more than one expert). An expert whose table fails the product-path check
// encodes each element by boundary comparisons, which measured about 1.5x the product path's time
// per unit on GB300; with equal unit counts per CTA, the CTAs inside such an expert set the
// kernel's end while the rest of the GPU idles. So a check kernel (one warp per expert) turns the
// amax bits into the coarse scale s ahead of the encode kernel and records the outcome of the
// check in the sign bit of s_w (s >= 0, so the bit is free until the finalize kernel clears it),
// and the encode kernel gives each CTA an equal share of the summed unit costs. The flag steers
// only the split: every warp still takes its own mode decision from its table.
constexpr int WC_WARPS = 4;

__global__ void __launch_bounds__(WC_WARPS * 32)
nvfp4_weight_check_kernel(uint32_t* __restrict__ s_w, int64_t E) {
    griddep_begin();
    __shared__ Nvfp4Table tables[WC_WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t e = (int64_t)blockIdx.x * WC_WARPS + warp;
    if (e >= E) return;                                        // uniform over the warp
    const float s = nvfp4_coarse_scale(__uint_as_float(s_w[e]));
    const bool exact = make_nvfp4_scope(s).exact;
    const bool all = __all_sync(0xffffffffu, nvfp4_table_build_warp(tables[warp], s, lane));
    if (lane == 0) s_w[e] = __float_as_uint(s) | ((exact || !all) ? 0x80000000u : 0u);
}

// Relative cost of one unit of an expert, from its flagged scale: product path 2, boundary
// comparisons 3, exact decisions (tiny or zero scale; rare) 6.
__device__ __forceinline__ int64_t we_unit_cost(uint32_t sbits) {
    const float s = __uint_as_float(sbits & 0x7FFFFFFFu);
    return !(s >= NVQ_FAST_MIN_SCALE) ? 6 : ((sbits >> 31) ? 3 : 2);
}

// Units [u0, u1) of CTA b of G when the CTAs take equal shares of the summed unit costs; units
// run in expert order, per_e per expert, and a cost position x maps to the first unit whose cost
// starts at or after x (so neighbouring CTAs meet at the same unit). Called by one whole warp.
__device__ __noinline__ void we_weighted_range(const uint32_t* __restrict__ s_w, int64_t E, int64_t per_e, int64_t b, int64_t G,
                                  int lane, int64_t& u0, int64_t& u1) {
    int64_t t = 0;
    for (int64_t e = lane; e < E; e += 32) t += we_unit_cost(s_w[e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const int64_t T = t * per_e;
    const int64_t x0 = T * b / G, x1 = T * (b + 1) / G;
    int64_t r0 = -1, r1 = -1, P = 0;                           // P: cost of the experts before this chunk
    for (int64_t base = 0; base < E; base += 32) {
        const int64_t e = base + lane;
        const int64_t c = e < E ? we_unit_cost(s_w[e]) : 0;
        int64_t incl = c * per_e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int64_t end = P + incl, start = end - c * per_e;  // expert e's cost range [start, end)
        if (c > 0 && x0 >= start && x0 < end) r0 = e * per_e + (x0 - start + c - 1) / c;
        if (c > 0 && x1 >= start && x1 < end) r1 = e * per_e + (x1 - start + c - 1) / c;
        P += __shfl_sync(0xffffffffu, incl, 31);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        r0 = max(r0, (int64_t)__shfl_xor_sync(0xffffffffu, r0, o));
        r1 = max(r1, (int64_t)__shfl_xor_sync(0xffffffffu, r1, o));
    }
    u0 = r0 < 0 ? E * per_e : r0;                              // x == T: past the last unit
    u1 = r1 < 0 ? E * per_e : r1;
}

__global__ void __launch_bounds__(WE_THREADS, 4)
nvfp4_weight_encode_kernel(const uint16_t* __restrict__ w, int64_t K, int64_t N, int64_t tiles_k, int64_t strips,
                           int64_t total, uint8_t* __restrict__ qT, uint8_t* __restrict__ sfT,
                           const uint32_t* __restrict__ amax_bits, int mma_layout, int weighted) {
    griddep_begin();
    extern __shared__ __align__(128) uint8_t we_stage[];
    __shared__ Nvfp4Table tables[WE_WARPS];                    // each warp's current expert
    __shared__ Nvfp4CodeInfo I;
    __shared__ int64_t range[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t per_e = tiles_k * strips;
    for (uint32_t c = threadIdx.x; c < 128u; c += WE_THREADS) nvfp4_code_info_build(I, c);
    if (warp == 0) {
        int64_t b0, b1;
        if (weighted) {
            we_weighted_range(amax_bits, total / per_e, per_e, blockIdx.x, gridDim.x, lane, b0, b1);
        } else {
            b0 = total * blockIdx.x / gridDim.x;
            b1 = total * (blockIdx.x + 1) / gridDim.x;
        }
        if (lane == 0) {
            range[0] = b0;
            range[1] = b1;
        }
    }
    __syncthreads();

    Nvfp4Table& T = tables[warp];
    const int64_t u_begin = range[0], u_end = range[1];
    if (u_begin >= u_end) return;                              // uniform over the CTA
    WeCursor cur;                                              // the half tile being encoded
    cur.e = u_begin / per_e;
    cur.st = (u_begin - cur.e * per_e) / tiles_k;
    cur.kt = u_begin - cur.e * per_e - cur.st * tiles_k;
    cur.half = 0;
    WeCursor fill = cur;                                       // the next half tile to request
    const int64_t halves = 2 * (u_end - u_begin);
    int64_t requested = 0;
    int fill_slot = 0, read_slot = 0;                          // ring slots of the next request / read
    const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(we_stage)) +
                          (uint32_t)(warp * WE_STAGES * WE_HALF_BYTES);
    // copy i of lane l: row 4i + l / 8 of the half tile, 16-byte chunk l % 8 of it
    const int lr = lane >> 3, lch = lane & 7;
    const uint32_t lane_dst = (uint32_t)(lr * 128 + lch * 16);

    // request half tile `fill` into ring slot fill_slot (one cp.async group per half tile, empty
    // past the range or for a strip beyond N); rows past K and columns past N are zero-filled
    auto request = [&]() {
        if (requested < halves) {
            const int64_t n0 = (fill.st * WE_WARPS + warp) * WE_N;
            if (n0 < N) {
                const int64_t k0 = fill.kt * WE_K + fill.half * (WE_K / 2);
                const uint16_t* src = w + (fill.e * K + k0 + lr) * N + n0 + lch * 8;
                const uint32_t dst = ring + (uint32_t)fill_slot * WE_HALF_BYTES + lane_dst;
                if (k0 + WE_K / 2 <= K && n0 + WE_N <= N) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                                     ::"r"(dst + (uint32_t)(i * 512)), "l"(src + (int64_t)(4 * i) * N) : "memory");
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        // N % 8 == 0: chunks are wholly in or out
                        const bool in = k0 + 4 * i + lr < K && n0 + lch * 8 < N;
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                                     ::"r"(dst + (uint32_t)(i * 512)), "l"(in ? src + (int64_t)(4 * i) * N : w),
                                     "r"(in ? 16 : 0)
                                     : "memory");
                    }
                }
            }
            fill.next(tiles_k, strips);
        }
        ++requested;
        if (++fill_slot == WE_STAGES) fill_slot = 0;
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int i = 0; i < WE_STAGES - 1; ++i) request();

    const int64_t nkb = K >> 4, half_k = K >> 1;
    // whole tiles of K: one 32-byte code store per column (when the rows start on 32 bytes) and
    // one 4-byte scale store
    const bool whole_k = (K & 63) == 0;
    const bool sector_rows = whole_k && ((reinterpret_cast<uintptr_t>(qT) & 31u) == 0);
    int64_t cur_e = -1;
    int mode = ENC_EXACT;
    Nvfp4Scope sc = make_nvfp4_scope(0.0f);

    for (int64_t u = u_begin; u < u_end; ++u) {
        const int64_t e = cur.e, kt = cur.kt;
        const int64_t n0 = (cur.st * WE_WARPS + warp) * WE_N;
        const bool live = n0 < N;                              // uniform over the warp
        if (live && e != cur_e) {
            __syncwarp();                                      // the previous expert's table reads are done
            cur_e = e;
            const uint32_t sb = amax_bits[e];              // amax bits, or the flagged scale when weighted
            const float s = weighted ? __uint_as_float(sb & 0x7FFFFFFFu) : nvfp4_coarse_scale(__uint_as_float(sb));
            sc = make_nvfp4_scope(s);
            const bool all = __all_sync(0xffffffffu, nvfp4_table_build_warp(T, s, lane));
            __syncwarp();
            mode = sc.exact ? ENC_EXACT : (all ? ENC_PRODUCT : ENC_TABLE);
        }
        uint32_t code[2][8], sfw[2] = {0u, 0u};                // [column][word] / [column] scale word
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            // refill the slot read last (every lane is done with it), then wait for this half tile
            __syncwarp();
            request();
            asm volatile("cp.async.wait_group %0;" ::"n"(WE_STAGES - 1) : "memory");
            __syncwarp();
            const uint32_t slot = ring + (uint32_t)read_slot * WE_HALF_BYTES + (uint32_t)(lane * 4);
            if (++read_slot == WE_STAGES) read_slot = 0;
            cur.next(tiles_k, strips);
            if (!live) continue;
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int b = 2 * hh + bb;
                uint32_t rb[16];
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(rb[r]) : "r"(slot + (uint32_t)((16 * bb + r) * 128)));
                uint32_t m = 0;
#pragma unroll
                for (int r = 0; r < 16; ++r) m = absmax2_bf16x2(m, rb[r]);
                m &= 0x7FFF7FFFu;
                const BlockCodes lo = column_block<false>(rb, m & 0xFFFFu, mode, sc, T, I);
                const BlockCodes hi = column_block<true>(rb, m >> 16, mode, sc, T, I);
                code[0][2 * b] = lo.c0;
                code[0][2 * b + 1] = lo.c1;
                code[1][2 * b] = hi.c0;
                code[1][2 * b + 1] = hi.c1;
                sfw[0] |= lo.sfc << (8 * b);                   // blocks past K (zero rows) have scale 0
                sfw[1] |= hi.sfc << (8 * b);
            }
        }
        const int64_t n = n0 + 2 * lane;
        if (live && n < N) {
            const int64_t kb0 = kt * (WE_K / 16);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int64_t row = e * N + n + j;
                uint8_t* qd = qT + row * half_k + kb0 * 8;
                if (sector_rows) {
                    st_sector(qd, make_uint4(code[j][0], code[j][1], code[j][2], code[j][3]),
                              make_uint4(code[j][4], code[j][5], code[j][6], code[j][7]));
                } else {
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        if (kb0 + b < nkb)
                            *reinterpret_cast<uint2*>(qd + 8 * b) = make_uint2(code[j][2 * b], code[j][2 * b + 1]);
                }
                if (mma_layout) {
                    // kb0 is a multiple of 4: the word is one whole 4-column group, padding included
                    *reinterpret_cast<uint32_t*>(sfT + mma_sf_offset(row, kb0, nkb)) = sfw[j];
                } else if (whole_k) {
                    *reinterpret_cast<uint32_t*>(sfT + row * nkb + kb0) = sfw[j];
                } else {
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        if (kb0 + b < nkb) sfT[row * nkb + kb0 + b] = (uint8_t)(sfw[j] >> (8 * b));
                }
            }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// s_w <- RN(amax / 2688) from the amax bits, or (weighted) the check kernel's scale without its flag
__global__ void nvfp4_weight_finalize_kernel(float* s_w, int64_t E, int weighted) {
    griddep_begin();
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t* bits = reinterpret_cast<uint32_t*>(s_w);
    if (e < E) {
        if (weighted) bits[e] &= 0x7FFFFFFFu;
        else s_w[e] = nvfp4_coarse_scale(__uint_as_float(bits[e]));
    }
}

// zero the padding rows of an MMA-layout scale buffer beyond `rows` (rows not multiple of 128)
__global__ void zero_bytes_kernel(uint8_t* p, int64_t n) {
    griddep_begin();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) p[i] = 0;
}

cudaError_t launch_nvfp4_quantize_weights(const uint16_t* w, int64_t E, int64_t K, int64_t N,
                                          uint8_t* qT, uint8_t* sfT, float* s_w, int mma_layout,
                                          cudaStream_t stream) {
    int launched = 0;
    cudaError_t err;
    // s_w accumulates the amax bits per expert: clear it first
    if ((err = launch_pdl(zero_bytes_kernel, dim3((unsigned)((4 * E + 255) / 256)), dim3(256), 0, stream,
                          reinterpret_cast<uint8_t*>(s_w), 4 * E)) != cudaSuccess)
        return err;
    ++launched;
    const int64_t per_expert = K * N;
    // enough CTAs in total to fill the GPU a few times over, at least one per expert
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 148;
    int64_t blocks = ((int64_t)sms * 8 + E - 1) / E;
    const int64_t max_blocks = (per_expert / 8 + 255) / 256;
    if (blocks > max_blocks) blocks = max_blocks;
    if (blocks < 1) blocks = 1;
    if ((err = launch_pdl(nvfp4_weight_amax_kernel, dim3((unsigned)blocks, (unsigned)E), dim3(256), 0, stream, w,
                          per_expert, reinterpret_cast<uint32_t*>(s_w))) != cudaSuccess)
        return err;
    ++launched;
    // more than one expert: coarse scales and product-path flags for the weighted split
    const int weighted = E > 1 ? 1 : 0;
    if (weighted) {
        if ((err = launch_pdl(nvfp4_weight_check_kernel, dim3((unsigned)((E + WC_WARPS - 1) / WC_WARPS)),
                              dim3(WC_WARPS * 32), 0, stream, reinterpret_cast<uint32_t*>(s_w), E)) != cudaSuccess)
            return err;
        ++launched;
    }
    if (mma_layout) {
        // rows of the stacked [E*N, K/16] scale matrix are padded to 128; the encode kernel writes
        // every real row's tile bytes (column padding included), so only trailing pad rows remain:
        // zero the last row tile before the encode kernel fills its real rows
        const int64_t rows = E * N, kb = K >> 4;
        const int64_t padded_rows = (rows + 127) & ~int64_t(127);
        if (padded_rows > rows) {
            const int64_t start = mma_sf_offset(padded_rows - 128, 0, kb);
            const int64_t bytes = ((kb + 3) >> 2) * 512;
            if ((err = launch_pdl(zero_bytes_kernel, dim3((unsigned)((bytes + 255) / 256)), dim3(256), 0, stream,
                                  sfT + start, bytes)) != cudaSuccess)
                return err;
            ++launched;
        }
    }
    // one resident wave of encode CTAs over every super-tile of every expert
    static int enc_per_sm = 0;
    static cudaError_t enc_attr = cudaSuccess;
    static std::once_flag enc_once;
    std::call_once(enc_once, [] {
        enc_attr = cudaFuncSetAttribute(nvfp4_weight_encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        WE_SMEM_BYTES);
        if (enc_attr == cudaSuccess &&
            (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&enc_per_sm, nvfp4_weight_encode_kernel, WE_THREADS,
                                                           WE_SMEM_BYTES) != cudaSuccess || enc_per_sm < 1))
            enc_per_sm = 1;
    });
    if (enc_attr != cudaSuccess) return enc_attr;
    const int64_t tiles_k = (K + WE_K - 1) / WE_K, strips = (N + WE_WARPS * WE_N - 1) / (WE_WARPS * WE_N);
    const int64_t total = E * tiles_k * strips;
    const int64_t enc_grid = std::min<int64_t>(total, (int64_t)sms * enc_per_sm);
    if ((err = launch_pdl(nvfp4_weight_encode_kernel, dim3((unsigned)enc_grid), dim3(WE_THREADS), WE_SMEM_BYTES,
                          stream, w, K, N, tiles_k, strips, total, qT, sfT, reinterpret_cast<const uint32_t*>(s_w),
                          mma_layout, weighted)) != cudaSuccess)
        return err;
    ++launched;
    if ((err = launch_pdl(nvfp4_weight_finalize_kernel, dim3((unsigned)((E + 255) / 256)), dim3(256), 0, stream,
                          s_w, E, weighted)) != cudaSuccess)
        return err;
    count_launches(launched + 1);
    return cudaSuccess;
}

}  // namespace nvq
