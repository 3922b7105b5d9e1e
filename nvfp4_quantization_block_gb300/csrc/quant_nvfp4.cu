// NVFP4 quantizers: per-token activations and per-expert-matrix weights.
//
// Definition [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本":
// section "为什么需要 Blackwell 原生方案？" (E2M1 values, one E4M3 scale per 16 values rounded to
// nearest, a coarse FP32 scale on top); section "逐 Token 激活值缩放" (one FP32 scale per token computed
// online, fused into the quantization call that also emits the packed FP4 values and the block
// scales; gate/up weights share one FP32 scale); section "比特精确量化器合约" (bit-exact contract,
// no fast math)]. Coarse scale s = RN(amax / 2688); block scale = E4M3 RNE of amax_b / (6 s);
// code = E2M1 RNE (saturating) of x / (E4M3(sf) s). Exactness: see nvq_device.cuh.
//
// Per-token design: one warp per token row, one 16-element block per lane per step (see the
// kernel). Weights: one warp per 64 x 64 tile, two columns and four 16-row blocks per lane. A scope
// whose table passes the product-path check (nvq_device.cuh) encodes its elements by one fp32
// multiply and the hardware E2M1 conversion; any other scope compares each element with its block's
// exact boundaries.
#include <algorithm>
#include <mutex>

#include "nvq_device.cuh"
#include "nvq_internal.h"

namespace nvq {

constexpr int TOK_THREADS = 128;          // 4 rows per CTA
constexpr int TOK_NREG = 4;               // 4 x 32 blocks of 16 = 2048 elements held in registers per row

template <bool V8>
__device__ __forceinline__ void load_block(const uint16_t* p, uint4& a, uint4& b) {
    if (V8) {
        ld_v8(p, a, b);
    } else {
        a = ld_stream_v4(p);
        b = ld_stream_v4(p + 8);
    }
}

// SwiGLU of a fused gate||up activation, rounded to bf16 (the down projection's input). The pages'
// SwiGLU experts run gate and up as one GEMM [Miles-zh, "逐 Token 激活值缩放"]; the activation is
// silu(g) u with silu(g) = g / (1 + exp(-g)) (Shazeer 2020), computed in float32 with one rounding
// per operation (no contraction: __f*_rn), so that it is reproducible bit for bit. exp is our own:
// Cody and Waite's two-constant range reduction (clamped to [-87, 88] so 2^n stays normal) and a
// degree-6 Taylor polynomial in Horner order.
__device__ __forceinline__ float swiglu_exp(float x) {
    x = fminf(fmaxf(x, -87.0f), 88.0f);
    const float n = __fsub_rn(__fadd_rn(__fmul_rn(x, (float)1.4426950408889634), 12582912.0f), 12582912.0f);
    const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, 0.693145751953125f)),
                              __fmul_rn(n, (float)(0.6931471805599453 - 0.693145751953125)));
    float p = (float)(1.0 / 720.0);
    p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 120.0));
    p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 24.0));
    p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 6.0));
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    return __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
}

__device__ __forceinline__ float swiglu(float g, float u) {
    const float d = __fadd_rn(1.0f, swiglu_exp(-g));
    return __fmul_rn(__fdiv_rn(g, d), u);
}

// bf16x2 words of SwiGLU(gate, up) for two bf16x2 words
__device__ __forceinline__ uint32_t swiglu2(uint32_t g, uint32_t u) {
    return cvt_bf16x2(swiglu(bf16_lo(g), bf16_lo(u)), swiglu(bf16_hi(g), bf16_hi(u)));
}

// One 16-element block of the row: loaded as is, or (SWIGLU) formed from the gate block at p and
// the up block at p + up.
template <bool V8, bool SWIGLU>
__device__ __forceinline__ void row_block(const uint16_t* p, int64_t up, uint4& a, uint4& b) {
    load_block<V8>(p, a, b);
    if (SWIGLU) {
        uint4 ua, ub;
        load_block<V8>(p + up, ua, ub);
        a = make_uint4(swiglu2(a.x, ua.x), swiglu2(a.y, ua.y), swiglu2(a.z, ua.z), swiglu2(a.w, ua.w));
        b = make_uint4(swiglu2(b.x, ub.x), swiglu2(b.y, ub.y), swiglu2(b.z, ub.z), swiglu2(b.w, ub.w));
    }
}

// How a scope's blocks are encoded: by the product path (its table passed the check), by the
// table's boundary comparisons, or by exact fp64 decisions (a scope with a tiny or zero coarse scale).
enum : int { ENC_TABLE = 0, ENC_EXACT = 1, ENC_PRODUCT = 2 };

// Scale code and the 16 codes of one block (two uint4 of 8 bf16, magnitude maximum mb as bf16
// bits); branch-free in the table and product modes.
template <int MODE>
__device__ __forceinline__ uint32_t encode_block(const uint4& a, const uint4& b, uint32_t mb, const Nvfp4Scope& sc,
                                                 const Nvfp4Table& T, const Nvfp4CodeInfo& I, uint32_t& c0,
                                                 uint32_t& c1) {
    if (MODE == ENC_EXACT) {
        const uint32_t sfc = nvfp4_block_scale(__uint_as_float(mb << 16), sc);
        c0 = nvfp4_encode8_exact(a, sfc, sc);
        c1 = nvfp4_encode8_exact(b, sfc, sc);
        return sfc;
    }
    const uint32_t sfc = nvfp4_block_scale_t(mb, sc, T);
    if (MODE == ENC_PRODUCT) {
        const float g = nvfp4_block_g(sfc, T, I);
        c0 = nvfp4_codes8_mul(a, g);
        c1 = nvfp4_codes8_mul(b, g);
    } else {
        const E2M1Bounds bd = nvfp4_block_bounds_t(sfc, T, I);
        c0 = nvfp4_codes8(a, bd);
        c1 = nvfp4_codes8(b, bd);
    }
    return sfc;
}

// Where one token row's outputs go: its packed codes and its scale bytes (canonical row, or the
// row's place in the MMA tile layout, to which a 4-block group adds (kb / 4) * 512).
struct TokenRowOut {
    uint8_t* q;          // row of packed codes
    uint8_t* sf;         // canonical: row of scale bytes; MMA: row's base inside its tile column
    int64_t nkb;
    int mma_layout;
};

// Stores of one 16-element block kb of the row (codes c0, c1, scale code sfc), one block per lane:
// the four lanes l..l+3 (l a multiple of 4 within the row's lanes) hold four consecutive blocks and
// share one scale word. Called by all 32 lanes of the warp together (shuffles).
__device__ __forceinline__ void token_store(uint32_t sfc, uint32_t c0, uint32_t c1, int64_t kb, int l, bool real,
                                            const TokenRowOut& o) {
    if (real && kb < o.nkb) *reinterpret_cast<uint2*>(o.q + kb * 8) = make_uint2(c0, c1);
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, sfc, 1);
    const uint32_t s2 = __shfl_down_sync(0xffffffffu, sfc, 2);
    const uint32_t s3 = __shfl_down_sync(0xffffffffu, sfc, 3);
    if ((l & 3) == 0 && kb < o.nkb && o.sf != nullptr) {
        const uint32_t word = sfc | (s1 << 8) | (s2 << 16) | (s3 << 24);
        if (o.mma_layout) {
            *reinterpret_cast<uint32_t*>(o.sf + ((kb >> 2) << 9)) = word;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (kb + j < o.nkb) o.sf[kb + j] = (uint8_t)(word >> (8 * j));
        }
    }
}

// Encode and store one block; the encoding mode is the same for every lane.
template <int MODE>
__device__ __forceinline__ void token_block(const uint4& a, const uint4& b, uint32_t mb, int64_t kb, int l, bool real,
                                            const Nvfp4Scope& sc, const Nvfp4Table& T, const Nvfp4CodeInfo& I,
                                            const TokenRowOut& o) {
    uint32_t c0, c1;
    const uint32_t sfc = encode_block<MODE>(a, b, mb, sc, T, I, c0, c1);
    token_store(sfc, c0, c1, kb, l, real, o);
}

// Encode and store one block when the two rows of a warp may take different paths: the encoding
// branches per row, the stores (shuffles) run with the whole warp.
__device__ __forceinline__ void token_block_mixed(const uint4& a, const uint4& b, uint32_t mb, int64_t kb, int l,
                                                  bool real, int mode, const Nvfp4Scope& sc, const Nvfp4Table& T,
                                                  const Nvfp4CodeInfo& I, const TokenRowOut& o) {
    uint32_t c0, c1, sfc;
    if (mode == ENC_PRODUCT) sfc = encode_block<ENC_PRODUCT>(a, b, mb, sc, T, I, c0, c1);
    else if (mode == ENC_TABLE) sfc = encode_block<ENC_TABLE>(a, b, mb, sc, T, I, c0, c1);
    else sfc = encode_block<ENC_EXACT>(a, b, mb, sc, T, I, c0, c1);
    __syncwarp();
    token_store(sfc, c0, c1, kb, l, real, o);
}

// The scope table of a row built by its LPR lanes (32: nvfp4_table_build_warp, with the product
// path's check; 16: each lane takes the class boundaries of thresholds j and j + 2 (and their
// j + 4 partners) of class l & 7, and the block-scale boundary of code l). Called by all 32 lanes of
// the warp together; returns whether the lane's class has a product-path multiplier. Rows of 16
// lanes never take the product path: with at most four blocks per lane, the check (five candidate
// multipliers at up to four boundaries per lane) costs more than it saves (measured: the MoE down
// projection's 768-wide rows and the SwiGLU rows ran 7% and 17% slower with it).
template <int LPR>
__device__ __forceinline__ bool nvfp4_table_build_row(Nvfp4Table& T, float s, int l) {
    if (LPR == 32) return nvfp4_table_build_warp(T, s, l);
    const uint32_t f = (uint32_t)l & 7u;
    const float v = (float)(8u + f) * 0x1p-9f;                     // value of E4M3 code 8 + f
#pragma unroll
    for (uint32_t t = 0; t < 2; ++t) {
        const uint32_t j = ((uint32_t)l >> 3) + 2u * t;            // 0..3
        uint32_t b = bf16_boundary((float)(2u * j + 1u) * 0.25f * v, s, (j & 1u) != 0u);
        T.bp[f][j] = b | (b << 16);
        if (j < 3u) T.bp[f][8u + j] = (b | (b << 16)) ^ 0x80008000u;
        const uint32_t j2 = j + 4u;
        if (j2 < 7u) {
            const float m = (j2 == 6u) ? 5.0f : (float)j2 - 1.5f;
            b = bf16_boundary(m * v, s, (j2 & 1u) != 0u);
            T.bp[f][j2] = b | (b << 16);
        }
    }
    T.bs[l] = bf16_boundary((float)(3 * (2 * l + 1)) * 0x1p-9f, s, (l & 1) != 0);
    if (l < 12) T.bp[8][l] = l < 7 ? 0x7F007F00u : (l >= 8 && l < 11 ? 0xFF00FF00u : 0u);
    return false;
}

// LPR lanes per token row (32: one row per warp; 16: two rows per warp, for rows of at most 64
// blocks, so that rows of 48 blocks keep every lane busy), one 16-element block per lane per step:
// the row is loaded once with 32-byte coalesced loads (held in registers up to TOK_NREG steps),
// reduced to its amax with shuffles among the row's lanes, and encoded from registers, so each
// input byte is read from HBM once.
template <bool V8, bool SWIGLU, int LPR>
__global__ void __launch_bounds__(TOK_THREADS)
nvfp4_token_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ldx,
                   uint8_t* __restrict__ q, uint8_t* __restrict__ sf, float* __restrict__ s_tok,
                   int mma_layout, int64_t rows_cover) {
    griddep_begin();
    constexpr int RPW = 32 / LPR;                              // rows per warp
    __shared__ Nvfp4Table tables[(TOK_THREADS / 32) * RPW];   // one per row
    __shared__ Nvfp4CodeInfo info;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane / LPR, l = lane % LPR;               // row of the warp, lane within the row
    for (uint32_t c = threadIdx.x; c < 128u; c += TOK_THREADS) nvfp4_code_info_build(info, c);
    __syncthreads();
    const int64_t row0 = ((int64_t)blockIdx.x * (TOK_THREADS / 32) + warp) * RPW;
    if (row0 >= rows_cover) return;                            // uniform over the warp
    const int64_t row = row0 + half;
    const bool covered = row < rows_cover;                     // the second row of a warp may not be
    Nvfp4Table& T = tables[warp * RPW + half];
    const bool real = row < R;
    const int64_t nkb = C >> 4;                                // 16-element blocks
    const int iters = (int)((nkb + LPR - 1) / LPR);
    const uint16_t* xr = x + (real ? row : 0) * ldx;

    // pass 1: load (into registers where possible) and reduce the row's amax
    uint4 va[TOK_NREG], vb[TOK_NREG];
    uint32_t mbk[TOK_NREG];                                    // block maxima of the register-resident blocks
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < TOK_NREG; ++i) {
        va[i] = vb[i] = make_uint4(0u, 0u, 0u, 0u);
        const int64_t kb = (int64_t)i * LPR + l;
        if (real && i < iters && kb < nkb) row_block<V8, SWIGLU>(xr + kb * 16, C, va[i], vb[i]);
        mbk[i] = max(absmax_bits_8(va[i]), absmax_bits_8(vb[i]));
        m = max(m, mbk[i]);
    }
    for (int i = TOK_NREG; i < iters; ++i) {
        const int64_t kb = (int64_t)i * LPR + l;
        if (real && kb < nkb) {
            uint4 a, b;
            row_block<V8, SWIGLU>(xr + kb * 16, C, a, b);
            m = max(m, max(absmax_bits_8(a), absmax_bits_8(b)));
        }
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = nvfp4_coarse_scale(__uint_as_float(m << 16));
    const Nvfp4Scope sc = make_nvfp4_scope(s);
    if (real && l == 0) s_tok[row] = s;
    // every row builds a table (all lanes take part in its shuffles); an exact-path row ignores it
    const bool ok = nvfp4_table_build_row<LPR>(T, s, l);
    __syncwarp();
    const uint32_t bad = __ballot_sync(0xffffffffu, !ok);
    const uint32_t row_bad = LPR == 32 ? bad : (bad >> (half * LPR)) & ((1u << LPR) - 1u);
    const int mode = sc.exact ? ENC_EXACT : ((LPR == 32 && row_bad == 0u) ? ENC_PRODUCT : ENC_TABLE);

    // pass 2: per 1x16 block scale and codes (register-resident blocks first, then any reloads)
    TokenRowOut o;
    o.q = q + (real ? row : 0) * (C >> 1);
    o.nkb = nkb;
    o.mma_layout = mma_layout;
    o.sf = !covered ? nullptr : (mma_layout ? sf + mma_sf_offset(row, 0, nkb) : sf + row * nkb);
    const uint32_t same = __match_any_sync(0xffffffffu, mode);
    if (same == 0xffffffffu && mode == ENC_PRODUCT) {
#pragma unroll
        for (int i = 0; i < TOK_NREG; ++i)
            if (i < iters)
                token_block<ENC_PRODUCT>(va[i], vb[i], mbk[i], (int64_t)i * LPR + l, l, real, sc, T, info, o);
    } else if (same == 0xffffffffu && mode == ENC_TABLE) {
#pragma unroll
        for (int i = 0; i < TOK_NREG; ++i)
            if (i < iters) token_block<ENC_TABLE>(va[i], vb[i], mbk[i], (int64_t)i * LPR + l, l, real, sc, T, info, o);
    } else if (same == 0xffffffffu) {
#pragma unroll
        for (int i = 0; i < TOK_NREG; ++i)
            if (i < iters) token_block<ENC_EXACT>(va[i], vb[i], mbk[i], (int64_t)i * LPR + l, l, real, sc, T, info, o);
    } else {
        // the two rows of the warp take different modes
#pragma unroll
        for (int i = 0; i < TOK_NREG; ++i)
            if (i < iters)
                token_block_mixed(va[i], vb[i], mbk[i], (int64_t)i * LPR + l, l, real, mode, sc, T, info, o);
    }
    for (int i = TOK_NREG; i < iters; ++i) {
        const int64_t kb = (int64_t)i * LPR + l;
        uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
        if (real && kb < nkb) row_block<V8, SWIGLU>(xr + kb * 16, C, a, b);
        const uint32_t mb = max(absmax_bits_8(a), absmax_bits_8(b));
        token_block_mixed(a, b, mb, kb, l, real, mode, sc, T, info, o);
    }
}

template <bool SWIGLU>
static cudaError_t launch_token(const uint16_t* x, int64_t R, int64_t C, int64_t ldx, uint8_t* q, uint8_t* sf,
                                float* s_tok, int mma_layout, cudaStream_t stream) {
    const int64_t cover = mma_layout ? ((R + 127) & ~int64_t(127)) : R;
    // two rows per warp when a row has at most 4 x 16 blocks: all 16 lanes of a row stay busy
    const bool pair = (C >> 4) <= 4 * 16;
    const int rows_per_cta = (TOK_THREADS / 32) * (pair ? 2 : 1);
    const int64_t grid = (cover + rows_per_cta - 1) / rows_per_cta;
    const bool v8 = ((reinterpret_cast<uintptr_t>(x) & 31u) == 0) && (ldx % 16 == 0) && (!SWIGLU || C % 16 == 0);
    cudaError_t lerr;
#define NVQ_TOK(V, L)                                                                                             \
    lerr = launch_pdl(nvfp4_token_kernel<V, SWIGLU, L>, dim3((unsigned)grid), dim3(TOK_THREADS), 0, stream, x, R, C, \
                      ldx, q, sf, s_tok, mma_layout, cover)
    if (v8) {
        if (pair) NVQ_TOK(true, 16);
        else NVQ_TOK(true, 32);
    } else {
        if (pair) NVQ_TOK(false, 16);
        else NVQ_TOK(false, 32);
    }
#undef NVQ_TOK
    const cudaError_t err = lerr != cudaSuccess ? lerr : cudaGetLastError();
    if (err == cudaSuccess) count_launches(1);
    return err;
}

cudaError_t launch_nvfp4_quantize_per_token(const uint16_t* x, int64_t R, int64_t C, int64_t ldx,
                                            uint8_t* q, uint8_t* sf, float* s_tok, int mma_layout,
                                            cudaStream_t stream) {
    return launch_token<false>(x, R, C, ldx, q, sf, s_tok, mma_layout, stream);
}

cudaError_t launch_nvfp4_swiglu_quantize(const uint16_t* gate_up, int64_t R, int64_t I, int64_t ld, uint8_t* q,
                                         uint8_t* sf, float* s_tok, int mma_layout, cudaStream_t stream) {
    return launch_token<true>(gate_up, R, I, ld, q, sf, s_tok, mma_layout, stream);
}

// ------------------------------------------------------------------------------------------------
// Weights: W [E, K, N] -> qT [E, N, K/2], sfT [E, N, K/16], s_w [E]; coarse scope = expert matrix.
// Three kernels: amax per expert (atomic max on the fp32 bits, kept in s_w), encode, finalize
// (s_w <- RN(amax / 2688)).
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

// Encode: every warp works on its own, over a contiguous range of the (expert, n tile, k tile)
// sequence of 64 k x 64 n tiles, so the load is even for any expert count and a warp rebuilds its
// scope table only when its range enters the next expert. Lane l owns columns n0 + 2l and
// n0 + 2l + 1 and the tile's four 16-row blocks: it loads the tile's 64 rows of its two columns (one
// 4-byte load per row, 128 contiguous bytes per row across the warp; each 32-row half of the next
// tile is requested as soon as the same half of this one is encoded), so each column's block is
// the low or high halves of one word per row and no transpose is needed. Its outputs are whole per column: the four blocks' 32 code bytes (one L2 sector, one
// store) and their 4 scale bytes (one 4-column group). K is the fastest tile index, so a row's
// scale bytes are written by consecutive tiles of one warp. (Half-sector code stores, 16 bytes per
// tile, made L2 write partial sectors back: 3.4x the output bytes in DRAM writes.)
constexpr int WE_K = 64, WE_N = 64, WE_THREADS = 128, WE_WARPS = WE_THREADS / 32;

// Pairs (x[2i], x[2i + 1]) of one column of 8 rows, as the bf16x2 words of the table and exact
// paths: the column is the low (HI false) or high half of each row's word.
template <bool HI>
__device__ __forceinline__ uint4 column_pairs(const uint32_t* r) {
    constexpr uint32_t sel = HI ? 0x7632u : 0x5410u;
    return make_uint4(__byte_perm(r[0], r[1], sel), __byte_perm(r[2], r[3], sel), __byte_perm(r[4], r[5], sel),
                      __byte_perm(r[6], r[7], sel));
}

// fp32 values of 8 rows of one column, times g, to 8 E2M1 codes (product path)
template <bool HI>
__device__ __forceinline__ uint32_t column_codes_mul(const uint32_t* r, float g) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(HI ? bf16_hi(r[i]) : bf16_lo(r[i]), g);
    return cvt_e2m1x8(x[0], x[1], x[2], x[3], x[4], x[5], x[6], x[7]);
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

__global__ void __launch_bounds__(WE_THREADS, 3)
nvfp4_weight_encode_kernel(const uint16_t* __restrict__ w, int64_t K, int64_t N, int64_t tiles_k, int64_t tiles_n,
                           int64_t total, uint8_t* __restrict__ qT, uint8_t* __restrict__ sfT,
                           const uint32_t* __restrict__ amax_bits, int mma_layout) {
    griddep_begin();
    __shared__ Nvfp4Table tables[WE_WARPS];                    // each warp's current expert
    __shared__ Nvfp4CodeInfo I;
    for (uint32_t c = threadIdx.x; c < 128u; c += WE_THREADS) nvfp4_code_info_build(I, c);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Nvfp4Table& T = tables[warp];
    const int64_t gw = (int64_t)blockIdx.x * WE_WARPS + warp, nw = (int64_t)gridDim.x * WE_WARPS;
    const int64_t t_begin = total * gw / nw, t_end = total * (gw + 1) / nw;
    if (t_begin >= t_end) return;                              // uniform over the warp
    const int64_t per_e = tiles_k * tiles_n;
    int64_t e = t_begin / per_e;
    int64_t nt = (t_begin - e * per_e) / tiles_k;
    int64_t kt = t_begin - e * per_e - nt * tiles_k;
    const int64_t nkb = K >> 4, half_k = K >> 1;
    // whole tiles of K: one 32-byte code store per column (when the rows start on 32 bytes) and
    // one 4-byte scale store
    const bool whole_k = (K & 63) == 0;
    const bool sector_rows = whole_k && ((reinterpret_cast<uintptr_t>(qT) & 31u) == 0);
    int64_t cur_e = -1;
    int mode = ENC_EXACT;
    Nvfp4Scope sc = make_nvfp4_scope(0.0f);

    // rows [0, 32) and [32, 64) of the tile's two columns (low / high half of each word); the next
    // tile's half is loaded as soon as this tile's half is encoded, so loads stay in flight while
    // the warp computes
    uint32_t xa[WE_K / 2], xb[WE_K / 2];
    auto load_half = [&](uint32_t (&x)[WE_K / 2], int64_t te, int64_t tn, int64_t tk, int h) {
        const int64_t k0 = tk * WE_K + h * (WE_K / 2), n0 = tn * WE_N + 2 * lane;
        const bool ok = n0 < N;                                // N even: both columns in or out together
        const int64_t rows = K - k0;
        const uint16_t* src = w + (te * K + k0) * N + n0;
#pragma unroll
        for (int r = 0; r < WE_K / 2; ++r) x[r] = ld_stream_u32_if(src + r * N, ok && r < rows);
    };
    load_half(xa, e, nt, kt, 0);
    load_half(xb, e, nt, kt, 1);

    for (int64_t t = t_begin; t < t_end; ++t) {
        if (e != cur_e) {
            __syncwarp();                                      // the previous expert's table reads are done
            cur_e = e;
            const float s = nvfp4_coarse_scale(__uint_as_float(amax_bits[e]));
            sc = make_nvfp4_scope(s);
            const bool all = __all_sync(0xffffffffu, nvfp4_table_build_warp(T, s, lane));
            __syncwarp();
            mode = sc.exact ? ENC_EXACT : (all ? ENC_PRODUCT : ENC_TABLE);
        }
        // the next tile (k fastest)
        int64_t e1 = e, nt1 = nt, kt1 = kt + 1;
        if (kt1 == tiles_k) {
            kt1 = 0;
            if (++nt1 == tiles_n) {
                nt1 = 0;
                ++e1;
            }
        }
        const bool more = t + 1 < t_end;
        uint32_t code[2][8], sfw[2] = {0u, 0u};                // [column][word] / [column] scale word
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t* rb = (b < 2 ? xa : xb) + 16 * (b & 1);
            uint32_t m = 0;
#pragma unroll
            for (int r = 0; r < 16; ++r) m = __vmaxu2(m, rb[r] & 0x7FFF7FFFu);
            const BlockCodes lo = column_block<false>(rb, m & 0xFFFFu, mode, sc, T, I);
            const BlockCodes hi = column_block<true>(rb, m >> 16, mode, sc, T, I);
            code[0][2 * b] = lo.c0;
            code[0][2 * b + 1] = lo.c1;
            code[1][2 * b] = hi.c0;
            code[1][2 * b + 1] = hi.c1;
            sfw[0] |= lo.sfc << (8 * b);                       // blocks past K (zero rows) have scale 0
            sfw[1] |= hi.sfc << (8 * b);
            if (b == 1 && more) load_half(xa, e1, nt1, kt1, 0);
            if (b == 3 && more) load_half(xb, e1, nt1, kt1, 1);
        }
        const int64_t n = nt * WE_N + 2 * lane;
        if (n < N) {
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
        e = e1;
        nt = nt1;
        kt = kt1;
    }
}

__global__ void nvfp4_weight_finalize_kernel(float* s_w, int64_t E) {
    griddep_begin();
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e < E) s_w[e] = nvfp4_coarse_scale(__uint_as_float(reinterpret_cast<uint32_t*>(s_w)[e]));
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
    // one resident wave of encode warps over every tile of every expert
    static int enc_per_sm = 0;
    static std::once_flag enc_once;
    std::call_once(enc_once, [] {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&enc_per_sm, nvfp4_weight_encode_kernel, WE_THREADS, 0) !=
            cudaSuccess || enc_per_sm < 1)
            enc_per_sm = 1;
    });
    const int64_t tiles_k = (K + WE_K - 1) / WE_K, tiles_n = (N + WE_N - 1) / WE_N;
    const int64_t total = E * tiles_k * tiles_n;
    const int64_t enc_grid = std::min<int64_t>((total + WE_WARPS - 1) / WE_WARPS, (int64_t)sms * enc_per_sm);
    if ((err = launch_pdl(nvfp4_weight_encode_kernel, dim3((unsigned)enc_grid), dim3(WE_THREADS), 0, stream, w, K, N,
                          tiles_k, tiles_n, total, qT, sfT, reinterpret_cast<const uint32_t*>(s_w), mma_layout)) !=
        cudaSuccess)
        return err;
    ++launched;
    if ((err = launch_pdl(nvfp4_weight_finalize_kernel, dim3((unsigned)((E + 255) / 256)), dim3(256), 0, stream,
                          s_w, E)) != cudaSuccess)
        return err;
    count_launches(launched + 1);
    return cudaSuccess;
}

}  // namespace nvq
