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
// kernel). Weights: one thread per (column, 16-row block) after a shared-memory transpose. A scope
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
#define NVQ_TOK(V, L) \
    nvfp4_token_kernel<V, SWIGLU, L><<<(unsigned)grid, TOK_THREADS, 0, stream>>>(x, R, C, ldx, q, sf, s_tok, mma_layout, cover)
    if (v8) {
        if (pair) NVQ_TOK(true, 16);
        else NVQ_TOK(true, 32);
    } else {
        if (pair) NVQ_TOK(false, 16);
        else NVQ_TOK(false, 32);
    }
#undef NVQ_TOK
    const cudaError_t err = cudaGetLastError();
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
constexpr int WT_K = 64, WT_N = 64, WT_THREADS = 256;
constexpr int WT_STRIDE = 36;            // words per transposed smem row (64 k = 32 k-pair words + 4)

__global__ void __launch_bounds__(256)
nvfp4_weight_amax_kernel(const uint16_t* __restrict__ w, int64_t per_expert, uint32_t* __restrict__ amax_bits) {
    const int64_t e = blockIdx.y;
    const uint16_t* we = w + e * per_expert;
    const int64_t nvec = per_expert >> 3;
    uint32_t m = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x)
        m = max(m, absmax_bits_8(ld_stream_v4(we + i * 8)));
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

// Encode: a persistent loop over tiles of 64 k x 64 n. CTA b takes the contiguous range
// [total b / G, total (b + 1) / G) of the (expert, k tile, n tile) sequence, so the load is even
// for any expert count and a CTA rebuilds its scope table only when its range enters the next
// expert. A tile arrives as row pairs (k, k + 1): byte permutes interleave them into words
// (x[k][n], x[k+1][n]) stored transposed, [n][k pair], in shared memory, the k-pair index of row
// n XOR-ed with 4 (n / 8) so that the stores and the 128-bit loads are free of bank conflicts.
// Each thread then encodes one 16-k block of one column, read with two 128-bit loads. The next
// tile's rows are in flight while the current tile is encoded (two buffers, one barrier a tile).
__global__ void __launch_bounds__(WT_THREADS)
nvfp4_weight_encode_kernel(const uint16_t* __restrict__ w, int64_t K, int64_t N, int64_t tiles_k, int64_t tiles_n,
                           int64_t total, uint8_t* __restrict__ qT, uint8_t* __restrict__ sfT,
                           const uint32_t* __restrict__ amax_bits, int mma_layout) {
    __shared__ __align__(16) uint32_t tile[2][WT_N * WT_STRIDE];
    __shared__ Nvfp4Table T;                                   // the current expert's scope table
    __shared__ Nvfp4CodeInfo I;
    if (threadIdx.x < 128) nvfp4_code_info_build(I, threadIdx.x);

    const int64_t per_e = tiles_k * tiles_n;
    const int64_t t_begin = total * blockIdx.x / gridDim.x, t_end = total * (blockIdx.x + 1) / gridDim.x;
    const int lp = threadIdx.x >> 3, lc = threadIdx.x & 7;     // loader: k pair, 8-column chunk
    const int en = threadIdx.x >> 2, ekb = threadIdx.x & 3;    // encoder: column, 16-k block
    const int64_t nkb = K >> 4;

    // tile cursor (expert, k tile, n tile), advanced without divisions
    struct Cursor {
        int64_t e, kt, nt;
    };
    auto advance = [&](Cursor& c) {
        if (++c.nt == tiles_n) {
            c.nt = 0;
            if (++c.kt == tiles_k) {
                c.kt = 0;
                ++c.e;
            }
        }
    };
    auto load = [&](const Cursor& c, uint4& A, uint4& B) {
        const int64_t k = c.kt * WT_K + 2 * lp, n = c.nt * WT_N + 8 * lc;
        A = B = make_uint4(0u, 0u, 0u, 0u);
        if (k < K && n < N) {                                  // K even: row k + 1 exists too
            const uint16_t* src = w + (c.e * K + k) * N + n;
            A = ld_stream_v4(src);
            B = ld_stream_v4(src + N);
        }
    };

    Cursor cur;
    cur.e = t_begin / per_e;
    cur.kt = (t_begin - cur.e * per_e) / tiles_n;
    cur.nt = t_begin - cur.e * per_e - cur.kt * tiles_n;
    Cursor nxt = cur;
    uint4 A, B;
    if (t_begin < t_end) load(cur, A, B);
    int64_t cur_e = -1;
    bool new_scope = false;
    int mode = ENC_EXACT;
    Nvfp4Scope sc = make_nvfp4_scope(0.0f);
    for (int64_t t = t_begin; t < t_end; ++t) {
        uint32_t* buf = tile[(t - t_begin) & 1];
        {
            const uint32_t a[4] = {A.x, A.y, A.z, A.w}, b[4] = {B.x, B.y, B.z, B.w};
            const int col = lp ^ (4 * lc);                     // row n = 8 lc + m: n / 8 = lc
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n0 = 8 * lc + 2 * j;                 // word j holds columns n0, n0 + 1
                buf[n0 * WT_STRIDE + col] = __byte_perm(a[j], b[j], 0x5410);
                buf[(n0 + 1) * WT_STRIDE + col] = __byte_perm(a[j], b[j], 0x7632);
            }
        }
        cur = nxt;
        advance(nxt);
        if (t + 1 < t_end) load(nxt, A, B);
        const int64_t e = cur.e;
        if (e != cur_e) {                                      // uniform across the CTA
            __syncthreads();                                   // the previous expert's table is done
            cur_e = e;
            const float s = nvfp4_coarse_scale(__uint_as_float(amax_bits[e]));
            sc = make_nvfp4_scope(s);
            if (threadIdx.x < 32) {
                const bool all = __all_sync(0xffffffffu, nvfp4_table_build_warp(T, s, threadIdx.x));
                if (threadIdx.x == 0) T.product = all ? 1u : 0u;
            }
            new_scope = true;
        }
        __syncthreads();
        if (new_scope) {
            mode = sc.exact ? ENC_EXACT : (T.product ? ENC_PRODUCT : ENC_TABLE);
            new_scope = false;
        }

        const int64_t k0 = cur.kt * WT_K, n = cur.nt * WT_N + en;
        const uint32_t* rowp = buf + en * WT_STRIDE;
        const int sw = 4 * (en >> 3);
        const uint4 lo = *reinterpret_cast<const uint4*>(rowp + ((8 * ekb) ^ sw));
        const uint4 hi = *reinterpret_cast<const uint4*>(rowp + ((8 * ekb + 4) ^ sw));
        uint32_t c0, c1;
        const uint32_t mb = max(absmax_bits_8(lo), absmax_bits_8(hi));
        uint32_t sfc;
        if (mode == ENC_PRODUCT) sfc = encode_block<ENC_PRODUCT>(lo, hi, mb, sc, T, I, c0, c1);
        else if (mode == ENC_TABLE) sfc = encode_block<ENC_TABLE>(lo, hi, mb, sc, T, I, c0, c1);
        else sfc = encode_block<ENC_EXACT>(lo, hi, mb, sc, T, I, c0, c1);
        const int64_t kb0 = k0 >> 4, kb = kb0 + ekb;
        const int64_t row = e * N + n;
        if (n < N && kb < nkb) *reinterpret_cast<uint2*>(qT + row * (K >> 1) + kb * 8) = make_uint2(c0, c1);
        // scale bytes: the 4 lanes of one column hold 4 consecutive blocks
        const uint32_t s1 = __shfl_down_sync(0xffffffffu, sfc, 1);
        const uint32_t s2 = __shfl_down_sync(0xffffffffu, sfc, 2);
        const uint32_t s3 = __shfl_down_sync(0xffffffffu, sfc, 3);
        if (ekb == 0 && n < N) {
            const uint32_t word = sfc | (s1 << 8) | (s2 << 16) | (s3 << 24);
            if (mma_layout) {
                *reinterpret_cast<uint32_t*>(sfT + mma_sf_offset(row, kb0, nkb)) = word;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (kb0 + j < nkb) sfT[row * nkb + kb0 + j] = (uint8_t)(word >> (8 * j));
            }
        }
    }
}

__global__ void nvfp4_weight_finalize_kernel(float* s_w, int64_t E) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e < E) s_w[e] = nvfp4_coarse_scale(__uint_as_float(reinterpret_cast<uint32_t*>(s_w)[e]));
}

// zero the padding rows of an MMA-layout scale buffer beyond `rows` (rows not multiple of 128)
__global__ void zero_bytes_kernel(uint8_t* p, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) p[i] = 0;
}

cudaError_t launch_nvfp4_quantize_weights(const uint16_t* w, int64_t E, int64_t K, int64_t N,
                                          uint8_t* qT, uint8_t* sfT, float* s_w, int mma_layout,
                                          cudaStream_t stream) {
    int launched = 0;
    cudaError_t err;
    // s_w accumulates the amax bits per expert: clear it first
    zero_bytes_kernel<<<(unsigned)((4 * E + 255) / 256), 256, 0, stream>>>(reinterpret_cast<uint8_t*>(s_w), 4 * E);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
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
    nvfp4_weight_amax_kernel<<<dim3((unsigned)blocks, (unsigned)E), 256, 0, stream>>>(
        w, per_expert, reinterpret_cast<uint32_t*>(s_w));
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
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
            zero_bytes_kernel<<<(unsigned)((bytes + 255) / 256), 256, 0, stream>>>(sfT + start, bytes);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
            ++launched;
        }
    }
    // one resident wave of encode CTAs over every tile of every expert
    static int enc_per_sm = 0;
    static std::once_flag enc_once;
    std::call_once(enc_once, [] {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&enc_per_sm, nvfp4_weight_encode_kernel, WT_THREADS, 0) !=
            cudaSuccess || enc_per_sm < 1)
            enc_per_sm = 1;
    });
    const int64_t tiles_k = (K + WT_K - 1) / WT_K, tiles_n = (N + WT_N - 1) / WT_N;
    const int64_t total = E * tiles_k * tiles_n;
    const int64_t enc_grid = std::min<int64_t>(total, (int64_t)sms * enc_per_sm);
    nvfp4_weight_encode_kernel<<<(unsigned)enc_grid, WT_THREADS, 0, stream>>>(
        w, K, N, tiles_k, tiles_n, total, qT, sfT, reinterpret_cast<const uint32_t*>(s_w), mma_layout);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    ++launched;
    nvfp4_weight_finalize_kernel<<<(unsigned)((E + 255) / 256), 256, 0, stream>>>(s_w, E);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    count_launches(launched + 1);
    return cudaSuccess;
}

}  // namespace nvq
