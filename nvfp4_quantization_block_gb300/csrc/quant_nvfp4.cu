// NVFP4 per-token quantizer (activations; the expert weights are in quant_nvfp4_weights.cu).
//
// Definition [Miles-zh = page "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本":
// section "为什么需要 Blackwell 原生方案？" (E2M1 values, one E4M3 scale per 16 values rounded to
// nearest, a coarse FP32 scale on top); section "逐 Token 激活值缩放" (one FP32 scale per token computed
// online, fused into the quantization call that also emits the packed FP4 values and the block
// scales; gate/up weights share one FP32 scale); section "比特精确量化器合约" (bit-exact contract,
// no fast math)]. Coarse scale s = RN(amax / 2688); block scale = E4M3 RNE of amax_b / (6 s);
// code = E2M1 RNE (saturating) of x / (E4M3(sf) s). Exactness: see nvq_device.cuh.
//
// Design: one warp per token row, one 16-element block per lane per step (see the kernel). A scope
// whose table passes the product-path check (nvq_device.cuh) encodes its elements by one fp32
// multiply and the hardware E2M1 conversion; any other scope compares each element with its block's
// exact boundaries.

#include "../../include/nvq.h"
#include "nvq_device.cuh"
#include "nvq_internal.h"
#include "nvq_nvfp4_encode.cuh"

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
// silu(g) u with silu(g) = g / (1 + exp(-g)) (Shazeer 2020), computed with float32 significands and
// one rounding per operation (no contraction), so that it is reproducible bit for bit. exp is our
// own: x = -g clamped to [-87, 300] (neither bound changes a result), Cody and Waite's two-constant
// range reduction x = n ln2 + r, and a degree-6 Taylor polynomial p of e^r in Horner order, so
// exp(-g) ~ p 2^n. For x <= 87, 2^n is a normal float32 and the steps are plain IEEE float32:
// e = p 2^n, d = 1 + e, s = g / d, h = s u. For x > 87 exp(-g) may leave float32's range; its
// exponent is kept apart instead (swiglu_wide), so silu(g) u keeps its value there too. The two
// elements of a bf16x2 word go through every add, subtract and multiply together as one packed
// f32x2 operation (two IEEE operations, each rounded once, no flush to zero: the same values as the
// scalar steps); the divisions are scalar IEEE ones.
__device__ __forceinline__ void f2_add(float& y0, float& y1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(y0), "=f"(y1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void f2_sub(float& y0, float& y1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(y0), "=f"(y1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void f2_mul(float& y0, float& y1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(y0), "=f"(y1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void f2_fma(float& y0, float& y1, float a0, float a1, float b0, float b1, float c0,
                                       float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(y0), "=f"(y1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// div_markstein (nvq_device.cuh) for the two elements of a word at once: the same steps, each an
// IEEE operation on both elements (packed f32x2: one rounding each, no flush to zero), so the
// same quotients; `ok` covers both.
__device__ __forceinline__ void div_markstein2(float g0, float g1, float d0, float d1, float& q0, float& q1, bool& ok) {
    float y00, y01;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y00) : "f"(d0));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y01) : "f"(d1));
    const float n0 = __uint_as_float(__float_as_uint(d0) ^ 0x80000000u);   // -d, exactly
    const float n1 = __uint_as_float(__float_as_uint(d1) ^ 0x80000000u);
    float e0, e1, y0, y1, a0, a1, r0, r1;
    f2_fma(e0, e1, n0, n1, y00, y01, 1.0f, 1.0f);              // 1 - d y0
    f2_fma(y0, y1, y00, y01, e0, e1, y00, y01);                // y = y0 + y0 (1 - d y0)
    f2_mul(a0, a1, g0, g1, y0, y1);                            // q0 = RN(g y)
    f2_fma(r0, r1, n0, n1, a0, a1, g0, g1);                    // r = g - d q0 (exact)
    f2_fma(q0, q1, r0, r1, y0, y1, a0, a1);                    // RN(q0 + r y)
    ok = fabsf(a0) >= 0x1p-100f && fabsf(a1) >= 0x1p-100f;
}

// h for -g > 87, where exp(-g) = p 2^n may lie beyond float32's range (n up to 433): d = 1 + p 2^n
// is p 2^n exactly (1 is far below half an ulp of it), so s = g / d = RN(g / p) 2^-n, formed as
// q = RN((g 2^-16) / p) (finite for any bf16 g, the same rounding), and h = s u rounded once to
// float32 (gradual underflow) from the exact float64 product q u 2^(16 - n) (24 x 8 significant
// bits, times a power of two). m = 1.5 2^23 + n as computed by the caller.
__device__ __noinline__ float swiglu_wide(float g, float u, float p, float m) {
    const int n = (int)(__float_as_uint(m) - 0x4B400000u);
    const float q = __fdiv_rn(__fmul_rn(g, 0x1p-16f), p);
    const double pow2 = __longlong_as_double((long long)(1023 + 16 - n) << 52);
    return __double2float_rn(__dmul_rn(__dmul_rn((double)q, (double)u), pow2));
}

// bf16x2 word of SwiGLU(gate, up) for the bf16x2 words g and u; `rare` is set when an element
// needs the exact path (swiglu2_exact below): a gate with -g > 87 or a quotient the fast
// division does not cover.
__device__ __forceinline__ uint32_t swiglu2_fast(uint32_t g, uint32_t u, bool& rare) {
    constexpr float L2E = (float)1.4426950408889634, LN2_HI = 0.693145751953125f;
    constexpr float LN2_LO = (float)(0.6931471805599453 - 0.693145751953125), MAGIC = 12582912.0f;
    // x = -g clamped below at -87 in both halves at once (bf16 comparisons are exact; -87 = 0xC2AE);
    // no upper clamp here: an element with x > 87 sends its block to the exact steps anyway
    uint32_t xc;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(xc) : "r"(g ^ 0x80008000u), "r"(0xC2AEC2AEu));
    const float x0 = bf16_lo(xc), x1 = bf16_hi(xc);
    float t0, t1, m0, m1, n0, n1, a0, a1, r0, r1;
    f2_mul(t0, t1, x0, x1, L2E, L2E);
    f2_add(m0, m1, t0, t1, MAGIC, MAGIC);                      // 1.5 * 2^23 + n: n in the low mantissa bits
    f2_sub(n0, n1, m0, m1, MAGIC, MAGIC);                      // nearest integer to x log2(e), exactly
    f2_mul(a0, a1, n0, n1, LN2_HI, LN2_HI);
    f2_sub(r0, r1, x0, x1, a0, a1);
    f2_mul(a0, a1, n0, n1, LN2_LO, LN2_LO);
    f2_sub(r0, r1, r0, r1, a0, a1);
    float p0 = (float)(1.0 / 720.0), p1 = p0;
    const float c[6] = {(float)(1.0 / 120.0), (float)(1.0 / 24.0), (float)(1.0 / 6.0), 0.5f, 1.0f, 1.0f};
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        f2_mul(p0, p1, p0, p1, r0, r1);
        f2_add(p0, p1, p0, p1, c[i], c[i]);
    }
    // 2^n from the bits of 1.5 * 2^23 + n (n in [-126, 126] when x <= 87): (bits - 0x4B400000 + 127)
    // << 23 equals (bits << 23) + 0x3F800000 modulo 2^32 (0x4B400000 << 23 wraps to 0)
    const float s0 = __uint_as_float((__float_as_uint(m0) << 23) + 0x3F800000u);
    const float s1 = __uint_as_float((__float_as_uint(m1) << 23) + 0x3F800000u);
    float e0, e1, d0, d1, h0, h1;
    f2_mul(e0, e1, p0, p1, s0, s1);                            // exp(-g)
    f2_add(d0, d1, e0, e1, 1.0f, 1.0f);
    bool ok;
    float q0, q1;
    div_markstein2(bf16_lo(g), bf16_hi(g), d0, d1, q0, q1, ok);
    f2_mul(h0, h1, q0, q1, bf16_lo(u), bf16_hi(u));
    rare = rare || !(ok && x0 <= 87.0f && x1 <= 87.0f);
    return cvt_bf16x2(h0, h1);
}

// bf16x2 word of SwiGLU(gate, up) for the bf16x2 words g and u (every element exact)
__device__ __noinline__ uint32_t swiglu2(uint32_t g, uint32_t u) {
    constexpr float L2E = (float)1.4426950408889634, LN2_HI = 0.693145751953125f;
    constexpr float LN2_LO = (float)(0.6931471805599453 - 0.693145751953125), MAGIC = 12582912.0f;
    const uint32_t xw = g ^ 0x80008000u;                       // x = -g, both halves
    const float x0 = fminf(fmaxf(bf16_lo(xw), -87.0f), 300.0f), x1 = fminf(fmaxf(bf16_hi(xw), -87.0f), 300.0f);
    float t0, t1, m0, m1, n0, n1, a0, a1, r0, r1;
    f2_mul(t0, t1, x0, x1, L2E, L2E);
    f2_add(m0, m1, t0, t1, MAGIC, MAGIC);                      // 1.5 * 2^23 + n: n in the low mantissa bits
    f2_sub(n0, n1, m0, m1, MAGIC, MAGIC);                      // nearest integer to x log2(e), exactly
    f2_mul(a0, a1, n0, n1, LN2_HI, LN2_HI);
    f2_sub(r0, r1, x0, x1, a0, a1);
    f2_mul(a0, a1, n0, n1, LN2_LO, LN2_LO);
    f2_sub(r0, r1, r0, r1, a0, a1);
    float p0 = (float)(1.0 / 720.0), p1 = p0;
    const float c[6] = {(float)(1.0 / 120.0), (float)(1.0 / 24.0), (float)(1.0 / 6.0), 0.5f, 1.0f, 1.0f};
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        f2_mul(p0, p1, p0, p1, r0, r1);
        f2_add(p0, p1, p0, p1, c[i], c[i]);
    }
    // 2^n from the bits of 1.5 * 2^23 + n (n in [-126, 126] when x <= 87; the other lanes'
    // values here are discarded)
    const float s0 = __uint_as_float((__float_as_uint(m0) - 0x4B400000u + 127u) << 23);
    const float s1 = __uint_as_float((__float_as_uint(m1) - 0x4B400000u + 127u) << 23);
    float e0, e1, d0, d1, h0, h1;
    f2_mul(e0, e1, p0, p1, s0, s1);                            // exp(-g)
    f2_add(d0, d1, e0, e1, 1.0f, 1.0f);
    const float q0 = __fdiv_rn(bf16_lo(g), d0), q1 = __fdiv_rn(bf16_hi(g), d1);
    f2_mul(h0, h1, q0, q1, bf16_lo(u), bf16_hi(u));
    if (x0 > 87.0f) h0 = swiglu_wide(bf16_lo(g), bf16_lo(u), p0, m0);
    if (x1 > 87.0f) h1 = swiglu_wide(bf16_hi(g), bf16_hi(u), p1, m1);
    return cvt_bf16x2(h0, h1);
}

// One 16-element block of the row: loaded as is, or (SWIGLU) formed from the gate block at p and
// the up block at p + up.
template <bool V8, bool SWIGLU>
__device__ __forceinline__ void row_block(const uint16_t* p, int64_t up, uint4& a, uint4& b) {
    load_block<V8>(p, a, b);
    if (SWIGLU) {
        uint4 ua, ub;
        load_block<V8>(p + up, ua, ub);
        // the fast steps for the whole block; a block with any element outside their range (rare)
        // is formed again element by element with the exact steps
        bool rare = false;
        a = make_uint4(swiglu2_fast(a.x, ua.x, rare), swiglu2_fast(a.y, ua.y, rare), swiglu2_fast(a.z, ua.z, rare),
                       swiglu2_fast(a.w, ua.w, rare));
        b = make_uint4(swiglu2_fast(b.x, ub.x, rare), swiglu2_fast(b.y, ub.y, rare), swiglu2_fast(b.z, ub.z, rare),
                       swiglu2_fast(b.w, ub.w, rare));
        if (rare) {
            // the block's gate and up words again (rare: no registers kept for them)
            load_block<V8>(p, a, b);
            load_block<V8>(p + up, ua, ub);
            a = make_uint4(swiglu2(a.x, ua.x), swiglu2(a.y, ua.y), swiglu2(a.z, ua.z), swiglu2(a.w, ua.w));
            b = make_uint4(swiglu2(b.x, ub.x), swiglu2(b.y, ub.y), swiglu2(b.z, ub.z), swiglu2(b.w, ub.w));
        }
    }
}

// Where one lane's outputs of one token row go: the lane holds blocks l, l + LPR, l + 2 LPR, ...
// of the row (step i: block i LPR + l), with their packed codes at q + i LPR 8 and their scale
// bytes at sf + i SF_STEP (canonical rows: consecutive bytes; MMA layout: the row's place in its
// tile column, LPR / 4 tile columns further per step).
struct TokenLaneOut {
    uint8_t* q;          // codes of the lane's block of step 0
    uint8_t* sf;         // scale byte of the lane's block of step 0, or nullptr (row not covered)
    int nkb_lane;        // the row's blocks from block l on: step i holds codes when i LPR < nkb_lane
    int nsf_lane;        // the same for scale bytes (MMA layout: up to the padded multiple of 4 blocks,
                         // whose padding bytes are the zero codes of the zero blocks beyond the row)
};

// Stores of the lane's block of step i (codes c0, c1, scale code sfc); each lane stores its own
// scale byte (the four bytes of a scale word come from four neighbouring lanes in one instruction).
// FULL: every lane of the warp has a block at every step taken, in a real row (no guards).
template <int LPR, bool FULL, bool MMA>
__device__ __forceinline__ void token_store(uint32_t sfc, uint32_t c0, uint32_t c1, int i, bool real,
                                            const TokenLaneOut& o) {
    constexpr int SF_STEP = MMA ? (LPR / 4) * 512 : LPR;
    if (FULL || (real && i * LPR < o.nkb_lane))
        *reinterpret_cast<uint2*>(o.q + (int64_t)i * LPR * 8) = make_uint2(c0, c1);
    if (FULL || (o.sf != nullptr && i * LPR < o.nsf_lane)) o.sf[(int64_t)i * SF_STEP] = (uint8_t)sfc;
}

// Encode and store one block; the encoding mode is the same for every lane.
template <int MODE, int LPR, bool FULL, bool MMA>
__device__ __forceinline__ void token_block(const uint4& a, const uint4& b, uint32_t mb, int i, bool real,
                                            const Nvfp4Scope& sc, const Nvfp4Table& T, const Nvfp4CodeInfo& I,
                                            const TokenLaneOut& o) {
    uint32_t c0, c1;
    const uint32_t sfc = encode_block<MODE>(a, b, mb, sc, T, I, c0, c1);
    token_store<LPR, FULL, MMA>(sfc, c0, c1, i, real, o);
}

// Encode and store one block when the two rows of a warp may take different paths.
template <int LPR, bool FULL, bool MMA>
__device__ __forceinline__ void token_block_mixed(const uint4& a, const uint4& b, uint32_t mb, int i, bool real,
                                                  int mode, const Nvfp4Scope& sc, const Nvfp4Table& T,
                                                  const Nvfp4CodeInfo& I, const TokenLaneOut& o) {
    uint32_t c0, c1, sfc;
    if (mode == ENC_PRODUCT) sfc = encode_block<ENC_PRODUCT>(a, b, mb, sc, T, I, c0, c1);
    else if (mode == ENC_TABLE) sfc = encode_block<ENC_TABLE>(a, b, mb, sc, T, I, c0, c1);
    else sfc = encode_block<ENC_EXACT>(a, b, mb, sc, T, I, c0, c1);
    token_store<LPR, FULL, MMA>(sfc, c0, c1, i, real, o);
}

// The scope table of a row built by its LPR lanes, with the product path's multipliers (32:
// nvfp4_table_build_warp; 16: lane l takes thresholds j = (l >> 3) + 2t, t = 0, 1, of class l & 7
// and their j + 4 partners, and the block-scale boundary of code l; a class's two lanes are l and
// l ^ 8 of the same half-warp). Called by all 32 lanes of the warp together; returns whether the
// lane's class has a product-path multiplier. Every row searches (131072 x 768 SwiGLU rows: 0.1604
// ms without the search, 0.1584-0.1593 with it, once the SwiGLU divisions ran packed; plain
// 768-wide rows: 0.076 ms without, 0.072 with).
template <int LPR, bool SEARCH>
__device__ __forceinline__ bool nvfp4_table_build_row(Nvfp4Table& T, float s, int l) {
    if (LPR == 32) return nvfp4_table_build_warp(T, s, l);
    const uint32_t f = (uint32_t)l & 7u, jb = (uint32_t)l >> 3;
    const float v = (float)(8u + f) * 0x1p-9f;                     // value of E4M3 code 8 + f
    const uint32_t g0 = nvfp4_class_g0(v, s);
    uint32_t bd[4];                                                // thresholds jb, jb + 4, jb + 2, jb + 6
#pragma unroll
    for (uint32_t t = 0; t < 2; ++t) {
        const uint32_t j = jb + 2u * t;                            // 0..3
        const uint32_t b = bf16_boundary((float)(2u * j + 1u) * 0.25f * v, s, (j & 1u) != 0u);
        T.bp[f][j] = b | (b << 16);
        if (j < 3u) T.bp[f][8u + j] = (b | (b << 16)) ^ 0x80008000u;
        bd[2 * t] = b;
        bd[2 * t + 1] = 0u;
        const uint32_t j2 = j + 4u;
        if (j2 < 7u) {
            const float m = (j2 == 6u) ? 5.0f : (float)j2 - 1.5f;
            const uint32_t b2 = bf16_boundary(m * v, s, (j2 & 1u) != 0u);
            T.bp[f][j2] = b2 | (b2 << 16);
            bd[2 * t + 1] = b2;
        }
    }
    const uint32_t g = !SEARCH ? 0u : nvfp4_search_multiplier(g0, [&](uint32_t gk) {
        uint32_t m = 0u;
#pragma unroll
        for (uint32_t t = 0; t < 2; ++t) {
            const uint32_t j = jb + 2u * t;
            m |= nvfp4_product_miss(bd[2 * t], j, __uint_as_float(gk));
            if (j + 4u < 7u) m |= nvfp4_product_miss(bd[2 * t + 1], j + 4u, __uint_as_float(gk));
        }
        return m | __shfl_xor_sync(0xffffffffu, m, 8);
    });
    T.bs[l] = bf16_boundary((float)(3 * (2 * l + 1)) * 0x1p-9f, s, (l & 1) != 0);
    if (l < 12) T.bp[8][l] = l < 7 ? 0x7F007F00u : (l >= 8 && l < 11 ? 0xFF00FF00u : 0u);
    if (l < 8) T.g[l] = g;
    if (l == 8) T.g[8] = 0u;
    return g != 0u;
}

// The rows of one warp (LPR lanes each), from their loads to their stores. FULL: every row of the
// warp is real and every lane has a block at each of the row's steps (the block count a multiple of
// LPR, at most TOK_NREG steps), so no load or store needs a guard.
template <bool V8, bool SWIGLU, int LPR, bool FULL, bool MMA>
__device__ __forceinline__ void token_rows(const uint16_t* __restrict__ x, int64_t C, int64_t ldx,
                                           uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                           float* __restrict__ s_tok, int64_t row, bool covered, bool real,
                                           int l, int half, Nvfp4Table& T, const Nvfp4CodeInfo& info) {
    const int64_t nkb = C >> 4;                                // 16-element blocks
    const int iters = (int)((nkb + LPR - 1) / LPR);
    const int nkb_lane = (int)(nkb - l);                       // step i holds a block when i LPR < nkb_lane
    const uint16_t* xl = x + (real ? row : 0) * ldx + l * 16;  // the lane's block of step 0

    // pass 1: load (into registers where possible) and reduce the row's amax
    uint4 va[TOK_NREG], vb[TOK_NREG];
    uint32_t mbk[TOK_NREG];                                    // block maxima of the register-resident blocks
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < TOK_NREG; ++i) {
        if (FULL && i < iters) {
            row_block<V8, SWIGLU>(xl + i * LPR * 16, C, va[i], vb[i]);
        } else {
            va[i] = vb[i] = make_uint4(0u, 0u, 0u, 0u);
            if (!FULL && real && i * LPR < nkb_lane) row_block<V8, SWIGLU>(xl + i * LPR * 16, C, va[i], vb[i]);
        }
        mbk[i] = absmax_bits_16(va[i], vb[i]);
        m = max(m, mbk[i]);
    }
    if (!FULL) {
        for (int i = TOK_NREG; i < iters; ++i) {
            if (real && i * LPR < nkb_lane) {
                uint4 a, b;
                row_block<V8, SWIGLU>(xl + (int64_t)i * LPR * 16, C, a, b);
                m = max(m, absmax_bits_16(a, b));
            }
        }
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = nvfp4_coarse_scale(__uint_as_float(m << 16));
    const Nvfp4Scope sc = make_nvfp4_scope(s);
    if (real && l == 0) s_tok[row] = s;
    // every row builds a table (all lanes take part in its shuffles); an exact-path row ignores it
    constexpr bool SEARCH = true;                              // rows that may take the product path
    const bool ok = nvfp4_table_build_row<LPR, SEARCH>(T, s, l);
    __syncwarp();
    const uint32_t bad = __ballot_sync(0xffffffffu, !ok);
    const uint32_t row_bad = LPR == 32 ? bad : (bad >> (half * LPR)) & ((1u << LPR) - 1u);
    const int mode = sc.exact ? ENC_EXACT : ((SEARCH && row_bad == 0u) ? ENC_PRODUCT : ENC_TABLE);

    // pass 2: per 1x16 block scale and codes (register-resident blocks first, then any reloads)
    TokenLaneOut o;
    o.q = q + (real ? row : 0) * (C >> 1) + l * 8;
    o.nkb_lane = nkb_lane;
    o.nsf_lane = (int)((MMA ? (nkb + 3) & ~int64_t(3) : nkb) - l);
    o.sf = !covered ? nullptr : (MMA ? sf + mma_sf_offset(row, l, nkb) : sf + row * nkb + l);
    const uint32_t same = __match_any_sync(0xffffffffu, mode);
    if (same == 0xffffffffu && mode == ENC_PRODUCT) {
#pragma unroll
        for (int i = 0; i < TOK_NREG; ++i)
            if (i < iters) token_block<ENC_PRODUCT, LPR, FULL, MMA>(va[i], vb[i], mbk[i], i, real, sc, T, info, o);
    } else if (same == 0xffffffffu && mode == ENC_TABLE) {
#pragma unroll
        for (int i = 0; i < TOK_NREG; ++i)
            if (i < iters) token_block<ENC_TABLE, LPR, FULL, MMA>(va[i], vb[i], mbk[i], i, real, sc, T, info, o);
    } else if (same == 0xffffffffu) {
#pragma unroll
        for (int i = 0; i < TOK_NREG; ++i)
            if (i < iters) token_block<ENC_EXACT, LPR, FULL, MMA>(va[i], vb[i], mbk[i], i, real, sc, T, info, o);
    } else {
        // the two rows of the warp take different modes
#pragma unroll
        for (int i = 0; i < TOK_NREG; ++i)
            if (i < iters) token_block_mixed<LPR, FULL, MMA>(va[i], vb[i], mbk[i], i, real, mode, sc, T, info, o);
    }
    if (!FULL) {
        for (int i = TOK_NREG; i < iters; ++i) {
            uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
            if (real && i * LPR < nkb_lane) row_block<V8, SWIGLU>(xl + (int64_t)i * LPR * 16, C, a, b);
            token_block_mixed<LPR, FULL, MMA>(a, b, absmax_bits_16(a, b), i, real, mode, sc, T, info, o);
        }
    }
}

// LPR lanes per token row (32: one row per warp; 16: two rows per warp, for rows of at most 64
// blocks, so that rows of 48 blocks keep every lane busy), one 16-element block per lane per step:
// the row is loaded once with 32-byte coalesced loads (held in registers up to TOK_NREG steps),
// reduced to its amax with shuffles among the row's lanes, and encoded from registers, so each
// input byte is read from HBM once. MMA: scale bytes in the tile layout (else canonical rows).
template <bool V8, bool SWIGLU, int LPR, bool MMA>
// 6 CTAs per SM (80 registers, no spills; 24 warps keep enough row loads in flight: 131072 x 2048
// rows 0.218 ms at 142 registers, 0.179 at 128, 0.158 at 96, 0.146 at 80); the SwiGLU variant keeps
// 5 (96 registers; at 80 it spills).
__global__ void __launch_bounds__(TOK_THREADS, SWIGLU ? 5 : 6)
nvfp4_token_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ldx,
                   uint8_t* __restrict__ q, uint8_t* __restrict__ sf, float* __restrict__ s_tok,
                   int64_t rows_cover) {
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
    const int64_t nkb = C >> 4;
    // uniform over the warp: whole steps for every lane, and every row of the warp real
    const bool full = nkb % LPR == 0 && nkb <= (int64_t)TOK_NREG * LPR && row0 + RPW - 1 < R;
    if (full)
        token_rows<V8, SWIGLU, LPR, true, MMA>(x, C, ldx, q, sf, s_tok, row, covered, real, l, half, T, info);
    else
        token_rows<V8, SWIGLU, LPR, false, MMA>(x, C, ldx, q, sf, s_tok, row, covered, real, l, half, T, info);
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
#define NVQ_TOK(V, L, M)                                                                                          \
    lerr = launch_pdl(nvfp4_token_kernel<V, SWIGLU, L, M>, dim3((unsigned)grid), dim3(TOK_THREADS), 0, stream, x, R, \
                      C, ldx, q, sf, s_tok, cover)
#define NVQ_TOK_L(V, M)                                                                                           \
    if (pair) NVQ_TOK(V, 16, M);                                                                                  \
    else NVQ_TOK(V, 32, M)
    if (v8) {
        if (mma_layout) NVQ_TOK_L(true, true);
        else NVQ_TOK_L(true, false);
    } else {
        if (mma_layout) NVQ_TOK_L(false, true);
        else NVQ_TOK_L(false, false);
    }
#undef NVQ_TOK_L
#undef NVQ_TOK
    const cudaError_t err = lerr != cudaSuccess ? lerr : cudaGetLastError();
    if (err == cudaSuccess) count_launches(1);
    return err;
}

// ------------------------------------------------------------------------------------------------
// Quantize-once dispatch. Per-token scales make a token's NVFP4 bytes independent of every other
// row [Miles-zh, "逐 Token 激活值缩放"], so a routed MoE layer can quantize each token once and copy
// its bytes to every expert segment it is routed to. One warp per token: the token is quantized by
// the per-token path above (one row of 32 lanes) into the warp's staging area in shared memory
// (codes, canonical scale bytes, token scale), then the warp writes the staged row to each of the
// token's routed rows: 16-byte code stores (8-byte when a row of codes is not a multiple of 16
// bytes), one 4-byte scale word per 4-column group, the token scale. Warps past the tokens zero the
// MMA layout's padding rows below the last routed row (what the gather and the per-token quantizer
// leave there). Each input byte is read once; each routed row is written once.
// ------------------------------------------------------------------------------------------------
constexpr int64_t DSP_MAX_COLS = 16384;

__host__ __device__ __forceinline__ int64_t dsp_stage_bytes(int64_t C) {
    const int64_t qb = C >> 1, nkb4 = ((C >> 4) + 3) & ~int64_t(3);
    return ((qb + nkb4 + 15) & ~int64_t(15)) + 16;             // codes, scale bytes, token scale
}

template <bool V8, bool MMA>
__global__ void __launch_bounds__(TOK_THREADS, 5)
nvfp4_dispatch_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t C, int64_t ldx,
                      const int32_t* __restrict__ dest, int topk, int64_t R, int64_t pad_rows,
                      uint8_t* __restrict__ q, uint8_t* __restrict__ sf, float* __restrict__ s_tok,
                      int32_t* __restrict__ status) {
    griddep_begin();
    extern __shared__ __align__(16) uint8_t dsp_stage[];
    __shared__ Nvfp4Table tables[TOK_THREADS / 32];
    __shared__ Nvfp4CodeInfo info;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (uint32_t c = threadIdx.x; c < 128u; c += TOK_THREADS) nvfp4_code_info_build(info, c);
    __syncthreads();
    const int64_t w = (int64_t)blockIdx.x * (TOK_THREADS / 32) + warp;   // token w, then padding rows
    const int64_t nkb = C >> 4, qb = C >> 1, ngr = (nkb + 3) >> 2;       // blocks, code bytes, scale words
    if (w >= T) {
        const int64_t r = R + (w - T);                         // uniform over the warp
        if (MMA && r < R + pad_rows)
            for (int64_t g = lane; g < ngr; g += 32) *reinterpret_cast<uint32_t*>(sf + mma_sf_offset(r, 4 * g, nkb)) = 0u;
        return;
    }
    const int32_t mine = lane < topk ? dest[w * topk + lane] : -1;   // in flight while the token is quantized
    const int64_t sb = dsp_stage_bytes(C);
    uint8_t* sq = dsp_stage + warp * sb;                       // staged codes [qb]
    uint8_t* ssf = sq + qb;                                    // staged scale bytes [nkb]
    float* ss = reinterpret_cast<float*>(sq + sb - 16);        // staged token scale
    // the token quantized as a one-row batch (rows of 32 lanes, canonical scale bytes)
    const uint16_t* xt = x + w * ldx;
    if (nkb % 32 == 0 && nkb <= (int64_t)TOK_NREG * 32)
        token_rows<V8, false, 32, true, false>(xt, C, ldx, sq, ssf, ss, 0, true, true, lane, 0, tables[warp], info);
    else
        token_rows<V8, false, 32, false, false>(xt, C, ldx, sq, ssf, ss, 0, true, true, lane, 0, tables[warp], info);
    __syncwarp();
    const float s = *ss;
    if (qb <= 1024 && (qb & 15) == 0) {
        // rows of at most 2048 elements: each lane's share of the staged token (two 16-byte code
        // pieces and one scale word) is read from shared memory once and stored from registers to
        // every routed row
        const int64_t o0 = (int64_t)lane * 16, o1 = o0 + 512;
        uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
        if (o0 < qb) c0 = *reinterpret_cast<const uint4*>(sq + o0);
        if (o1 < qb) c1 = *reinterpret_cast<const uint4*>(sq + o1);
        uint32_t word = 0u;
        const int64_t valid = nkb - 4 * (int64_t)lane;         // scale bytes of the lane's group that exist
        if (lane < ngr) {
            word = *reinterpret_cast<const uint32_t*>(ssf + 4 * lane);
            if (valid < 4) word &= (1u << (8 * valid)) - 1u;
        }
        for (int k = 0; k < topk; ++k) {
            const int32_t r = __shfl_sync(0xffffffffu, mine, k);
            if (r == -1) continue;                             // uniform over the warp
            if (r < 0 || r >= R) {
                if (lane == 0 && status != nullptr) atomicExch(status, NVQ_DEV_BAD_INDEX);
                continue;
            }
            uint8_t* qd = q + (int64_t)r * qb;
            if (o0 < qb) *reinterpret_cast<uint4*>(qd + o0) = c0;
            if (o1 < qb) *reinterpret_cast<uint4*>(qd + o1) = c1;
            if (lane < ngr) {
                if (MMA) {
                    *reinterpret_cast<uint32_t*>(sf + mma_sf_offset(r, 4 * lane, nkb)) = word;
                } else if ((nkb & 3) == 0) {
                    *reinterpret_cast<uint32_t*>(sf + (int64_t)r * nkb + 4 * lane) = word;
                } else {
                    for (int64_t j = 0; j < 4 && j < valid; ++j)
                        sf[(int64_t)r * nkb + 4 * lane + j] = (uint8_t)(word >> (8 * j));
                }
            }
            if (lane == 0) s_tok[r] = s;
        }
        return;
    }
    for (int k = 0; k < topk; ++k) {
        const int32_t r = __shfl_sync(0xffffffffu, mine, k);
        if (r == -1) continue;                                 // uniform over the warp
        if (r < 0 || r >= R) {
            if (lane == 0 && status != nullptr) atomicExch(status, NVQ_DEV_BAD_INDEX);
            continue;
        }
        uint8_t* qd = q + (int64_t)r * qb;
        if ((qb & 15) == 0) {
            for (int64_t c = lane * 16; c < qb; c += 32 * 16)
                *reinterpret_cast<uint4*>(qd + c) = *reinterpret_cast<const uint4*>(sq + c);
        } else {
            for (int64_t c = lane * 8; c < qb; c += 32 * 8)
                *reinterpret_cast<uint2*>(qd + c) = *reinterpret_cast<const uint2*>(sq + c);
        }
        for (int64_t g = lane; g < ngr; g += 32) {
            uint32_t word = *reinterpret_cast<const uint32_t*>(ssf + 4 * g);
            const int64_t valid = nkb - 4 * g;                 // scale bytes of this group that exist
            if (valid < 4) word &= (1u << (8 * valid)) - 1u;
            if (MMA) {
                *reinterpret_cast<uint32_t*>(sf + mma_sf_offset(r, 4 * g, nkb)) = word;
            } else if ((nkb & 3) == 0) {
                *reinterpret_cast<uint32_t*>(sf + (int64_t)r * nkb + 4 * g) = word;
            } else {
                for (int64_t j = 0; j < 4 && j < valid; ++j) sf[(int64_t)r * nkb + 4 * g + j] = (uint8_t)(word >> (8 * j));
            }
        }
        if (lane == 0) s_tok[r] = s;
    }
}

cudaError_t launch_nvfp4_quantize_dispatch(const uint16_t* x, int64_t T, int64_t C, int64_t ldx, const int32_t* dest,
                                           int topk, int64_t R, uint8_t* q, uint8_t* sf, float* s_tok, int mma_layout,
                                           int32_t* status, cudaStream_t stream) {
    const int64_t pad_rows = mma_layout ? (((R + 127) & ~int64_t(127)) - R) : 0;
    const int64_t warps = T + pad_rows;
    if (warps == 0) return cudaSuccess;
    const int64_t grid = (warps + TOK_THREADS / 32 - 1) / (TOK_THREADS / 32);
    const size_t smem = (size_t)(TOK_THREADS / 32) * (size_t)dsp_stage_bytes(C);
    const bool v8 = ((reinterpret_cast<uintptr_t>(x) & 31u) == 0) && (ldx % 16 == 0);
    cudaError_t err;
    if (v8) {
        if (mma_layout) err = launch_pdl(nvfp4_dispatch_kernel<true, true>, dim3((unsigned)grid), dim3(TOK_THREADS), smem,
                                         stream, x, T, C, ldx, dest, topk, R, pad_rows, q, sf, s_tok, status);
        else err = launch_pdl(nvfp4_dispatch_kernel<true, false>, dim3((unsigned)grid), dim3(TOK_THREADS), smem,
                              stream, x, T, C, ldx, dest, topk, R, pad_rows, q, sf, s_tok, status);
    } else {
        if (mma_layout) err = launch_pdl(nvfp4_dispatch_kernel<false, true>, dim3((unsigned)grid), dim3(TOK_THREADS), smem,
                                         stream, x, T, C, ldx, dest, topk, R, pad_rows, q, sf, s_tok, status);
        else err = launch_pdl(nvfp4_dispatch_kernel<false, false>, dim3((unsigned)grid), dim3(TOK_THREADS), smem,
                              stream, x, T, C, ldx, dest, topk, R, pad_rows, q, sf, s_tok, status);
    }
    if (err == cudaSuccess) err = cudaGetLastError();
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

}  // namespace nvq
