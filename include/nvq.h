/*
 * nvq.h — C-ABI of the GB300 (sm_103a) MXFP8 / per-token NVFP4 quantizers and the block-scaled
 * grouped GEMM they feed.
 *
 * Sources (page titles):
 *   [Miles-zh]  "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本" — Chinese translation of the
 *               Miles post on Blackwell-native 8-bit / 4-bit RL (the most detailed page).
 *   [Miles-fr]  "Miles Blackwell remplace l'uniformité BF16 par MXFP8 et NVFP4 natifs".
 *   [NVFP4-ru]  "NVIDIA верифицировала 4-битный формат NVFP4 на Mamba-Transformer (12B) при 10 трлн
 *               токенов".
 *
 * Conventions that hold for every entry point:
 *   - Every pointer argument is a DEVICE pointer (CUDA global memory) unless stated; the caller
 *     allocates and owns every buffer. The library never allocates, frees or synchronises.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *     stream) and runs asynchronously; outputs are valid once the stream reaches that point.
 *   - Argument errors are detected on the host before anything is launched; the call then
 *     returns a non-zero nvq_status and leaves every output untouched.
 *   - bf16 inputs are row-major with a leading dimension `ld*` in elements; they must be finite
 *     (non-finite inputs are outside the quantizer contract, and the outputs are then unspecified).
 *   - Pointers must be 16-byte aligned; leading dimensions of bf16 inputs multiples of 8.
 *   - Quantized codes and scales are bytes. Scale matrices are either CANONICAL (row-major
 *     [rows, cols/block]) or MMA (the tcgen05 block-scale tile layout: 128-row x 4-column tiles of
 *     512 bytes, the scale of (r, c) at tile (r/128, c/4) offset (r%32)*16 + (r%128/32)*4 + c%4,
 *     tiles row-tile major, rows padded to 128 and columns to 4 with zero bytes; size from
 *     nvq_sf_bytes).
 */
#ifndef NVQ_H
#define NVQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVQ_OK = 0,
    NVQ_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, size out of range or not a required multiple */
    NVQ_ERR_MISALIGNED = 2,    /* a pointer or leading dimension violates the alignment rules */
    NVQ_ERR_UNSUPPORTED = 3,   /* a valid combination this build does not implement */
    NVQ_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    NVQ_ERR_TIMEOUT = 5        /* a kernel gave up a bounded wait (reported through a status word) */
} nvq_status;

typedef enum { NVQ_SF_CANONICAL = 0, NVQ_SF_MMA = 1 } nvq_sf_layout;
typedef enum { NVQ_MXFP8 = 0, NVQ_NVFP4 = 1, NVQ_BF16 = 2 } nvq_format;   /* NVQ_BF16: GEMM operands only */
typedef enum { NVQ_SCOPE_ROW = 0, NVQ_SCOPE_MATRIX = 1 } nvq_scope;

/* Human-readable name of a status code (static string). */
const char* nvq_status_string(nvq_status s);

/* Number of kernels this library has enqueued since it was loaded, counted on the host at each
 * successful launch (diagnostics: lets a caller confirm which work ran in these kernels). */
uint64_t nvq_launch_count(void);

/* Bytes of a scale matrix for `rows` rows and `cols` elements per row quantized in blocks of
 * `block` (32 for MXFP8, 16 for NVFP4): rows*cols/block (CANONICAL) or the padded tile size (MMA).
 * Returns -1 on invalid arguments. Host-only; touches no device state. */
int64_t nvq_sf_bytes(int64_t rows, int64_t cols, int32_t block, nvq_sf_layout layout);

/*
 * mxfp8_quantize — MXFP8 rowwise (1x32) and columnwise (32x1) copies of X in one pass over HBM.
 *
 * Defines: per block of 32, amax = max|x|; e = the smallest integer with amax <= 448 * 2^e,
 * clamped to [-127, 127] (E8M0 scale "rounded up so the block max is not clipped"); scale byte =
 * e + 127; codes = E4M3 round-to-nearest-even, satfinite, of x * 2^-e (sign kept on zeros).
 * [Miles-zh, "为什么需要 Blackwell 原生方案？" (MXFP8 paragraph); "方案 1：端到端 MXFP8 强化学习": the
 * rowwise and columnwise copies are numerically different, each is quantized independently from
 * the full-precision input, and both are materialised during quantization.]
 *
 *   x        bf16 [rows, cols], leading dimension ldx (elements).
 *   q_row    [rows, cols] E4M3 codes (dense), blocks along a row;        NULL = skip the rowwise copy.
 *   sf_row   scales of q_row: [rows, cols/32] or MMA layout of that;     NULL iff q_row is NULL.
 *   q_colT   [cols, rows] E4M3 codes = columnwise copy stored transposed (each stored row is one
 *            input column; blocks of 32 run along it);                   NULL = skip the columnwise copy.
 *   sf_colT  scales of q_colT: [cols, rows/32] or MMA layout of that;    NULL iff q_colT is NULL.
 * Requires cols % 32 == 0; rows % 32 == 0 when the columnwise copy is requested. rows or cols = 0
 * is a no-op.
 */
nvq_status mxfp8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                          uint8_t* q_row, uint8_t* sf_row, uint8_t* q_colT, uint8_t* sf_colT,
                          nvq_sf_layout sf_layout, void* stream);

/*
 * nvfp4_quantize_per_token — per-token NVFP4: packed E2M1 values, E4M3 block scales and one FP32
 * scale per row, from one call.
 *
 * Defines: per row, s = RN_fp32(amax_row / 2688) (2688 = 6 * 448, the largest E2M1 value times
 * the largest E4M3 scale; subnormal s kept); per block of 16, sf = E4M3 round-to-nearest-even,
 * satfinite, of amax_block / (6 s) (0 when s = 0); code = E2M1 round-to-nearest-even, satfinite,
 * of x / (E4M3(sf) * s) (signed zero when E4M3(sf) = 0). Every quotient is rounded once from its
 * exact value (no fast math). Element 2j is the low nibble of byte j.
 * [Miles-zh, "逐 Token 激活值缩放": one FP32 activation scale per token computed online, fused into
 * the activation-quantization call that also emits packed FP4 values and E4M3 block scales;
 * "为什么需要 Blackwell 原生方案？" (NVFP4: 16-value blocks, E4M3 scale rounded to nearest, coarse FP32
 * scale); "比特精确量化器合约": bit-exact quantizer contract, fast math disabled.]
 *
 *   x      bf16 [rows, cols], leading dimension ldx.
 *   q      [rows, cols/2] packed codes (dense).
 *   sf     [rows, cols/16] scales, or MMA layout of that.
 *   s_tok  [rows] float32 coarse scales (decode multipliers: x ~ E2M1 * E4M3(sf) * s_tok).
 * Requires cols % 16 == 0, cols <= 2^30 and rows <= 2^32 (NVQ_ERR_INVALID_ARG otherwise). rows = 0
 * is a no-op.
 */
nvq_status nvfp4_quantize_per_token(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                    uint8_t* q, uint8_t* sf, float* s_tok,
                                    nvq_sf_layout sf_layout, void* stream);

/*
 * nvfp4_quantize_dispatch — quantize-once dispatch: per-token NVFP4 of each token, written straight
 * to every routed row the token is dispatched to (its top-k experts' segments), in one pass.
 *
 * Defines: for every token t and k < topk with r = dest[t * topk + k] >= 0, routed row r of the
 * outputs (codes, block scales, token scale) is byte for byte nvfp4_quantize_per_token of row t of x.
 * Because a token's per-token bytes depend on that row only, this equals quantizing the routed
 * (gathered) bf16 rows, and equals nvfp4_quantize_per_token of the tokens followed by
 * quantized_gather_rows with the inverse index. [Miles-zh, "逐 Token 激活值缩放": one FP32 scale per
 * token computed online, so the rollout can quantize once and dispatch the packed values.]
 *
 *   x      bf16 [tokens, cols], leading dimension ldx.
 *   dest   device int32 [tokens, topk]: the routed row of each (token, k), or -1 (not dispatched).
 *          Any other value outside [0, rows) sets *status to NVQ_DEV_BAD_INDEX (when status is
 *          non-NULL) and that entry is skipped. Each routed row should be named at most once (otherwise one of the
 *          tokens naming it wins).
 *   rows   routed rows of the outputs.
 *   q      [rows, cols/2] packed codes; sf [rows, cols/16] scales or MMA layout of that (its padding
 *          rows below `rows` are zeroed); s_tok [rows] float32.
 *   Routed rows that no entry of dest names are left as they were.
 * Requires cols % 16 == 0, 0 < cols <= 16384, 1 <= topk <= 32, tokens <= 2^32, rows < 2^31;
 * x, q and sf 16-byte aligned, dest, s_tok and status 4-byte aligned. tokens = rows = 0 is a no-op.
 */
nvq_status nvfp4_quantize_dispatch(const void* x, int64_t tokens, int64_t cols, int64_t ldx,
                                   const int32_t* dest, int32_t topk, int64_t rows,
                                   uint8_t* q, uint8_t* sf, float* s_tok, nvq_sf_layout sf_layout,
                                   int32_t* status, void* stream);

/*
 * nvfp4_swiglu_quantize_per_token — the down projection's per-token NVFP4 input straight from the
 * fused gate||up GEMM output: SwiGLU, then per-token NVFP4, without writing the bf16 activation.
 *
 * Defines: h[i, j] = RN_bf16(silu(g) * u), g = gate_up[i, j], u = gate_up[i, cols + j], silu(g) =
 * g / (1 + exp(-g)) with float32 significands and one rounding per operation, exp(x) = p(r) * 2^n
 * (x = -g clamped to [-87, 300], which changes no result; n the nearest integer to x log2(e);
 * r = (x - n ln2_hi) - n ln2_lo with ln2_hi = 0x3F317200; p the degree-6 Taylor polynomial of e^r
 * in Horner order). exp(-g), 1 + exp(-g) and the quotient carry an unbounded exponent (for
 * x <= 87 these are the plain IEEE float32 steps); the product with u is rounded once to float32
 * (gradual underflow), then to bf16. Then exactly nvfp4_quantize_per_token of h.
 * [Miles-zh, "逐 Token 激活值缩放": SwiGLU experts run gate and up as one fused GEMM; one call emits
 * FP4 values, E4M3 block scales and per-token FP32 scales; "结果": the unfused scaling op is what
 * slowed the training path.]
 *
 *   gate_up  bf16 [rows, 2*cols], leading dimension ld (>= 2*cols, multiple of 8): gate in the
 *            first cols columns, up in the next cols.
 *   q, sf, s_tok  as nvfp4_quantize_per_token for h [rows, cols].
 * Requires cols % 16 == 0, cols <= 2^30 and rows <= 2^32. Inputs whose SwiGLU overflows bf16 are
 * outside the contract.
 */
nvq_status nvfp4_swiglu_quantize_per_token(const void* gate_up, int64_t rows, int64_t cols, int64_t ld,
                                           uint8_t* q, uint8_t* sf, float* s_tok,
                                           nvq_sf_layout sf_layout, void* stream);

/*
 * nvfp4_quantize_weights — NVFP4 expert weights with one FP32 scale per expert matrix, 1x16 blocks
 * along the reduction dimension K, written K-major (transposed) for the GEMM.
 *
 * Defines: as nvfp4_quantize_per_token, with the coarse-scale scope = the whole [K, N] matrix of
 * an expert, so fused gate/up projections (concatenated along N) share one scale.
 * [Miles-zh, "逐 Token 激活值缩放": gate and up feed one fused GEMM and must share one FP32 scale,
 * enforced by quantizing the pair together; "移除额外的 BF16 权重副本": 1-D 1x16 weight layout.]
 *
 *   w    bf16 [experts, K, N] dense (Y = X W per expert).
 *   qT   [experts, N, K/2] packed codes.
 *   sfT  [experts, N, K/16] scales, or MMA layout of the stacked [experts*N, K/16] matrix.
 *   s_w  [experts] float32. Used as scratch between the kernels this call enqueues (it holds
 *        the running amax bits, then, for more than one expert, the scales with a work-split flag
 *        in the sign bit, until the last kernel writes the scales).
 * Requires K % 16 == 0, N % 8 == 0 and experts <= 65535. experts = 0 is a no-op.
 */
nvq_status nvfp4_quantize_weights(const void* w, int64_t experts, int64_t k, int64_t n,
                                  uint8_t* qT, uint8_t* sfT, float* s_w,
                                  nvq_sf_layout sf_layout, void* stream);

/*
 * dequantize_bf16 — BF16 reconstruction of quantized operands for the dequantized-backward mode.
 *
 * Defines: out = RN_bf16(exact value), exact value = E4M3(q) * 2^(sf-127) (MXFP8) or
 * E2M1(q) * E4M3(sf) * s (NVFP4). [Miles-zh, "高精度反向和去量化反向": the dequantized backward runs
 * BF16 GEMMs on the BF16 dequantization of the exact low-precision forward operands.]
 *
 *   fmt     NVQ_MXFP8: q [groups*rows, cols] codes, sf scales of it, s ignored (may be NULL).
 *           NVQ_NVFP4: q [groups*rows, cols/2] packed, sf scales of it, s coarse scales:
 *           [groups*rows] for NVQ_SCOPE_ROW, [groups] for NVQ_SCOPE_MATRIX.
 *   out     bf16 [groups*rows, cols] (dense).
 * Requires cols % 32 == 0 (MXFP8) or % 16 == 0 (NVFP4).
 */
nvq_status dequantize_bf16(nvq_format fmt, const uint8_t* q, const uint8_t* sf, const float* s,
                           nvq_scope scope, int64_t groups, int64_t rows, int64_t cols,
                           nvq_sf_layout sf_layout, void* out, void* stream);

typedef enum {
    NVQ_GEMM_GROUP_M = 0,   /* rows of A are grouped by expert (forward, data gradient) */
    NVQ_GEMM_GROUP_K = 1    /* the reduction is grouped by expert (weight gradient) */
} nvq_gemm_mode;

typedef enum { NVQ_OUT_BF16 = 0, NVQ_OUT_F32 = 1 } nvq_out_type;

/*
 * sf_layout_convert — the explicit permutation between canonical scale bytes [rows, kb] and the
 * tcgen05 tile layout described above (both directions).
 *
 * Defines: a pure permutation (NVQ_SF_MMA output: padding bytes zero). [Miles-zh, "重构权重更新接口":
 * backend-specific swizzled layouts must stay explicit and verifiable, e.g. across a live weight
 * update.]
 *
 *   src, src_layout   scales [rows, kb] in that layout (nvq_sf_bytes(rows, kb*block, block, layout)).
 *   dst, dst_layout   the other layout; src_layout == dst_layout is rejected (NVQ_ERR_INVALID_ARG).
 * rows = 0 or kb = 0 is a no-op. src and dst must not overlap.
 */
nvq_status sf_layout_convert(const uint8_t* src, nvq_sf_layout src_layout, int64_t rows, int64_t kb,
                             uint8_t* dst, nvq_sf_layout dst_layout, void* stream);

/*
 * quantized_gather_rows — quantize-once dispatch: gather quantized rows (codes, block scales and,
 * for NVFP4, token scales) into a new row order, e.g. tokens into expert-sorted routed rows.
 *
 * Defines: row i of the outputs = row index[i] of the inputs, byte for byte; index[i] = -1 gives
 * a zero row (codes 0, scales 0, token scale 0 — what quantizing a zero padding row gives). Because
 * per-token NVFP4 and rowwise MXFP8 bytes depend on their own row only, gathering quantized tokens
 * equals quantizing the gathered bf16 rows. [Miles-zh, "逐 Token 激活值缩放": one FP32 scale per
 * token computed online, so the rollout can quantize once; per-token invariance.]
 *
 *   fmt         NVQ_NVFP4 (codes cols/2 bytes per row, scales cols/16, token scales) or NVQ_MXFP8
 *               (rowwise copy: codes cols bytes per row, scales cols/32; s and s_out ignored).
 *   q, sf, s    source rows [src_rows] (s: float32 [src_rows], NVFP4 only), sf in src_layout.
 *   index       device int32 [rows]; values in [-1, src_rows). An out-of-range value sets *status
 *               to NVQ_DEV_BAD_INDEX (when status is non-NULL) and that row is written as a zero row.
 *   q_out, sf_out, s_out  destination rows [rows], sf_out in dst_layout (MMA padding rows zeroed).
 * Requires cols % 16 (NVFP4) or % 32 (MXFP8) == 0. q, sf, q_out and sf_out 16-byte aligned; index,
 * s, s_out and status 4-byte aligned (NVQ_ERR_MISALIGNED otherwise). rows = 0 is a no-op.
 */
nvq_status quantized_gather_rows(nvq_format fmt, const uint8_t* q, const uint8_t* sf, const float* s,
                                 int64_t src_rows, int64_t cols, nvq_sf_layout src_layout,
                                 const int32_t* index, int64_t rows, uint8_t* q_out, uint8_t* sf_out,
                                 float* s_out, nvq_sf_layout dst_layout, int32_t* status, void* stream);

/* Device status word values written by block_scaled_grouped_gemm (when `status` is non-NULL). */
#define NVQ_DEV_OK 0
#define NVQ_DEV_TIMEOUT 1          /* a pipeline wait exceeded its time limit (wait_limit_ns) */
#define NVQ_DEV_BAD_OFFSETS 2      /* offsets not monotone, past the buffer, or (GROUP_K) not multiples of 32 */
#define NVQ_DEV_BAD_INDEX 3        /* quantized_gather_rows / nvfp4_quantize_dispatch: an index out of range */


typedef struct {
    nvq_format fmt;          /* NVQ_MXFP8 (E4M3 x E8M0 / 32), NVQ_NVFP4 (E2M1 x E4M3 / 16), NVQ_BF16 */
    nvq_gemm_mode mode;
    nvq_out_type out_type;   /* bf16 (round to nearest even) or float32                           */
    int64_t groups;          /* E: experts                                                        */
    int64_t m;               /* GROUP_M: rows of the A buffer; GROUP_K: rows of A = output rows    */
    int64_t n;               /* GROUP_M: rows of each B[e]; GROUP_K: rows of B; = output columns   */
    int64_t k;               /* GROUP_M: reduction length; GROUP_K: columns of A and of B          */
    const void* a;           /* [m, k] codes, K-major (NVFP4 packed: k/2 bytes per row; BF16: bf16) */
    const void* sfa;         /* scales of a in the MMA layout (ignored for NVQ_BF16)               */
    const float* s_a;        /* [m] per-row FP32 scales (NVFP4 tokens) or NULL (= 1)               */
    const void* b;           /* GROUP_M: [groups, n, k]; GROUP_K: [n, k]; codes, K-major           */
    const void* sfb;         /* scales of b (stacked rows) in the MMA layout (ignored for NVQ_BF16) */
    const float* s_b;        /* [groups] per-expert FP32 scales or NULL (= 1)                      */
    const int64_t* offsets;  /* device [groups+1]: group e owns rows (GROUP_M) or reduction columns
                                (GROUP_K) offsets[e] .. offsets[e+1]-1; offsets[0] = 0, monotone,
                                offsets[groups] <= m (GROUP_M) or <= k (GROUP_K); any row for
                                GROUP_M, multiples of 32 for GROUP_K (a 32-element block of the
                                reduction never straddles two groups)                         */
    void* d;                 /* GROUP_M: [m, n] rows of groups written, others untouched;
                                GROUP_K: [groups, m, n] (empty groups are written as zeros)        */
    int64_t ldd;             /* leading dimension of d in elements (>= n, multiple of 8)           */
    int32_t* status;         /* optional device int32: NVQ_DEV_* after the call (set, never cleared) */
    int64_t wait_limit_ns;   /* bound of each wait between the kernel's pipeline roles, in ns of
                                %globaltimer; 0 = 2 s. A wait that runs out sets *status to
                                NVQ_DEV_TIMEOUT; the kernel then drains its in-flight copies and
                                tensor-core work, frees its tensor memory and returns (the output
                                is then incomplete).                                              */
    int32_t inject_timeout_stage;  /* 0 = off. Fault injection for tests of that watchdog: k > 0
                                makes the first CTA's load stage k (1-based) never arrive, so the
                                waits on it run out and the call ends with NVQ_DEV_TIMEOUT.     */
} nvq_gemm_args;

/*
 * block_scaled_grouped_gemm — routed-expert GEMM on tcgen05 block-scaled tensor cores with fp32
 * accumulation and the per-token x per-expert FP32 scaling fused in the epilogue.
 *
 * Defines, with deq() = element value x its block scale (FP32 scales kept apart):
 *   GROUP_M: D[i, j] = s_a[i] * s_b[e] * sum_k deq(A)[i, k] * deq(B[e])[j, k],  offsets[e] <= i < offsets[e+1]
 *   GROUP_K: D[e][i, j] = sum_{offsets[e] <= k < offsets[e+1]} deq(A)[i, k] * deq(B)[j, k]
 * [Miles-zh, "方案 1": forward, weight-gradient and data-gradient GEMMs in MXFP8, blocks along the
 * reduction dimension; "结果": the per-token NVFP4 GEMM fuses the FP32 scaling into the kernel
 * epilogue; NVFP4-ru: block-scaled FP4 GEMMs run natively on Blackwell tensor cores.]
 * Accuracy: |D - D_exact| <= 2e-3 * sum_k |s_a s_b deq(A) deq(B)| before the output rounding.
 *
 * Requires: n % 128 == 0; GROUP_M: k % 128 == 0; GROUP_K: k % 32 == 0, m % 128 == 0,
 * fmt == NVQ_MXFP8 or NVQ_BF16 and s_a == NULL; groups <= 1024. offsets are validated on the device
 * (status NVQ_DEV_BAD_OFFSETS, nothing written). Scale buffers: sfa = MMA layout of [m, k/block],
 * sfb = MMA layout of the stacked [groups*n, k/block] (GROUP_M) or [n, k/block] (GROUP_K).
 *
 * fmt == NVQ_BF16: the same grouped GEMM on bf16 operands (a [m, k], b [groups*n, k] or [n, k],
 * k-major) with fp32 accumulation; sfa and sfb are ignored (may be NULL); k % 16 == 0 in both
 * modes. [Miles-zh, "高精度反向和去量化反向": the high-precision and the dequantized backward run BF16
 * GEMMs, the latter on the BF16 dequantization (dequantize_bf16) of the low-precision operands.]
 */
nvq_status block_scaled_grouped_gemm(const nvq_gemm_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NVQ_H */
