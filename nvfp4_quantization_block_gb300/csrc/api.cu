// C-ABI entry points (include/nvq.h): argument validation on the host, then kernel launches.
// Nothing here allocates, frees or synchronises.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/nvq.h"
#include "nvq_internal.h"

namespace nvq {
static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace nvq

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline nvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVQ_OK : NVQ_ERR_CUDA; }

inline bool valid_layout(nvq_sf_layout l) { return l == NVQ_SF_CANONICAL || l == NVQ_SF_MMA; }

// per-token quantizers: block counts per row fit an int, and the grid (4 rows per CTA) fits its x limit
constexpr int64_t NVQ_TOKEN_MAX_COLS = int64_t(1) << 30;
constexpr int64_t NVQ_TOKEN_MAX_ROWS = int64_t(1) << 32;

}  // namespace

extern "C" {

const char* nvq_status_string(nvq_status s) {
    switch (s) {
        case NVQ_OK: return "NVQ_OK";
        case NVQ_ERR_INVALID_ARG: return "NVQ_ERR_INVALID_ARG";
        case NVQ_ERR_MISALIGNED: return "NVQ_ERR_MISALIGNED";
        case NVQ_ERR_UNSUPPORTED: return "NVQ_ERR_UNSUPPORTED";
        case NVQ_ERR_CUDA: return "NVQ_ERR_CUDA";
        case NVQ_ERR_TIMEOUT: return "NVQ_ERR_TIMEOUT";
    }
    return "NVQ_ERR_UNKNOWN";
}

uint64_t nvq_launch_count(void) { return nvq::g_launches.load(std::memory_order_relaxed); }

int64_t nvq_sf_bytes(int64_t rows, int64_t cols, int32_t block, nvq_sf_layout layout) {
    if (rows < 0 || cols < 0 || (block != 16 && block != 32) || cols % block || !valid_layout(layout))
        return -1;
    const int64_t kb = cols / block;
    if (layout == NVQ_SF_CANONICAL) return rows * kb;
    return ((rows + 127) / 128 * 128) * ((kb + 3) / 4 * 4);
}

nvq_status mxfp8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q_row,
                          uint8_t* sf_row, uint8_t* q_colT, uint8_t* sf_colT, nvq_sf_layout sf_layout,
                          void* stream) {
    if (rows < 0 || cols < 0 || !valid_layout(sf_layout)) return NVQ_ERR_INVALID_ARG;
    if ((q_row == nullptr) != (sf_row == nullptr) || (q_colT == nullptr) != (sf_colT == nullptr))
        return NVQ_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0 || (q_row == nullptr && q_colT == nullptr)) return NVQ_OK;
    if (x == nullptr || cols % 32 || ldx < cols) return NVQ_ERR_INVALID_ARG;
    if (q_colT != nullptr && rows % 32) return NVQ_ERR_INVALID_ARG;
    if (rows > (int64_t)65535 * 128) return NVQ_ERR_INVALID_ARG;
    if (!aligned16(x) || ldx % 8) return NVQ_ERR_MISALIGNED;
    if ((q_row && !aligned16(q_row)) || (q_colT && !aligned16(q_colT))) return NVQ_ERR_MISALIGNED;
    if ((sf_row && !aligned16(sf_row)) || (sf_colT && !aligned16(sf_colT))) return NVQ_ERR_MISALIGNED;
    return from_cuda(nvq::launch_mxfp8_quantize(static_cast<const uint16_t*>(x), rows, cols, ldx, q_row,
                                                sf_row, q_colT, sf_colT, sf_layout == NVQ_SF_MMA,
                                                static_cast<cudaStream_t>(stream)));
}

nvq_status nvfp4_quantize_per_token(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                    uint8_t* sf, float* s_tok, nvq_sf_layout sf_layout, void* stream) {
    if (rows < 0 || cols < 0 || !valid_layout(sf_layout)) return NVQ_ERR_INVALID_ARG;
    if (rows == 0) return NVQ_OK;
    if (x == nullptr || q == nullptr || sf == nullptr || s_tok == nullptr) return NVQ_ERR_INVALID_ARG;
    if (cols == 0 || cols % 16 || ldx < cols) return NVQ_ERR_INVALID_ARG;
    if (cols > NVQ_TOKEN_MAX_COLS || rows > NVQ_TOKEN_MAX_ROWS) return NVQ_ERR_INVALID_ARG;
    if (!aligned16(x) || ldx % 8 || !aligned16(q) || !aligned16(sf) || !aligned16(s_tok))
        return NVQ_ERR_MISALIGNED;
    return from_cuda(nvq::launch_nvfp4_quantize_per_token(static_cast<const uint16_t*>(x), rows, cols, ldx, q,
                                                          sf, s_tok, sf_layout == NVQ_SF_MMA,
                                                          static_cast<cudaStream_t>(stream)));
}

nvq_status nvfp4_quantize_dispatch(const void* x, int64_t tokens, int64_t cols, int64_t ldx, const int32_t* dest,
                                   int32_t topk, int64_t rows, uint8_t* q, uint8_t* sf, float* s_tok,
                                   nvq_sf_layout sf_layout, int32_t* status, void* stream) {
    if (tokens < 0 || cols < 0 || rows < 0 || !valid_layout(sf_layout)) return NVQ_ERR_INVALID_ARG;
    if (topk < 1 || topk > 32) return NVQ_ERR_INVALID_ARG;
    if (tokens == 0 && rows == 0) return NVQ_OK;
    if (cols == 0 || cols % 16 || cols > 16384 || ldx < cols) return NVQ_ERR_INVALID_ARG;
    if (tokens > NVQ_TOKEN_MAX_ROWS || rows > ((int64_t)1 << 31) - 1) return NVQ_ERR_INVALID_ARG;
    if (q == nullptr || sf == nullptr || s_tok == nullptr || (tokens > 0 && (x == nullptr || dest == nullptr)))
        return NVQ_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || ldx % 8 || !aligned16(q) || !aligned16(sf) || !aligned4(s_tok) ||
        (dest && !aligned4(dest)) || (status && !aligned4(status)))
        return NVQ_ERR_MISALIGNED;
    return from_cuda(nvq::launch_nvfp4_quantize_dispatch(static_cast<const uint16_t*>(x), tokens, cols, ldx, dest, topk,
                                                         rows, q, sf, s_tok, sf_layout == NVQ_SF_MMA, status,
                                                         static_cast<cudaStream_t>(stream)));
}

nvq_status nvfp4_swiglu_quantize_per_token(const void* gate_up, int64_t rows, int64_t cols, int64_t ld,
                                           uint8_t* q, uint8_t* sf, float* s_tok, nvq_sf_layout sf_layout,
                                           void* stream) {
    if (rows < 0 || cols < 0 || !valid_layout(sf_layout)) return NVQ_ERR_INVALID_ARG;
    if (rows == 0) return NVQ_OK;
    if (gate_up == nullptr || q == nullptr || sf == nullptr || s_tok == nullptr) return NVQ_ERR_INVALID_ARG;
    if (cols == 0 || cols % 16 || ld < 2 * cols) return NVQ_ERR_INVALID_ARG;
    if (cols > NVQ_TOKEN_MAX_COLS || rows > NVQ_TOKEN_MAX_ROWS) return NVQ_ERR_INVALID_ARG;
    if (!aligned16(gate_up) || ld % 8 || !aligned16(q) || !aligned16(sf) || !aligned16(s_tok))
        return NVQ_ERR_MISALIGNED;
    return from_cuda(nvq::launch_nvfp4_swiglu_quantize(static_cast<const uint16_t*>(gate_up), rows, cols, ld, q, sf,
                                                       s_tok, sf_layout == NVQ_SF_MMA,
                                                       static_cast<cudaStream_t>(stream)));
}

nvq_status nvfp4_quantize_weights(const void* w, int64_t experts, int64_t k, int64_t n, uint8_t* qT,
                                  uint8_t* sfT, float* s_w, nvq_sf_layout sf_layout, void* stream) {
    if (experts < 0 || k < 0 || n < 0 || !valid_layout(sf_layout)) return NVQ_ERR_INVALID_ARG;
    if (experts == 0) return NVQ_OK;
    if (w == nullptr || qT == nullptr || sfT == nullptr || s_w == nullptr) return NVQ_ERR_INVALID_ARG;
    if (k == 0 || n == 0 || k % 16 || n % 8 || experts > 65535) return NVQ_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(qT) || !aligned16(sfT) || !aligned16(s_w)) return NVQ_ERR_MISALIGNED;
    return from_cuda(nvq::launch_nvfp4_quantize_weights(static_cast<const uint16_t*>(w), experts, k, n, qT, sfT,
                                                        s_w, sf_layout == NVQ_SF_MMA,
                                                        static_cast<cudaStream_t>(stream)));
}

nvq_status sf_layout_convert(const uint8_t* src, nvq_sf_layout src_layout, int64_t rows, int64_t kb, uint8_t* dst,
                             nvq_sf_layout dst_layout, void* stream) {
    if (!valid_layout(src_layout) || !valid_layout(dst_layout) || src_layout == dst_layout) return NVQ_ERR_INVALID_ARG;
    if (rows < 0 || kb < 0) return NVQ_ERR_INVALID_ARG;
    if (rows == 0 || kb == 0) return NVQ_OK;
    if (src == nullptr || dst == nullptr) return NVQ_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return NVQ_ERR_MISALIGNED;
    return from_cuda(nvq::launch_sf_layout_convert(src, dst_layout == NVQ_SF_MMA, rows, kb, dst,
                                                   static_cast<cudaStream_t>(stream)));
}

nvq_status quantized_gather_rows(nvq_format fmt, const uint8_t* q, const uint8_t* sf, const float* s,
                                 int64_t src_rows, int64_t cols, nvq_sf_layout src_layout, const int32_t* index,
                                 int64_t rows, uint8_t* q_out, uint8_t* sf_out, float* s_out,
                                 nvq_sf_layout dst_layout, int32_t* status, void* stream) {
    if ((fmt != NVQ_MXFP8 && fmt != NVQ_NVFP4) || !valid_layout(src_layout) || !valid_layout(dst_layout))
        return NVQ_ERR_INVALID_ARG;
    if (src_rows < 0 || cols < 0 || rows < 0) return NVQ_ERR_INVALID_ARG;
    if (rows == 0) return NVQ_OK;
    const int64_t block = fmt == NVQ_NVFP4 ? 16 : 32;
    if (cols == 0 || cols % block || q_out == nullptr || sf_out == nullptr || index == nullptr)
        return NVQ_ERR_INVALID_ARG;
    if (src_rows > 0 && (q == nullptr || sf == nullptr)) return NVQ_ERR_INVALID_ARG;
    if (fmt == NVQ_NVFP4 && (s_out == nullptr || (src_rows > 0 && s == nullptr))) return NVQ_ERR_INVALID_ARG;
    if ((q && !aligned16(q)) || (sf && !aligned16(sf)) || !aligned16(q_out) || !aligned16(sf_out))
        return NVQ_ERR_MISALIGNED;
    // 32-bit words the kernel reads or writes as such
    if (!aligned4(index) || (status && !aligned4(status)) ||
        (fmt == NVQ_NVFP4 && ((s && !aligned4(s)) || !aligned4(s_out))))
        return NVQ_ERR_MISALIGNED;
    const int64_t qbytes = fmt == NVQ_NVFP4 ? cols / 2 : cols;
    return from_cuda(nvq::launch_quantized_gather_rows(q, sf, fmt == NVQ_NVFP4 ? s : nullptr, src_rows, qbytes,
                                                       cols / block, src_layout == NVQ_SF_MMA, index, rows, q_out,
                                                       sf_out, fmt == NVQ_NVFP4 ? s_out : nullptr,
                                                       dst_layout == NVQ_SF_MMA, status,
                                                       static_cast<cudaStream_t>(stream)));
}

nvq_status dequantize_bf16(nvq_format fmt, const uint8_t* q, const uint8_t* sf, const float* s,
                           nvq_scope scope, int64_t groups, int64_t rows, int64_t cols,
                           nvq_sf_layout sf_layout, void* out, void* stream) {
    if ((fmt != NVQ_MXFP8 && fmt != NVQ_NVFP4) || !valid_layout(sf_layout)) return NVQ_ERR_INVALID_ARG;
    if (scope != NVQ_SCOPE_ROW && scope != NVQ_SCOPE_MATRIX) return NVQ_ERR_INVALID_ARG;
    if (groups < 0 || rows < 0 || cols < 0) return NVQ_ERR_INVALID_ARG;
    if (groups == 0 || rows == 0 || cols == 0) return NVQ_OK;
    if (q == nullptr || sf == nullptr || out == nullptr) return NVQ_ERR_INVALID_ARG;
    if (fmt == NVQ_MXFP8 && cols % 32) return NVQ_ERR_INVALID_ARG;
    if (fmt == NVQ_NVFP4 && (cols % 16 || s == nullptr)) return NVQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || (s && !aligned16(s))) return NVQ_ERR_MISALIGNED;
    return from_cuda(nvq::launch_dequantize_bf16(fmt == NVQ_NVFP4, q, sf, s, scope == NVQ_SCOPE_MATRIX, groups,
                                                 rows, cols, sf_layout == NVQ_SF_MMA,
                                                 static_cast<uint16_t*>(out), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
