// Internal launch functions behind the C-ABI (include/nvq.h). Each enqueues kernels on `stream`
// and returns the launch status; argument checking happens in api.cu before any of these runs.
#pragma once
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace nvq {

// Launch with programmatic stream serialization: the kernel may be scheduled while the kernel
// before it in the stream is still finishing (its last CTAs), which hides the launch gap between
// dependent kernels. Every kernel of this library starts with griddep_begin() (nvq_device.cuh):
// griddepcontrol.wait, so it touches no global memory before its predecessor has completed and
// its writes are visible.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_mxfp8_quantize(const uint16_t* x, int64_t R, int64_t C, int64_t ldx,
                                  uint8_t* q_row, uint8_t* sf_row, uint8_t* q_colT, uint8_t* sf_colT,
                                  int mma_layout, cudaStream_t stream);

cudaError_t launch_nvfp4_quantize_per_token(const uint16_t* x, int64_t R, int64_t C, int64_t ldx,
                                            uint8_t* q, uint8_t* sf, float* s_tok, int mma_layout,
                                            cudaStream_t stream);

cudaError_t launch_nvfp4_quantize_dispatch(const uint16_t* x, int64_t T, int64_t C, int64_t ldx, const int32_t* dest,
                                           int topk, int64_t R, uint8_t* q, uint8_t* sf, float* s_tok, int mma_layout,
                                           int32_t* status, cudaStream_t stream);

cudaError_t launch_nvfp4_swiglu_quantize(const uint16_t* gate_up, int64_t R, int64_t I, int64_t ld, uint8_t* q,
                                         uint8_t* sf, float* s_tok, int mma_layout, cudaStream_t stream);

cudaError_t launch_nvfp4_quantize_weights(const uint16_t* w, int64_t E, int64_t K, int64_t N,
                                          uint8_t* qT, uint8_t* sfT, float* s_w, int mma_layout,
                                          cudaStream_t stream);

cudaError_t launch_dequantize_bf16(int fmt_nvfp4, const uint8_t* q, const uint8_t* sf, const float* s,
                                   int scope_matrix, int64_t groups, int64_t rows, int64_t cols,
                                   int mma_layout, uint16_t* out, cudaStream_t stream);

cudaError_t launch_sf_layout_convert(const uint8_t* src, int to_mma, int64_t rows, int64_t kb, uint8_t* dst,
                                     cudaStream_t stream);

cudaError_t launch_quantized_gather_rows(const uint8_t* q, const uint8_t* sf, const float* s, int64_t src_rows,
                                         int64_t qbytes, int64_t kb, int src_mma, const int32_t* index, int64_t rows,
                                         uint8_t* q_out, uint8_t* sf_out, float* s_out, int dst_mma,
                                         int32_t* status, cudaStream_t stream);

// Host-side count of kernels this library has enqueued (diagnostics; see nvq_launch_count).
void count_launches(int n);
}  // namespace nvq
