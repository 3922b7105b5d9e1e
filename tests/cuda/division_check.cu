// Checks the quantizer's fast division (div_markstein, nvq_device.cuh) against IEEE division
// (__fdiv_rn) for every pair of bf16 significands (g, both signs) and float32 significands (d), at
// the exponent pairs given on the command line ("eg:ed ..."). Prints one line per pair:
// "<eg> <ed> <mismatches> <covered> <total>"; a mismatch is a covered pair (ok) whose result differs.
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "../../nvfp4_quantization_block_gb300/csrc/nvq_device.cuh"

__global__ void check(int eg, int ed, unsigned long long* bad, unsigned long long* covered) {
    const uint32_t dm = blockIdx.x * blockDim.x + threadIdx.x;   // 23-bit significand of d
    if (dm >= (1u << 23)) return;
    const float d = __uint_as_float(((uint32_t)(127 + ed) << 23) | dm);
    unsigned long long b = 0, c = 0;
    for (uint32_t gm = 0; gm < 128; ++gm) {
        for (uint32_t sg = 0; sg < 2; ++sg) {
            const float g = __uint_as_float((sg << 31) | ((uint32_t)(127 + eg) << 23) | (gm << 16));
            bool ok;
            const float q = nvq::div_markstein(g, d, ok);
            if (!ok) continue;
            ++c;
            if (__float_as_uint(q) != __float_as_uint(__fdiv_rn(g, d))) ++b;
        }
    }
    if (b) atomicAdd(bad, b);
    if (c) atomicAdd(covered, c);
}

int main(int argc, char** argv) {
    unsigned long long *bad, *covered;
    if (cudaMalloc(&bad, 8) != cudaSuccess || cudaMalloc(&covered, 8) != cudaSuccess) return 2;
    for (int i = 1; i < argc; ++i) {
        int eg = 0, ed = 0;
        if (sscanf(argv[i], "%d:%d", &eg, &ed) != 2 || eg < -126 || eg > 127 || ed < 0 || ed > 125) return 3;
        cudaMemset(bad, 0, 8);
        cudaMemset(covered, 0, 8);
        check<<<(1 << 23) / 256, 256>>>(eg, ed, bad, covered);
        if (cudaDeviceSynchronize() != cudaSuccess) return 4;
        unsigned long long hb = 0, hc = 0;
        cudaMemcpy(&hb, bad, 8, cudaMemcpyDeviceToHost);
        cudaMemcpy(&hc, covered, 8, cudaMemcpyDeviceToHost);
        printf("%d %d %llu %llu %llu\n", eg, ed, hb, hc, (1ull << 23) * 256);
    }
    return 0;
}
