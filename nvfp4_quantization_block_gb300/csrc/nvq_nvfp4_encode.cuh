// One NVFP4 block encoded in one of the three decision modes; shared by the per-token and the
// expert-weight quantizers (quant_nvfp4.cu, quant_nvfp4_weights.cu). The decisions themselves
// (block scale, boundaries, product-path multiplier) are defined in nvq_device.cuh.
#pragma once

#include "nvq_device.cuh"

namespace nvq {

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

}  // namespace nvq
