"""CPU oracle for the MXFP8 / per-token NVFP4 quantizer contract and the block-scaled GEMM.

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, obviously-correct definition that
the CUDA kernels are checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The product path
(the C-ABI library and its Python binding) never imports, links or executes anything here, and
nothing here imports the product path. The two share no code; the only module both sides use is
``workloads`` (seeded synthetic inputs, which holds none of the method's arithmetic).

Arithmetic is numpy float64 plus exact rational reasoning: every rounding step is a single
rounding of an exactly computed (or provably exactly decidable) real value, as the pages'
bit-exact contract requires. Each function cites the passage it follows.

Sources cited (page titles; each page is a translation of the same Miles/LMSYS post unless noted):
  [Miles-zh]  "Miles 在 Blackwell GPU 上实现低精度强化学习，降低训练成本" (Chinese translation of the
              Miles post "Towards Blackwell-native 8-bit and 4-bit RL").
  [Miles-fr]  "Miles Blackwell remplace l'uniformité BF16 par MXFP8 et NVFP4 natifs".
  [Miles-vi]  "Miles tối ưu hóa học tăng cường trên kiến trúc Blackwell với MXFP8 và NVFP4".
  [NVFP4-ru]  "NVIDIA верифицировала 4-битный формат NVFP4 на Mamba-Transformer (12B) при 10 трлн
              токенов" (summary of NVIDIA's NVFP4 pretraining paper).

Pinning status of each function is stated in its docstring; every function here is pinned by
tests under ``tests/test_oracle_*.py`` (hand-worked blocks, closed forms, exhaustive exact-rational
brute force, library routines, invariants) except where a docstring says "parity unpinned".
"""

from .formats import (  # noqa: F401
    E4M3_VALUES, E2M1_VALUES, E4M3_MAX, E2M1_MAX,
    bf16_bits_to_f64, f64_to_bf16_bits_rne, round_to_e4m3, round_to_e2m1,
    e8m0_exponent, e4m3_decode, e2m1_decode, e8m0_decode,
)
from .quant import (  # noqa: F401
    mxfp8_quantize, mxfp8_quantize_blocks, nvfp4_quantize_per_token, nvfp4_quantize_weights,
    nvfp4_quantize_rows, dequantize_mxfp8, dequantize_nvfp4, nvfp4_token_scale,
    unpack_e2m1, pack_e2m1,
)
from .layout import sf_to_mma_layout, sf_from_mma_layout, mma_layout_offset, mma_layout_bytes  # noqa: F401
from .gemm import grouped_gemm_reference, grouped_gemm_entries, deq_operand  # noqa: F401
from .swiglu import exp_f32, exp_parts, swiglu_f32, swiglu_bf16_bits, swiglu_rows  # noqa: F401
