"""GB300 (sm_103a) weight-only-quantized skinny matmul: Q8_1 activation quantizer,
Q4_0 and Q4_K x Q8_1 MMVQ at M = 1..8, NVFP4 W4A16 and FP8 W8A16 at M = 1..96 (one
weight pass per chunk of at most 16 rows).

The compute lives in the C-ABI CUDA library ``_build/libqmv.so`` (declared in
``include/qmv.h``); this package is its thin Python binding. Seeded synthetic
inputs are in ``gemm_qmv_quantize_gb300.synth``.
"""
from ._binding import (QmvError, QmvLibraryMissing, error_flags, get_launch_overlap, lib, library_path,
                       qgemm_fp8_w8a16, qgemm_fp8_w8a16_group, qgemm_nvfp4_w4a16_group, set_launch_overlap,
                       qgemm_nvfp4_w4a16, qmv_debug_q4_0_block_dots, qmv_q4_0_q8_1,
                       qmv_q4_0_q8_1_fused, qmv_q4_0_q8_1_fused_group, qmv_q4_0_q8_1_group, qmv_quantize_q8_1,
                       qmv_debug_q4_k_block_dots, qmv_q4_k_q8_1, qmv_q4_k_q8_1_fused, qmv_q4_k_q8_1_fused_group,
                       qmv_q4_k_q8_1_group, qmv_debug_wait_bound, qmv_debug_cta_abort, qmv_debug_plan_q4, qmv_debug_plan_wq,
                       route_counts, route_reset)

__all__ = ["QmvError", "QmvLibraryMissing", "error_flags", "get_launch_overlap", "set_launch_overlap", "lib", "library_path", "qgemm_fp8_w8a16", "qgemm_fp8_w8a16_group", "qgemm_nvfp4_w4a16_group",
           "qgemm_nvfp4_w4a16", "qmv_debug_q4_0_block_dots", "qmv_q4_0_q8_1", "qmv_q4_0_q8_1_fused", "qmv_q4_0_q8_1_fused_group", "qmv_q4_0_q8_1_group", "qmv_quantize_q8_1",
           "qmv_debug_q4_k_block_dots", "qmv_q4_k_q8_1", "qmv_q4_k_q8_1_fused", "qmv_q4_k_q8_1_fused_group",
           "qmv_q4_k_q8_1_group", "qmv_debug_wait_bound", "qmv_debug_cta_abort", "qmv_debug_plan_q4", "qmv_debug_plan_wq", "route_counts", "route_reset"]
