"""GB300 (sm_103a) dense GEMM library: C = alpha*A*op(B) + beta*C.

The compute runs in the CUDA kernels of libdgemm_sm103a.so; this package is
the ctypes binding (same names as the C ABI in include/dgemm.h), the nvcc
build step and the seeded synthetic-input generators.  PyTorch is used only
for device memory and streams.
"""
from ._lib import (  # noqa: F401
    DG_ERR_CUDA, DG_ERR_INVALID_ARG, DG_ERR_MISALIGNED, DG_ERR_NO_MEMORY, DG_ERR_TIMEOUT,
    DG_ERR_UNSUPPORTED, DG_KERNEL_NONE, DG_KERNEL_SCALE, DG_KERNEL_SIMT_F32, DG_KERNEL_THIN_BF16,
    DG_KERNEL_TC_BF16, DG_KERNEL_TC2_BF16, DG_OK, DG_OP_N, DG_OP_T, DG_OUT_BF16, DG_OUT_F32, EXPORTED, DgError,
    dg_device_status, dg_model_local_bytes, dg_model_quant_traffic_bytes, dg_model_traffic_bytes, dg_plan_gemm, dg_raster_tile,
    dg_release_workspace, dg_set_fault_injection, dg_status_string, dg_streamk_start, dg_version,
    attention_bf16, gemm_bf16, gemm_bf16_decode_chain, gemm_bf16_decode_noalloc, gemm_bf16_gate_up_silu, gemm_bf16_strided_batched, gemm_f32, gemm_fp8_e4m3, quantize_rows_e4m3, gemm_f32_strided_batched, library_path, load,
    status_string,
)
