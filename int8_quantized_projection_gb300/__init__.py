"""GB300-native int8 quantized projection: q8_0 activation quantization (standalone or
fused into RMSNorm / SwiGLU) feeding a batch-1 Q8_0 GEMV and a prefill Q8_0 GEMM.

The compute is in ``libq8proj.so`` (hand-written CUDA for sm_103a, C ABI in
``include/q8proj.h``); this package only builds it and binds it.  Importing
the package does not load the library; the first call does, and fails loudly
if it was not built.
"""
from ._binding import (  # noqa: F401
    Bound,
    Q8Error,
    empty_plane,
    gemm_workspace,
    lib,
    library_path,
    load,
    q8_0_gemm,
    q8_0_gemm_mma,
    q8_0_gemm_noalloc,
    q8_0_gemm_prepare_weights,
    q8_0_gemm_prepared,
    q8_0_gemm_prepared_weights_bytes,
    q8_0_gemm_prepared_workspace_bytes,
    q8_0_gemm_workspace_bytes,
    q8_0_gemv,
    q8_0_gemv_grouped,
    q8_0_gemv_fused,
    q8_0_gemv_gate_up,
    q8_0_gemv_batched,
    q8_0_gemv_batched_grouped,
    PRODUCER_QUANT,
    PRODUCER_RMSNORM,
    PRODUCER_SWIGLU,
    q4a_gemv,
    q4a_gemv_batched,
    q4a_gemv_batched_grouped,
    GEMV_MAX_TOKENS,
    q8_check,
    q8_num_sms,
    q8_plane_rows,
    quantize_q8_0,
    rmsnorm_quant,
    swiglu_quant,
)
