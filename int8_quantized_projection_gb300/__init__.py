"""GB300-native int8 quantized projection (q8_0 activation quantize -> Q8_0 GEMV / GEMM)."""
