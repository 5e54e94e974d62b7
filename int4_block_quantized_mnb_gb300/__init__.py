"""int4 block-quantized MatMulNBits decode GEMV for GB300 (sm_103a)."""
