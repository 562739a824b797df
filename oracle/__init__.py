"""fp64 CPU oracle for the small-M affine-quantized matmul (test infrastructure only)."""
