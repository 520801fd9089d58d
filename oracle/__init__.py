"""FP64 CPU oracle for HSTU jagged attention (test infrastructure only)."""
