"""CPU oracle for the quantize-once activation path (test infrastructure only)."""
