"""qk: quantize-once activation images for GB300 (sm_103a)."""
