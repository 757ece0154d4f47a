"""Sub-bit (binary / ternary) weight products on NVIDIA B300 (sm_103a)."""
