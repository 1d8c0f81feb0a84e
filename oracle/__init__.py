"""fp64 CPU oracle of the FlashAttention backward pass (test infrastructure only)."""
