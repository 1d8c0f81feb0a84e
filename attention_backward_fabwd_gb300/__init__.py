"""libfabwd: FlashAttention backward pass for GB300 (sm_103a).

The compute path is the C-ABI library libfabwd (hand-written CUDA); this package holds its
ctypes binding (argument marshalling only), a torch-facing convenience call and the seeded
synthetic input generators.
"""
