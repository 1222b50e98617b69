"""GB300-native dense GEMM: C = alpha * op(A) * op(B) + beta * C + bias.

The compute runs in hand-written sm_103a CUDA (TMA loads into a shared-memory
ring, tcgen05 MMAs accumulating in tensor memory, warp-specialised epilogue)
behind a C ABI (``include/gemm.h``); ``gemm`` is the thin ctypes binding.
"""
