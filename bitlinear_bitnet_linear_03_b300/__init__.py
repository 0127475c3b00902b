"""BitNet b1.58 BitLinear hot path for B300 (sm_103a): a thin ctypes binding
over the CUDA library libbitnet_b300.so (see include/bitnet_b300.h)."""
