"""BitNet b1.58 BitLinear hot path for B300 (sm_103a): a thin ctypes binding
over the CUDA library libbitnet_b300.so (include/bitnet_b300.h)."""
from ._lib import (BitnetError, bitnet_decode_chain_build, bitnet_decode_chain_run,
                   bitnet_device_error, bitnet_ffn, bitnet_ffn_workspace,
                   bitnet_linear, bitnet_linear_bf16, bitnet_linear_lut, bitnet_linear_workspace,
                   bitnet_quantize_act, bitnet_quantize_weights, bitnet_quantize_weights_noalloc,
                   bitnet_quantize_weights_workspace, bitnet_set_wait_limit, lib, library_path)

__all__ = ["BitnetError", "bitnet_decode_chain_build", "bitnet_decode_chain_run",
           "bitnet_device_error", "bitnet_ffn", "bitnet_ffn_workspace",
           "bitnet_linear", "bitnet_linear_bf16", "bitnet_linear_lut", "bitnet_linear_workspace",
           "bitnet_quantize_act",
           "bitnet_quantize_weights", "bitnet_quantize_weights_noalloc",
           "bitnet_quantize_weights_workspace", "bitnet_set_wait_limit", "lib", "library_path"]
