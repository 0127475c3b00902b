// decode_chain.cuh — host interface of the persistent decode chain
// (decode_chain.cu); the public calls are in include/bitnet_b300.h.
#pragma once
#include <cuda_runtime.h>

#include "../../include/bitnet_b300.h"

namespace bitnet {

// Checks a chain description on the host (shapes, overlaps, links; no device
// call) and gives the table size it needs (0 unless BITNET_OK).
bitnet_status check_decode_chain(const bitnet_decode_phase* phases, int nphases, int64_t M,
                                 size_t* table_bytes);
// Checks the description (shapes, pointers, overlaps, links), lays out and
// fills the table.  BITNET_ERR_CUDA sets *cuda_err.
bitnet_status build_decode_chain(const bitnet_decode_phase* phases, int nphases, int64_t M,
                                 void* table, size_t table_bytes, bitnet_decode_chain* chain,
                                 cudaError_t* cuda_err);
cudaError_t launch_decode_chain(const bitnet_decode_chain* chain, long long wait_cycles,
                                cudaStream_t s);

}  // namespace bitnet
