// gemm_tc.cuh — the tensor-core BitLinear for prefill-sized M (gemm_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bitnet {

// True when (M, N, K) runs on the tensor-core kernel rather than on CUDA cores.
bool gemm_tc_eligible(int64_t M, int64_t N, int64_t K);
size_t gemm_tc_workspace(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_tc(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                           const float* x_scale, int64_t M, int64_t N, int64_t K, float* y,
                           uint16_t* y_bf16, int32_t* acc_out, void* ws, long long wait,
                           cudaStream_t s);

// The FFN's up and gate products of the same activations in one GEMM
// (M > 256): u = BitLinear(Wu), v = BitLinear(Wg), h = relu(v)^2 * u, all
// [M, N] binary32; u and v are optional outputs, h is required.  hmax
// (optional, [M] words, 16-byte aligned, room for a multiple of 4): each
// row's max |h| as binary32 bits, for gemm_tc_from_f32.
size_t gemm_tc_gated_workspace(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_tc_gated(const uint8_t* Wu, const float* su, const uint8_t* Wg,
                                 const float* sg, const int8_t* xq, const float* x_scale,
                                 int64_t M, int64_t N, int64_t K, float* u, float* v, float* h,
                                 unsigned* hmax, void* ws, long long wait, cudaStream_t s);

// BitLinear of binary32 activation rows h [M, K] (the FFN's h before the
// down projection) whose row maxima hmax the gated GEMM wrote: the
// pre-pass quantises h per token (the rule of the activation quantiser)
// straight into the GEMM's digit operand, writes the scales sh [M] and,
// when hq is not null, the int8 codes.  Supported when
// gemm_tc_from_f32_supported(M, K); the workspace is gemm_tc_workspace.
bool gemm_tc_from_f32_supported(int64_t M, int64_t K);
cudaError_t launch_gemm_tc_from_f32(const uint8_t* Wq, const float* w_scale, const float* h,
                                    const unsigned* hmax, int64_t M, int64_t N, int64_t K,
                                    float* y, uint16_t* y_bf16, int32_t* acc_out, int8_t* hq,
                                    float* sh, void* ws, long long wait, cudaStream_t s);

// Reads and clears the per-device error word that bounded waits set.
cudaError_t read_and_clear_device_error(int* code, cudaStream_t s);

}  // namespace bitnet
