// gemm_tc.cu — tensor-core BitLinear (prefill).  Placeholder until the
// tcgen05 kernel lands: no shape is eligible, so every call runs on CUDA cores.
#include "gemm_tc.cuh"

namespace bitnet {

__device__ int g_device_error;

bool gemm_tc_eligible(int64_t, int64_t, int64_t) { return false; }
size_t gemm_tc_workspace(int64_t, int64_t, int64_t) { return 0; }
cudaError_t launch_gemm_tc(const uint8_t*, const float*, const int8_t*, const float*, int64_t,
                           int64_t, int64_t, float*, int32_t*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t read_and_clear_device_error(int* code, cudaStream_t s) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_device_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e;
}

}  // namespace bitnet
