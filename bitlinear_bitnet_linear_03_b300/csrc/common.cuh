// common.cuh — device helpers and the launch functions shared by the
// library's translation units.  Everything here is internal: the public
// interface is include/bitnet_b300.h.
//
// Floating-point rule for the whole library: every binary32 / binary64 step
// that decides a stored value is written with an explicit round-to-nearest
// intrinsic (__fmul_rn, __fdiv_rn, __dadd_rn, ...), and the library is built
// with -fmad=false, so no multiply-add is ever contracted.  Integer work
// (codes, dot products, partial sums) is exact by construction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bitnet {

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// 16-byte streaming load that is not kept in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Read-only 16-byte load (may be cached).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// acc + sum_t a.byte[t] * b.byte[t], a unsigned bytes, b signed bytes.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int acc) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(acc));
  return d;
}

// acc + sum_t a.byte[t] * b.byte[t], both signed bytes.
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int acc) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(acc));
  return d;
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialisation attribute may start before its predecessor in the
// stream has finished; griddep_wait() blocks until that predecessor's memory
// operations are complete and visible, so every kernel of this library calls
// it before reading or writing anything the predecessor may touch.
// griddep_launch_dependents() lets the successor start launching early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Asks the copy engine to bring [p, p + bytes) into L2 (a hint: no data is
// returned and nothing is written).  p and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ int warp_sum_i32(int v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Largest of the lanes' values; fmaxf keeps a non-NaN operand, so a NaN
// entry never becomes the maximum.
__device__ __forceinline__ float warp_max_f32(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// round-half-even of v, clipped to [lo, hi]; NaN gives 0.
__device__ __forceinline__ int round_clip(float v, float lo, float hi) {
  if (v != v) return 0;
  float r = rintf(v);
  r = fminf(fmaxf(r, lo), hi);
  return (int)r;
}

// round_clip(v, -128, 127) with full-rate float and integer operations only
// (the float-to-integer conversion units run at a fraction of that rate):
// clip (NaN to 0), then add 1.5 * 2^23.  The sum lies in [2^23, 2^24), where
// the unit in the last place is 1, so the addition's own rounding (to nearest,
// ties to even) leaves round-half-even of the clipped value in its low bits.
__device__ __forceinline__ int quant_i8(float v) {
  float c = fminf(fmaxf(v, -128.0f), 127.0f);
  c = v == v ? c : 0.0f;
  return __float_as_int(__fadd_rn(c, 12582912.0f)) - 0x4B400000;
}

// Per-token quantisation constants from the row's largest magnitude a:
// a' = max(a, 1e-5), inv = 127 / a', scale = a' / 127 (binary32 divisions).
struct ActScale {
  float inv;
  float scale;
};
__device__ __forceinline__ ActScale act_scale_from_absmax(float a) {
  float ap = a > 1e-5f ? a : 1e-5f;
  ActScale s;
  s.inv = __fdiv_rn(127.0f, ap);
  s.scale = __fdiv_rn(ap, 127.0f);
  return s;
}

// Nearest bf16 (ties to even) to a binary32 value, as its bit pattern.
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint32_t pack_i8x4(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) |
         ((uint32_t)(d & 0xff) << 24);
}

// ---------------------------------------------------------------- launchers
// Launches `kernel` on `s` with programmatic stream serialisation allowed, so
// it may overlap the tail of the previous kernel on the stream (the kernel
// itself calls griddep_wait() before touching dependent data).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Weight quantisation (absmean_weights.cu).
size_t quantize_weights_workspace(int64_t total);
cudaError_t launch_quantize_weights(const float* W, int64_t total, uint8_t* Wq, float* w_scale,
                                    void* ws, cudaStream_t s);

// The same, with its scratch in a device array of the library instead of a
// caller workspace (absmean_weights.cu); cudaErrorInvalidValue beyond the
// array's size.
size_t quantize_weights_noalloc_limit();
cudaError_t launch_quantize_weights_noalloc(const float* W, int64_t total, uint8_t* Wq,
                                            float* w_scale, cudaStream_t s);

// Activation quantisation (act_quant.cu).
cudaError_t launch_quantize_act_bf16(const uint16_t* x, int64_t M, int64_t K, int8_t* xq,
                                     float* x_scale, cudaStream_t s);
cudaError_t launch_quantize_act_f32(const float* x, int64_t M, int64_t K, int8_t* xq,
                                    float* x_scale, cudaStream_t s);
// subln RMSNorm followed by the per-token quantisation (act_quant.cu).
cudaError_t launch_rmsnorm_quant(const uint16_t* x, const float* g, float eps, int64_t M,
                                 int64_t H, int8_t* xq, float* x_scale, cudaStream_t s);
// h = relu(v)^2 * u followed by the per-token quantisation of h (act_quant.cu).
cudaError_t launch_relu2_quant(const float* u, const float* v, int64_t M, int64_t F, float* h,
                               int8_t* hq, float* h_scale, cudaStream_t s);

// One-token BitLinear with a table-lookup (variant 0) or dp4a (variant 1)
// inner product on one kernel skeleton (gemv_lut.cu); K <= kLutMaxK.
constexpr int64_t kLutMaxK = 12288;
cudaError_t launch_gemv_lut(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                            const float* x_scale, int64_t N, int64_t K, float* y,
                            int32_t* acc_out, int variant, cudaStream_t s);

// Decode BitLinear (M <= 4) on CUDA cores: one launch for up to
// kDecodeMaxTargets weight matrices sharing the same input, which is either
// int8 (xq, x_scale) or bf16 (quantised per token inside the kernel, bit for
// bit as launch_quantize_act_bf16).  Returns cudaErrorNotSupported when the
// shape is outside what the kernel handles (gemv_decode.cu).
constexpr int kDecodeMaxTargets = 8;
constexpr int kDecodeMaxM = 4;
struct DecodeTarget {
  const uint8_t* Wq;
  const float* w_scale;
  int64_t N;
  float* y;          // binary32 output, or null
  int32_t* acc_out;  // or null
  uint16_t* y_bf16;  // bf16 output (nearest, ties to even), or null
};
bool decode_supported(int64_t M, int64_t K);
cudaError_t launch_decode(const DecodeTarget* targets, int count, const int8_t* xq,
                          const float* x_scale, const uint16_t* x_bf16, int64_t M, int64_t K,
                          int8_t* xq_out, float* x_scale_out, bool weights_static,
                          long long wait_cycles, cudaStream_t s);
// Reads and clears the error word of the decode kernel's bounded waits.
cudaError_t read_and_clear_decode_error(int* code, cudaStream_t s);
// The same for decode chains (decode_chain.cu).
cudaError_t read_and_clear_chain_error(int* code, cudaStream_t s);

// Bound of the kernels' waits, in clocks (abi.cu; bitnet_set_wait_limit).
long long wait_limit_cycles();

// BitLinear on CUDA cores, any M (gemv.cu).
size_t gemv_workspace(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemv(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                        const float* x_scale, int64_t M, int64_t N, int64_t K, float* y,
                        uint16_t* y_bf16, int32_t* acc_out, void* ws, cudaStream_t s);

}  // namespace bitnet
