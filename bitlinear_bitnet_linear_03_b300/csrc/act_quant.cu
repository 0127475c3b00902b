// act_quant.cu — per-token absmax int8 activation quantisation and the two
// fused producers of quantised activations in the BitNet feed-forward block.
//
// "Microsoft BitNet b1.58 ... 1-bit AI model" (communeify), "Meet BitNet
// b1.58 2B4T": W1.58A8, i.e. 8-bit integer activations; the same page lists
// subln normalisation and the ReLU^2 activation.  "Microsoft BitNet: 100B
// models on CPU" (juejin), CPU-friendly matrix multiplication: INT8
// activations.  Per token (row):
//   a = max |x|, a' = max(a, 1e-5), inv = 127 / a',
//   q = clamp(round_half_even(x * inv), -128, 127), scale = a' / 127.
// The row maximum is exact whatever the order; every binary32 step is one
// explicitly rounded operation.
#include "common.cuh"
#include "exact_sumsq.cuh"

namespace bitnet {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max_f32(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

__global__ void __launch_bounds__(kThreads)
k_act_quant_bf16(const uint4* __restrict__ x, int K, uint2* __restrict__ xq,
                 float* __restrict__ x_scale) {
  __shared__ float red[kThreads / 32];
  const int row = blockIdx.x;
  const int nv = K >> 3;
  const uint4* xr = x + (int64_t)row * nv;
  float a = 0.0f;
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    uint4 p = xr[v];
    uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      a = fmaxf(a, fabsf(bf16_bits_to_float(w[j] & 0xffffu)));
      a = fmaxf(a, fabsf(bf16_bits_to_float(w[j] >> 16)));
    }
  }
  a = block_max(a, red);
  const ActScale sc = act_scale_from_absmax(a);
  if (threadIdx.x == 0) x_scale[row] = sc.scale;
  uint2* qr = xq + (int64_t)row * nv;
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    uint4 p = xr[v];
    uint32_t w[4] = {p.x, p.y, p.z, p.w};
    int q[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      q[2 * j] = round_clip(__fmul_rn(bf16_bits_to_float(w[j] & 0xffffu), sc.inv), -128.f, 127.f);
      q[2 * j + 1] = round_clip(__fmul_rn(bf16_bits_to_float(w[j] >> 16), sc.inv), -128.f, 127.f);
    }
    qr[v] = make_uint2(pack_i8x4(q[0], q[1], q[2], q[3]), pack_i8x4(q[4], q[5], q[6], q[7]));
  }
}

__global__ void __launch_bounds__(kThreads)
k_act_quant_f32(const float4* __restrict__ x, int K, uint32_t* __restrict__ xq,
                float* __restrict__ x_scale) {
  __shared__ float red[kThreads / 32];
  const int row = blockIdx.x;
  const int nv = K >> 2;
  const float4* xr = x + (int64_t)row * nv;
  float a = 0.0f;
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    float4 p = xr[v];
    a = fmaxf(fmaxf(fmaxf(a, fabsf(p.x)), fmaxf(fabsf(p.y), fabsf(p.z))), fabsf(p.w));
  }
  a = block_max(a, red);
  const ActScale sc = act_scale_from_absmax(a);
  if (threadIdx.x == 0) x_scale[row] = sc.scale;
  uint32_t* qr = xq + (int64_t)row * nv;
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    float4 p = xr[v];
    qr[v] = pack_i8x4(round_clip(__fmul_rn(p.x, sc.inv), -128.f, 127.f),
                      round_clip(__fmul_rn(p.y, sc.inv), -128.f, 127.f),
                      round_clip(__fmul_rn(p.z, sc.inv), -128.f, 127.f),
                      round_clip(__fmul_rn(p.w, sc.inv), -128.f, 127.f));
  }
}

// subln RMSNorm + quantisation, one warp per token.
//   ss = the exact sum of the binary32 squares x_k * x_k, rounded once to
//        binary32 (exact_sumsq.cuh: order-free, integer arithmetic);
//   r  = 1 / sqrt(ss / H + eps), four binary32 operations;
//   n  = (x * r) * g, then the per-token quantisation of n.
constexpr int kNormWarps = 8;
__global__ void __launch_bounds__(kNormWarps * 32)
k_rmsnorm_quant(const uint16_t* __restrict__ x, const float* __restrict__ g, float eps, int M,
                int H, int8_t* __restrict__ xq, float* __restrict__ x_scale) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kNormWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  const uint16_t* xr = x + (int64_t)row * H;
  sumsq::Acc acc;
  sumsq::zero(acc);
  for (int k = lane; k < H; k += 32) {
    const float f = bf16_bits_to_float(xr[k]);
    sumsq::add_term(acc, __fmul_rn(f, f));
  }
  sumsq::warp_reduce(acc, 16);
  const float r = sumsq::rms_scale(sumsq::round_to_f32(acc), H, eps);

  float a = 0.0f;
  for (int k = lane; k < H; k += 32) {
    float n = __fmul_rn(__fmul_rn(bf16_bits_to_float(xr[k]), r), g[k]);
    a = fmaxf(a, fabsf(n));
  }
  a = warp_max_f32(a);
  const ActScale sc = act_scale_from_absmax(a);
  if (lane == 0) x_scale[row] = sc.scale;
  int8_t* qr = xq + (int64_t)row * H;
  for (int k = lane; k < H; k += 32) {
    float n = __fmul_rn(__fmul_rn(bf16_bits_to_float(xr[k]), r), g[k]);
    qr[k] = (int8_t)round_clip(__fmul_rn(n, sc.inv), -128.f, 127.f);
  }
}

// h = (t * t) * u with t = max(v, 0), then the per-token quantisation of h.
__device__ __forceinline__ float relu2_mul(float u, float v) {
  float t = v > 0.0f ? v : 0.0f;
  return __fmul_rn(__fmul_rn(t, t), u);
}

__global__ void __launch_bounds__(kThreads)
k_relu2_quant(const float4* __restrict__ u, const float4* __restrict__ v, int F,
              float4* __restrict__ h, uint32_t* __restrict__ hq, float* __restrict__ h_scale) {
  __shared__ float red[kThreads / 32];
  const int row = blockIdx.x;
  const int nv = F >> 2;
  const int64_t base = (int64_t)row * nv;
  float a = 0.0f;
  for (int j = threadIdx.x; j < nv; j += kThreads) {
    float4 uu = u[base + j], vv = v[base + j];
    float4 hh = make_float4(relu2_mul(uu.x, vv.x), relu2_mul(uu.y, vv.y), relu2_mul(uu.z, vv.z),
                            relu2_mul(uu.w, vv.w));
    if (h) h[base + j] = hh;
    a = fmaxf(fmaxf(fmaxf(a, fabsf(hh.x)), fmaxf(fabsf(hh.y), fabsf(hh.z))), fabsf(hh.w));
  }
  a = block_max(a, red);
  const ActScale sc = act_scale_from_absmax(a);
  if (threadIdx.x == 0) h_scale[row] = sc.scale;
  for (int j = threadIdx.x; j < nv; j += kThreads) {
    float4 uu = u[base + j], vv = v[base + j];
    hq[base + j] = pack_i8x4(round_clip(__fmul_rn(relu2_mul(uu.x, vv.x), sc.inv), -128.f, 127.f),
                             round_clip(__fmul_rn(relu2_mul(uu.y, vv.y), sc.inv), -128.f, 127.f),
                             round_clip(__fmul_rn(relu2_mul(uu.z, vv.z), sc.inv), -128.f, 127.f),
                             round_clip(__fmul_rn(relu2_mul(uu.w, vv.w), sc.inv), -128.f, 127.f));
  }
}

}  // namespace

cudaError_t launch_quantize_act_bf16(const uint16_t* x, int64_t M, int64_t K, int8_t* xq,
                                     float* x_scale, cudaStream_t s) {
  k_act_quant_bf16<<<(unsigned)M, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(x), (int)K,
                                                    reinterpret_cast<uint2*>(xq), x_scale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_act_f32(const float* x, int64_t M, int64_t K, int8_t* xq,
                                    float* x_scale, cudaStream_t s) {
  k_act_quant_f32<<<(unsigned)M, kThreads, 0, s>>>(reinterpret_cast<const float4*>(x), (int)K,
                                                   reinterpret_cast<uint32_t*>(xq), x_scale);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_quant(const uint16_t* x, const float* g, float eps, int64_t M,
                                 int64_t H, int8_t* xq, float* x_scale, cudaStream_t s) {
  const unsigned grid = (unsigned)((M + kNormWarps - 1) / kNormWarps);
  k_rmsnorm_quant<<<grid, kNormWarps * 32, 0, s>>>(x, g, eps, (int)M, (int)H, xq, x_scale);
  return cudaGetLastError();
}

cudaError_t launch_relu2_quant(const float* u, const float* v, int64_t M, int64_t F, float* h,
                               int8_t* hq, float* h_scale, cudaStream_t s) {
  k_relu2_quant<<<(unsigned)M, kThreads, 0, s>>>(
      reinterpret_cast<const float4*>(u), reinterpret_cast<const float4*>(v), (int)F,
      reinterpret_cast<float4*>(h), reinterpret_cast<uint32_t*>(hq), h_scale);
  return cudaGetLastError();
}

}  // namespace bitnet
