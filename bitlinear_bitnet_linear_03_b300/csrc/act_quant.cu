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

// subln RMSNorm + quantisation, one CTA of kNormWarps warps per token.
//   ss = the exact sum of the binary32 squares x_k * x_k, rounded once to
//        binary32 (exact_sumsq.cuh: order-free, integer arithmetic): each
//        warp sums its squares in 128 bits anchored 88 bits below its own
//        largest square, the warp sums are brought to the common anchor and
//        added; a row whose squares span more than that window takes the
//        five-limb sum (exact_row_sumsq5);
//   r  = 1 / sqrt(ss / H + eps), four binary32 operations;
//   n  = (x * r) * g, then the per-token quantisation of n.
constexpr int kNormWarps = 8;
constexpr int kNormThreads = kNormWarps * 32;

// The five-limb exact sum of the row's squares (every thread of the CTA
// calls it; it synchronises them).
__device__ __noinline__ float exact_row_sumsq5(const uint16_t* xr, int H,
                                              unsigned long long (*s5)[5], uint32_t* s5f) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  sumsq::Acc acc;
  sumsq::zero(acc);
  for (int k = threadIdx.x; k < H; k += kNormThreads) {
    const float f = bf16_bits_to_float(xr[k]);
    sumsq::add_term(acc, __fmul_rn(f, f));
  }
  sumsq::warp_reduce(acc, 16);
  if (lane == 0) {
    for (int j = 0; j < 5; ++j) s5[warp][j] = acc.w[j];
    s5f[warp] = acc.nan_ | (acc.inf_ << 1);
  }
  __syncthreads();
  sumsq::Acc tot;
  sumsq::zero(tot);
  if (lane < kNormWarps) {
    for (int j = 0; j < 5; ++j) tot.w[j] = s5[lane][j];
    tot.nan_ = s5f[lane] & 1u;
    tot.inf_ = s5f[lane] >> 1;
  }
  sumsq::warp_reduce(tot, kNormWarps / 2);
  return __shfl_sync(0xffffffffu, sumsq::round_to_f32(tot), 0);
}

__global__ void __launch_bounds__(kNormThreads)
k_rmsnorm_quant(const uint16_t* __restrict__ x, const float* __restrict__ g, float eps, int M,
                int H, int8_t* __restrict__ xq, float* __restrict__ x_scale) {
  __shared__ unsigned long long s_part[kNormWarps][2];
  __shared__ uint32_t s_meta[kNormWarps];
  __shared__ float s_max[kNormWarps];
  __shared__ unsigned long long s5[kNormWarps][5];
  __shared__ uint32_t s5f[kNormWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x;
  const uint16_t* xr = x + (int64_t)row * H;

  // this warp's largest square (bit patterns: t >= 0; NaN or +Inf >= 255 << 23)
  uint32_t tb = 0u;
  for (int k = threadIdx.x; k < H; k += kNormThreads) {
    const float f = bf16_bits_to_float(xr[k]);
    tb = max(tb, __float_as_uint(__fmul_rn(f, f)));
  }
  tb = __reduce_max_sync(0xffffffffu, tb);
  uint64_t lo = 0ull, hi = 0ull;
  uint32_t fl = 0u;
  int aw = 0;
  if ((tb >> 23) >= 255u) {  // warp-uniform: ss is NaN or +Inf
    for (int k = threadIdx.x; k < H; k += kNormThreads) {
      const float f = bf16_bits_to_float(xr[k]);
      const float t = __fmul_rn(f, f);
      fl |= (t != t ? 1u : 0u) | (t == __uint_as_float(0x7f800000u) ? 2u : 0u);
    }
  } else {
    aw = max(max((int)(tb >> 23), 1) - 1 - 88, 0);
    sumsq::Lean ln = {0ull, 0ull, 0ull, 0u};
    for (int k = threadIdx.x; k < H; k += kNormThreads) {
      const float f = bf16_bits_to_float(xr[k]);
      sumsq::lean_add(ln, __fmul_rn(f, f), aw);
    }
    sumsq::lean_total(ln, lo, hi);
    sumsq::warp_sum128(lo, hi);
    fl = ln.lost << 2;
  }
  fl = __reduce_or_sync(0xffffffffu, fl);
  if (lane == 0) {
    s_part[warp][0] = lo;
    s_part[warp][1] = hi;
    s_meta[warp] = fl | ((uint32_t)aw << 8);
  }
  __syncthreads();
  lo = hi = 0ull;
  fl = 0u;
  int aj = 0;
  if (lane < kNormWarps) {
    lo = s_part[lane][0];
    hi = s_part[lane][1];
    fl = s_meta[lane] & 0xffu;
    aj = (int)(s_meta[lane] >> 8);
  }
  const int anchor = __reduce_max_sync(0xffffffffu, aj);
  if (sumsq::shift_right128(lo, hi, anchor - aj)) fl |= 4u;
  sumsq::warp_sum128(lo, hi);
  fl = __reduce_or_sync(0xffffffffu, fl);
  float ss;
  if (fl & 4u) {  // uniform over the CTA
    ss = exact_row_sumsq5(xr, H, s5, s5f);
  } else {
    sumsq::Acc128 tot;
    tot.lo = lo;
    tot.hi = hi;
    tot.nan_ = fl & 1u;
    tot.inf_ = (fl >> 1) & 1u;
    tot.lost = 0u;
    ss = sumsq::round_to_f32(tot, anchor);
  }
  const float r = sumsq::rms_scale(ss, H, eps);

  float a = 0.0f;
  for (int k = threadIdx.x; k < H; k += kNormThreads) {
    const float n = __fmul_rn(__fmul_rn(bf16_bits_to_float(xr[k]), r), g[k]);
    a = fmaxf(a, fabsf(n));
  }
  // a >= 0 and never NaN: its bit pattern orders like its value
  a = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(a)));
  if (lane == 0) s_max[warp] = a;
  __syncthreads();
  a = s_max[0];
#pragma unroll
  for (int w = 1; w < kNormWarps; ++w) a = fmaxf(a, s_max[w]);
  const ActScale sc = act_scale_from_absmax(a);
  if (threadIdx.x == 0) x_scale[row] = sc.scale;
  int8_t* qr = xq + (int64_t)row * H;
  for (int k = threadIdx.x; k < H; k += kNormThreads) {
    const float n = __fmul_rn(__fmul_rn(bf16_bits_to_float(xr[k]), r), g[k]);
    qr[k] = (int8_t)quant_i8(__fmul_rn(n, sc.inv));
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
  k_rmsnorm_quant<<<(unsigned)M, kNormThreads, 0, s>>>(x, g, eps, (int)M, (int)H, xq, x_scale);
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
