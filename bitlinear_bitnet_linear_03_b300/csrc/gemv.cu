// gemv.cu — BitLinear on CUDA cores for decode-sized M (one to a few tokens).
//
// "BitNet.cpp deep dive" (dashen-tech), §3.1 integer matrix multiplication:
// with ternary weights the product needs no multiplication, Y = sum_pos -
// sum_neg.  Here the stored code c = q + 1 in {0, 1, 2} is used directly:
//   sum_k q[n,k] x[k] = sum_k c[n,k] x[k] - sum_k x[k],
// and sum_k c x is formed with byte dot products (dp4a) on the packed words
// without unpacking them: in a 16-byte block, word i masked with
// 0x03030303 << 2s holds 4^s * (codes of weights 16s + 4i + {0..3}), so one
// AND and one dp4a cover four weights.  Each field s keeps its own int32
// accumulator (scaled by 4^s); the scales are removed exactly by arithmetic
// shifts at the end.  All sums are integers, so the result is exact and
// independent of order; the rescale y = (float)acc * (x_scale * w_scale) is
// two binary32 products, stored as binary32 and/or rounded to bf16.
//
// Work split: a CTA owns WARPS*RPW consecutive output rows, MT tokens and one
// K-slice.  The CTA stages its tokens' int8 activations for the slice in
// shared memory (swizzled so the 16-byte reads of a quarter-warp hit distinct
// banks) together with their byte sums.  Each warp streams RPW weight rows:
// lane l reads 16-byte packed chunks l, l+32, ... of every row (512
// contiguous bytes per row per warp step), so the packed matrix is read once,
// fully coalesced, with no reuse in L1.  A K-split writes int32 partials that a
// second kernel adds (integer sums: order-free) and rescales.
#include "common.cuh"

namespace bitnet {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSmem = 48 * 1024;
constexpr int kTargetCtas = 2 * 148;

template <int MT, int RPW>
__global__ void __launch_bounds__(kThreads)
k_gemv(const uint8_t* __restrict__ Wq, const float* __restrict__ w_scale,
       const int8_t* __restrict__ xq, const float* __restrict__ x_scale, int M, int N, int K,
       int ks_len, float* __restrict__ y, uint16_t* __restrict__ y_bf16,
       int32_t* __restrict__ acc_out, int32_t* __restrict__ part) {
  extern __shared__ uint4 xs[];
  __shared__ int sumx[MT];
  const int split = blockIdx.z;
  const int k0 = split * ks_len;
  const int klen = min(ks_len, K - k0);
  const int nch = klen >> 6;
  const int m0 = blockIdx.y * MT;

  if (threadIdx.x < MT) sumx[threadIdx.x] = 0;
  __syncthreads();
  // Stage x[m0 .. m0+MT, k0 .. k0+klen): segment s of chunk c of token m at
  // uint4 slot (m*nch + c)*4 + ((s + c/2) & 3).
  for (int idx = threadIdx.x; idx < MT * nch * 4; idx += kThreads) {
    const int m = idx / (nch * 4);
    const int rem = idx - m * nch * 4;
    const int c = rem >> 2, sg = rem & 3;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (m0 + m < M) v = ld_nc_v4(xq + (int64_t)(m0 + m) * K + k0 + c * 64 + sg * 16);
    xs[(m * nch + c) * 4 + ((sg + (c >> 1)) & 3)] = v;
    int sx = dp4a_ss(v.x, 0x01010101u, 0);
    sx = dp4a_ss(v.y, 0x01010101u, sx);
    sx = dp4a_ss(v.z, 0x01010101u, sx);
    sx = dp4a_ss(v.w, 0x01010101u, sx);
    if (sx) atomicAdd(&sumx[m], sx);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrow0 = blockIdx.x * (kWarps * RPW) + warp * RPW;
  const int64_t row_bytes = K >> 2;
  const uint8_t* wbase = Wq + (k0 >> 2);

  int acc[RPW][MT][4];
#pragma unroll
  for (int r = 0; r < RPW; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int s = 0; s < 4; ++s) acc[r][m][s] = 0;

  for (int c = lane; c < nch; c += 32) {
    uint4 w[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const int n = nrow0 + r;
      w[r] = n < N ? ld_stream_v4(wbase + (int64_t)n * row_bytes + c * 16)
                   : make_uint4(0, 0, 0, 0);
    }
    const int rot = c >> 1;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const uint4* xc = xs + (m * nch + c) * 4;
      uint4 xv[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) xv[s] = xc[(s + rot) & 3];
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const uint32_t ww[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t xw[4] = {i == 0 ? xv[0].x : i == 1 ? xv[0].y : i == 2 ? xv[0].z : xv[0].w,
                                  i == 0 ? xv[1].x : i == 1 ? xv[1].y : i == 2 ? xv[1].z : xv[1].w,
                                  i == 0 ? xv[2].x : i == 1 ? xv[2].y : i == 2 ? xv[2].z : xv[2].w,
                                  i == 0 ? xv[3].x : i == 1 ? xv[3].y : i == 2 ? xv[3].z : xv[3].w};
          acc[r][m][0] = dp4a_us(ww[i] & 0x03030303u, xw[0], acc[r][m][0]);
          acc[r][m][1] = dp4a_us(ww[i] & 0x0c0c0c0cu, xw[1], acc[r][m][1]);
          acc[r][m][2] = dp4a_us(ww[i] & 0x30303030u, xw[2], acc[r][m][2]);
          acc[r][m][3] = dp4a_us(ww[i] & 0xc0c0c0c0u, xw[3], acc[r][m][3]);
        }
      }
    }
  }

  const float ws = *w_scale;
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int t = acc[r][m][0] + (acc[r][m][1] >> 2) + (acc[r][m][2] >> 4) + (acc[r][m][3] >> 6);
      t = warp_sum_i32(t);
      const int n = nrow0 + r, mm = m0 + m;
      if (lane == ((r * MT + m) & 31) && n < N && mm < M) {
        const int a = t - sumx[m];
        if (part) {
          part[((int64_t)split * M + mm) * N + n] = a;
        } else {
          const float v = __fmul_rn(__int2float_rn(a), __fmul_rn(x_scale[mm], ws));
          if (y) y[(int64_t)mm * N + n] = v;
          if (y_bf16) y_bf16[(int64_t)mm * N + n] = f32_to_bf16_rn(v);
          if (acc_out) acc_out[(int64_t)mm * N + n] = a;
        }
      }
    }
  }
}

__global__ void k_splitk_reduce(const int32_t* __restrict__ part, int splits, int M, int N,
                                const float* __restrict__ w_scale,
                                const float* __restrict__ x_scale, float* __restrict__ y,
                                uint16_t* __restrict__ y_bf16, int32_t* __restrict__ acc_out) {
  const int64_t total = (int64_t)M * N;
  const float ws = *w_scale;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    int a = 0;
    for (int s = 0; s < splits; ++s) a += part[(int64_t)s * total + i];
    const int m = (int)(i / N);
    const float v = __fmul_rn(__int2float_rn(a), __fmul_rn(x_scale[m], ws));
    if (y) y[i] = v;
    if (y_bf16) y_bf16[i] = f32_to_bf16_rn(v);
    if (acc_out) acc_out[i] = a;
  }
}

struct Plan {
  int mt, rpw, splits, ks_len;
  dim3 grid;
  size_t smem;
};

Plan make_plan(int64_t M, int64_t N, int64_t K) {
  Plan p;
  const int64_t mm = M < 8 ? M : 8;
  p.mt = mm <= 1 ? 1 : mm <= 2 ? 2 : mm <= 4 ? 4 : 8;
  p.rpw = p.mt <= 2 ? 4 : 2;
  const int64_t rows = (int64_t)kWarps * p.rpw;
  const int64_t ctas_n = (N + rows - 1) / rows;
  const int64_t tiles_m = (M + p.mt - 1) / p.mt;
  const int64_t ks_max = (kMaxSmem / p.mt) / 64 * 64;
  int64_t splits = (K + ks_max - 1) / ks_max;
  while (ctas_n * tiles_m * splits < kTargetCtas && K / (splits * 2) >= 2048) splits *= 2;
  int64_t ks = (K + splits - 1) / splits;
  ks = (ks + 63) / 64 * 64;
  splits = (K + ks - 1) / ks;
  p.splits = (int)splits;
  p.ks_len = (int)ks;
  p.grid = dim3((unsigned)ctas_n, (unsigned)tiles_m, (unsigned)splits);
  p.smem = (size_t)p.mt * (size_t)ks;
  return p;
}

template <int MT, int RPW>
void launch_kernel(const Plan& p, cudaStream_t s, const uint8_t* Wq, const float* w_scale,
                   const int8_t* xq, const float* x_scale, int M, int N, int K, float* y,
                   uint16_t* y_bf16, int32_t* acc_out, int32_t* part) {
  k_gemv<MT, RPW><<<p.grid, kThreads, p.smem, s>>>(Wq, w_scale, xq, x_scale, M, N, K, p.ks_len,
                                                   y, y_bf16, acc_out, part);
}

}  // namespace

size_t gemv_workspace(int64_t M, int64_t N, int64_t K) {
  const Plan p = make_plan(M, N, K);
  return p.splits > 1 ? (size_t)p.splits * (size_t)M * (size_t)N * sizeof(int32_t) : 0;
}

cudaError_t launch_gemv(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                        const float* x_scale, int64_t M, int64_t N, int64_t K, float* y,
                        uint16_t* y_bf16, int32_t* acc_out, void* ws, cudaStream_t s) {
  const Plan p = make_plan(M, N, K);
  int32_t* part = p.splits > 1 ? static_cast<int32_t*>(ws) : nullptr;
  const int m = (int)M, n = (int)N, k = (int)K;
  switch (p.mt) {
    case 1: launch_kernel<1, 4>(p, s, Wq, w_scale, xq, x_scale, m, n, k, y, y_bf16, acc_out, part); break;
    case 2: launch_kernel<2, 4>(p, s, Wq, w_scale, xq, x_scale, m, n, k, y, y_bf16, acc_out, part); break;
    case 4: launch_kernel<4, 2>(p, s, Wq, w_scale, xq, x_scale, m, n, k, y, y_bf16, acc_out, part); break;
    default: launch_kernel<8, 2>(p, s, Wq, w_scale, xq, x_scale, m, n, k, y, y_bf16, acc_out, part); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  int64_t total = M * N;
  int64_t grid = (total + 255) / 256;
  if (grid > 148 * 8) grid = 148 * 8;
  k_splitk_reduce<<<(unsigned)grid, 256, 0, s>>>(part, p.splits, m, n, w_scale, x_scale, y,
                                                 y_bf16, acc_out);
  return cudaGetLastError();
}

}  // namespace bitnet
