// gemv_lut.cu — one-token BitLinear with a lookup-table inner product, the
// ablation of the dp4a inner loop.
//
// "BitNet.cpp deep dive" (dashen-tech), §3.2, lists the kernel families of
// the CPU library: I2_S (the 2-bit format this library packs, §2.3) and the
// table-lookup kernels TL1/TL2, which, like T-MAC ("Microsoft BitNet: 100B
// models on CPU" (juejin), T-MAC section), replace multiplications by
// lookups into tables of precomputed activation sums.  Here the table form is
// the TL1 one: the 2-bit codes of two weights make a 4-bit index, and for
// every pair of activations that shares a nibble of the packed weights a
// table of its 16 sums c0 x0 + c1 x1 (codes c in 0..3; code 3 never occurs)
// is built once per launch in shared memory.  A row then costs two table
// reads per byte of packed weights.  The product is the same integer as the
// dp4a path's, acc = sum_k c_k x_k - sum_k x_k ("BitNet.cpp deep dive" §3.1:
// sum_pos - sum_neg), and y = f32(acc) * (x_scale * w_scale), so both
// variants are bit-identical to the oracle.
//
// Both variants share everything but the inner product (grid-stride warps
// over rows, 16-byte streaming loads of each row, lane l taking the 64-weight
// blocks l, l + 32, ...), so the measured difference is the inner product
// alone:
//  * variant 0, table: in a 16-byte block, byte b holds the codes of weights
//    b + 16 s (s = 0..3, bits 2s); its low nibble pairs weights b and b + 16,
//    its high nibble b + 32 and b + 48.  Table word ((2 b + h) * 8 + e) * NB
//    + blk holds the entries 2e and 2e + 1 of pair (blk, b, h) as two int16,
//    so the 32 lanes (consecutive blocks) of one lookup fall in distinct
//    banks when they read the same entry word;
//  * variant 1, dp4a: the masked-field dp4a of the decode kernels, with the
//    block's activations held in registers.
#include "common.cuh"

namespace bitnet {
namespace {

constexpr int kLutThreads = 256;
constexpr int kLutWarps = kLutThreads / 32;

__device__ __forceinline__ uint4 ld_weights(const uint8_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Table words of K: 8 per activation pair, K / 2 pairs.
constexpr int64_t lut_words(int64_t K) { return 4 * K; }

template <bool LUT>
__global__ void __launch_bounds__(kLutThreads)
    k_gemv_lut(const uint8_t* __restrict__ Wq, const float* __restrict__ w_scale,
               const int8_t* __restrict__ xq, const float* __restrict__ x_scale, int N, int K,
               float* __restrict__ y, int32_t* __restrict__ acc_out) {
  extern __shared__ __align__(16) uint32_t tab[];  // table: 4 K words; dp4a: K / 4 words of x
  const int NB = K >> 6;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  if (LUT) {
    // word i = ((2 b + h) * 8 + e) * NB + blk: entries 2e, 2e + 1 of the pair
    // x0 = x[64 blk + b + 32 h], x1 = x[64 blk + b + 32 h + 16]; entry
    // c0 + 4 c1 = c0 x0 + c1 x1 (|entry| <= 3 * 128 * 2, an int16)
    for (int i = threadIdx.x; i < NB * 256; i += kLutThreads) {
      const int blk = i % NB, rest = i / NB;
      const int e = rest & 7, bh = rest >> 3, b = bh >> 1, h = bh & 1;
      const int x0 = xq[64 * blk + b + 32 * h], x1 = xq[64 * blk + b + 32 * h + 16];
      const int i0 = 2 * e, i1 = 2 * e + 1;
      const int v0 = (i0 & 3) * x0 + (i0 >> 2) * x1;
      const int v1 = (i1 & 3) * x0 + (i1 >> 2) * x1;
      tab[i] = ((uint32_t)v0 & 0xffffu) | ((uint32_t)v1 << 16);
    }
  } else {
    for (int i = threadIdx.x; i < K / 4; i += kLutThreads)
      tab[i] = reinterpret_cast<const uint32_t*>(xq)[i];
  }
  // sum of this lane's activations (its blocks lane, lane + 32, ...)
  int lsum = 0;
  for (int blk = lane; blk < NB; blk += 32) {
    const uint4* xb = reinterpret_cast<const uint4*>(xq + 64 * blk);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = xb[q];
      lsum = dp4a_ss(v.x, 0x01010101u, lsum);
      lsum = dp4a_ss(v.y, 0x01010101u, lsum);
      lsum = dp4a_ss(v.z, 0x01010101u, lsum);
      lsum = dp4a_ss(v.w, 0x01010101u, lsum);
    }
  }
  const float c = __fmul_rn(*x_scale, *w_scale);
  __syncthreads();

  const int64_t rb = K / 4;
  for (int row = blockIdx.x * kLutWarps + warp; row < N; row += gridDim.x * kLutWarps) {
    const uint8_t* wr = Wq + (int64_t)row * rb;
    int acc = 0;
    int accs[4] = {0, 0, 0, 0};
    for (int blk = lane; blk < NB; blk += 32) {
      const uint4 w4 = ld_weights(wr + 16 * blk);
      const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
      if (LUT) {
#pragma unroll
        for (int wi = 0; wi < 4; ++wi)
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int b = 4 * wi + t;
            const uint32_t byte = (ww[wi] >> (8 * t)) & 0xffu;
            const uint32_t lo = byte & 15u, hi = byte >> 4;
            const uint32_t wl = tab[((2 * b) * 8 + (int)(lo >> 1)) * NB + blk];
            const uint32_t wh = tab[((2 * b + 1) * 8 + (int)(hi >> 1)) * NB + blk];
            acc += (int)(int16_t)(uint16_t)(wl >> (16 * (lo & 1u))) +
                   (int)(int16_t)(uint16_t)(wh >> (16 * (hi & 1u)));
          }
      } else {
        // word wi masked with 0x03030303 << 2s: 4^s times the codes of the
        // block's weights 16 s + 4 wi + {0..3}, whose activations are x word
        // 4 s + wi of the block
        const uint4* xb = reinterpret_cast<const uint4*>(tab + 16 * blk);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint4 xv = xb[s];
          const uint32_t m = 0x03030303u << (2 * s);
          accs[s] = dp4a_us(ww[0] & m, xv.x, accs[s]);
          accs[s] = dp4a_us(ww[1] & m, xv.y, accs[s]);
          accs[s] = dp4a_us(ww[2] & m, xv.z, accs[s]);
          accs[s] = dp4a_us(ww[3] & m, xv.w, accs[s]);
        }
      }
    }
    if (!LUT) acc = accs[0] + (accs[1] >> 2) + (accs[2] >> 4) + (accs[3] >> 6);
    const int tot = __reduce_add_sync(0xffffffffu, acc - lsum);
    if (lane == 0) {
      y[row] = __fmul_rn(__int2float_rn(tot), c);
      if (acc_out) acc_out[row] = tot;
    }
  }
}

template <bool LUT>
cudaError_t launch_lut_t(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                         const float* x_scale, int64_t N, int64_t K, float* y, int32_t* acc_out,
                         cudaStream_t s) {
  const size_t smem = LUT ? (size_t)lut_words(K) * 4 : (size_t)K;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(k_gemv_lut<LUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)lut_words(kLutMaxK) * 4);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemv_lut<LUT>, kLutThreads, smem);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int64_t grid = (N + kLutWarps - 1) / kLutWarps;
  const int64_t full = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  if (grid > full) grid = full;
  return launch_pdl(k_gemv_lut<LUT>, dim3((unsigned)grid), dim3(kLutThreads), smem, s, Wq,
                    w_scale, xq, x_scale, (int)N, (int)K, y, acc_out);
}

}  // namespace

cudaError_t launch_gemv_lut(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                            const float* x_scale, int64_t N, int64_t K, float* y,
                            int32_t* acc_out, int variant, cudaStream_t s) {
  if (variant == 0) return launch_lut_t<true>(Wq, w_scale, xq, x_scale, N, K, y, acc_out, s);
  return launch_lut_t<false>(Wq, w_scale, xq, x_scale, N, K, y, acc_out, s);
}

}  // namespace bitnet
