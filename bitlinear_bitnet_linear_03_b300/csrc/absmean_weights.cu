// absmean_weights.cu — weight ternarisation and 2-bit packing.
//
// "How to run BitNet B1.58 locally" (onedollarvps), §2 Technical background:
// each weight is divided by the mean absolute value of the matrix, rounded
// and clipped to {-1, 0, +1}.  "BitNet.cpp deep dive" (dashen-tech), §2.3 I2_S
// format: two bits per weight.  "BitNet - 1-bit LLM inference framework"
// (news.hada.io), HN comment: two bits hold four values, so the stored code is
// q + 1 in {0, 1, 2}.
//
// The mean is exact: each |W| = m * 2^b (m a 24-bit integer, b = biased
// exponent - 1, in units of 2^-149) is added into a per-exponent 64-bit
// integer bin; bins are integers, so their sum is independent of the order
// in which blocks, warps and threads add.  One thread then forms the exact
// multi-word sum, divides by N*K and rounds once to binary32 (nearest, ties to
// even).  No floating-point reduction takes place anywhere.
#include <mutex>

#include "common.cuh"

namespace bitnet {
namespace {

constexpr int kBins = 254;        // b = 0 .. 253 (biased exponents 1 .. 254; subnormals share b = 0)
constexpr int kRow = 256;         // uint64 words per block: bins, then the non-finite count
constexpr int kNonfiniteSlot = 254;
constexpr int kMaxBlocks = 592;   // 4 x 148
constexpr int kStage1Threads = 256;
constexpr int kLimbs = 7;         // 448-bit exact sum

constexpr int stage1_blocks(int64_t total) {
  int64_t b = (total + 8191) / 8192;
  if (b < 1) b = 1;
  if (b > kMaxBlocks) b = kMaxBlocks;
  return (int)b;
}

// Stage 1: per-block exponent bins of sum(|W|) over a contiguous range.
__global__ void __launch_bounds__(kStage1Threads)
k_absmean_bins(const float4* __restrict__ W4, int64_t total4, unsigned long long* __restrict__ part) {
  __shared__ unsigned long long sbins[kStage1Threads / 32][kRow];
  __shared__ int s_nonfinite;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (kStage1Threads / 32) * kRow; i += blockDim.x)
    (&sbins[0][0])[i] = 0ull;
  if (threadIdx.x == 0) s_nonfinite = 0;
  __syncthreads();

  const int64_t begin = total4 * blockIdx.x / gridDim.x;
  const int64_t end = total4 * (blockIdx.x + 1) / gridDim.x;
  int nonfinite = 0;
  for (int64_t i = begin + threadIdx.x; i < end; i += blockDim.x) {
    float4 v = W4[i];
    uint32_t u[4] = {__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                     __float_as_uint(v.w)};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint32_t a = u[t] & 0x7fffffffu;
      uint32_t e = a >> 23;
      uint32_t m = a & 0x7fffffu;
      if (e == 255u) {
        nonfinite = 1;
        continue;
      }
      int bin = 0;
      if (e != 0u) {
        m |= 0x800000u;
        bin = (int)e - 1;
      }
      if (m) atomicAdd(&sbins[warp][bin], (unsigned long long)m);
    }
  }
  if (nonfinite) atomicOr(&s_nonfinite, 1);
  __syncthreads();
  for (int b = threadIdx.x; b < kRow; b += blockDim.x) {
    unsigned long long s = 0;
    if (b < kBins) {
#pragma unroll
      for (int w = 0; w < kStage1Threads / 32; ++w) s += sbins[w][b];
    } else if (b == kNonfiniteSlot) {
      s = (unsigned long long)s_nonfinite;
    }
    part[(int64_t)blockIdx.x * kRow + b] = s;
  }
}

// ---- small exact-integer helpers for the final division (one thread)
__device__ void big_add_u128_shifted(unsigned long long* S, unsigned long long lo,
                                     unsigned long long hi, int shift) {
  const int i = shift >> 6, o = shift & 63;
  unsigned long long p0, p1, p2;
  if (o == 0) {
    p0 = lo;
    p1 = hi;
    p2 = 0;
  } else {
    p0 = lo << o;
    p1 = (lo >> (64 - o)) | (hi << o);
    p2 = hi >> (64 - o);
  }
  unsigned long long add[3] = {p0, p1, p2};
  unsigned long long carry = 0;
  for (int j = i; j < kLimbs; ++j) {
    unsigned long long a = (j - i < 3) ? add[j - i] : 0ull;
    unsigned long long s1 = S[j] + a;
    unsigned long long c1 = s1 < a;
    unsigned long long s2 = s1 + carry;
    unsigned long long c2 = s2 < carry;
    S[j] = s2;
    carry = c1 + c2;
  }
}

__device__ int big_bit(const unsigned long long* S, int pos) {
  if (pos < 0 || pos >= kLimbs * 64) return 0;
  return (int)((S[pos >> 6] >> (pos & 63)) & 1ull);
}

__device__ int big_bitlen(const unsigned long long* S) {
  for (int j = kLimbs - 1; j >= 0; --j)
    if (S[j]) return j * 64 + 64 - __clzll((long long)S[j]);
  return 0;
}

// Any bit set below position `pos` (positions 0 .. pos-1)?
__device__ int big_any_below(const unsigned long long* S, int pos) {
  for (int p = 0; p < pos; ++p)
    if (big_bit(S, p)) return 1;
  return 0;
}

// Stage 2: one block.  gamma = round_to_binary32(S * 2^-149 / n);
// w_scale = max(gamma, 1e-5), or NaN when any entry was Inf or NaN.
__global__ void __launch_bounds__(256)
k_absmean_final(const unsigned long long* __restrict__ part, int nblocks, unsigned long long n,
                float* __restrict__ w_scale) {
  __shared__ unsigned long long s_lo[kRow], s_hi[kRow];
  const int t = threadIdx.x;
  {
    unsigned long long lo = 0, hi = 0;
    for (int b = 0; b < nblocks; ++b) {
      unsigned long long v = part[(int64_t)b * kRow + t];
      unsigned long long s = lo + v;
      hi += (s < v);
      lo = s;
    }
    s_lo[t] = lo;
    s_hi[t] = hi;
  }
  __syncthreads();
  if (t != 0) return;
  if (s_lo[kNonfiniteSlot] | s_hi[kNonfiniteSlot]) {
    *w_scale = __int_as_float(0x7fc00000);
    return;
  }
  unsigned long long S[kLimbs];
  for (int j = 0; j < kLimbs; ++j) S[j] = 0;
  for (int b = 0; b < kBins; ++b)
    if (s_lo[b] | s_hi[b]) big_add_u128_shifted(S, s_lo[b], s_hi[b], b);

  float gamma = 0.0f;
  const int L = big_bitlen(S);
  if (L > 0) {
    // Long division, one quotient bit per step, most significant first.  The
    // quotient bit at position j weighs 2^(j-149).  Keep 24 significant bits
    // (never a bit below position 0, the binary32 subnormal step), then round
    // half to even with the next bit and a sticky bit.
    unsigned long long r = 0;
    int P = -100000, lsb = 0, round_bit = 0, sticky = 0;
    unsigned long long mant = 0;
    for (int j = L - 1;; --j) {
      r = 2 * r + (unsigned long long)big_bit(S, j);
      int qb = r >= n;
      if (qb) r -= n;
      if (qb && P == -100000) {
        P = j;
        lsb = P - 23 > 0 ? P - 23 : 0;
      }
      if (j >= lsb) {
        mant = (mant << 1) | (unsigned long long)qb;
      } else {
        round_bit = qb;
        sticky = (r != 0) || big_any_below(S, j);
        break;
      }
    }
    if (round_bit && (sticky || (mant & 1ull))) mant += 1;
    // mant <= 2^24 and mant * 2^(lsb-149) is exactly a binary32 value.
    const double p2 = __longlong_as_double((long long)(1023 + lsb - 149) << 52);
    gamma = __double2float_rn(__dmul_rn((double)mant, p2));
  }
  *w_scale = gamma < 1e-5f ? 1e-5f : gamma;
}

// Stage 3: q = clamp(rint(W / w_scale), -1, 1), code = q + 1, packed so that
// weight j of each 64-weight block sits in byte j % 16 at bit shift
// 2 * (j / 16).  A warp handles 128 weights (two blocks): lane l holds
// weights 4l .. 4l+3, i.e. field s = (l%16)/4 of word (l%4) of its block.
__global__ void __launch_bounds__(256)
k_ternary_pack(const float4* __restrict__ W4, int64_t nblk64, const float* __restrict__ w_scale,
               uint32_t* __restrict__ Wq32) {
  const float g = *w_scale;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, L = lane & 15, s = L >> 2, i = L & 3;
  const int64_t nunits = (nblk64 + 1) / 2;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < nunits;
       u += warps_total) {
    const int64_t blk = 2 * u + half;
    const bool valid = blk < nblk64;
    uint32_t word = 0;
    if (valid) {
      float4 v = W4[blk * 16 + L];
      int q0 = round_clip(__fdiv_rn(v.x, g), -1.f, 1.f) + 1;
      int q1 = round_clip(__fdiv_rn(v.y, g), -1.f, 1.f) + 1;
      int q2 = round_clip(__fdiv_rn(v.z, g), -1.f, 1.f) + 1;
      int q3 = round_clip(__fdiv_rn(v.w, g), -1.f, 1.f) + 1;
      word = ((uint32_t)q0 | ((uint32_t)q1 << 8) | ((uint32_t)q2 << 16) | ((uint32_t)q3 << 24))
             << (2 * s);
    }
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    word |= __shfl_xor_sync(0xffffffffu, word, 8);
    if (valid && s == 0) Wq32[blk * 4 + i] = word;
  }
}

}  // namespace

size_t quantize_weights_workspace(int64_t total) {
  return (size_t)stage1_blocks(total) * kRow * sizeof(unsigned long long);
}

cudaError_t launch_quantize_weights(const float* W, int64_t total, uint8_t* Wq, float* w_scale,
                                    void* ws, cudaStream_t s) {
  const int nb = stage1_blocks(total);
  auto* part = static_cast<unsigned long long*>(ws);
  k_absmean_bins<<<nb, kStage1Threads, 0, s>>>(reinterpret_cast<const float4*>(W), total / 4,
                                               part);
  k_absmean_final<<<1, 256, 0, s>>>(part, nb, (unsigned long long)total, w_scale);
  const int64_t nblk64 = total / 64;
  const int64_t units = (nblk64 + 1) / 2;
  int64_t grid = (units + 7) / 8;
  if (grid > 148 * 16) grid = 148 * 16;
  if (grid < 1) grid = 1;
  k_ternary_pack<<<(unsigned)grid, 256, 0, s>>>(reinterpret_cast<const float4*>(W), nblk64,
                                                w_scale, reinterpret_cast<uint32_t*>(Wq));
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free variant (bitnet_quantize_weights_noalloc).  The stage-1
// partials live in this file-scope device array instead of caller-provided
// workspace.  Stage 1 never uses more than kMaxBlocks rows of kRow words,
// whatever N*K is, so the array covers every accepted size.  Each call writes
// every word it later reads, so nothing has to start at zero; calls that
// overlap on the GPU (other streams, other host threads) share the array and
// race.
constexpr size_t kNoAllocScratchBytes = (size_t)kMaxBlocks * kRow * sizeof(unsigned long long);
static __device__ __align__(256) unsigned long long g_absmean_scratch[kMaxBlocks * kRow];

namespace {
// Device address of g_absmean_scratch per device, looked up once with that
// device current (a host-side name of a __device__ array is not a device
// address).
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;
}  // namespace

size_t quantize_weights_noalloc_limit() { return kNoAllocScratchBytes; }

cudaError_t launch_quantize_weights_noalloc(const float* W, int64_t total, uint8_t* Wq,
                                            float* w_scale, cudaStream_t s) {
  // stage1_blocks caps the grid at kMaxBlocks, and the array holds kMaxBlocks
  // rows: every accepted size fits, so there is no size check here.  (Any
  // change to stage1_blocks that could exceed the array breaks the build.)
  static_assert((size_t)stage1_blocks((int64_t)1 << 40) * kRow * sizeof(unsigned long long) <=
                    kNoAllocScratchBytes,
                "the array holds the largest stage-1 grid");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
      e = cudaGetSymbolAddress(&ptr, g_absmean_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_ptr[dev] = ptr;
    }
    ptr = g_scratch_ptr[dev];
  }
  return launch_quantize_weights(W, total, Wq, w_scale, ptr, s);
}

}  // namespace bitnet
