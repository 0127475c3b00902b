// decode_common.cuh — device pieces shared by the decode kernels
// (gemv_decode.cu: single launches; decode_chain.cu: persistent chains).
//
// The dot product is the BitLinear of "BitNet.cpp deep dive" (dashen-tech),
// §3.1: acc = sum_pos - sum_neg over a row's ternary weights.  The stored
// 2-bit code c = q + 1 is used directly (sum q x = sum c x - sum x): in a
// 16-byte block of the packed layout, word i masked with 0x03030303 << 2s
// holds 4^s times the codes of weights 16s + 4i + {0..3}, so one AND and one
// byte dot product (dp4a) cover four weights; field s keeps its own
// accumulator and the 4^s is removed by an exact shift.
#pragma once

#include "common.cuh"

namespace bitnet {
namespace dec {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxRowsPerWarp = 8;         // rows of one stage handled by one warp
constexpr long long kDrainCycles = 2000000000ll;  // bound of the final copy drain (~1 s)

// ---- mbarrier / bulk-copy primitives (PTX ISA: mbarrier, cp.async.bulk)
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity; false after `limit`
// clocks.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Named barrier 1 over the consumer warps.
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}
// Consumer barrier that also ORs a flag over the consumers: every consumer
// leaves with the same answer (an abort decision taken after it is uniform,
// so no consumer is left waiting at a later barrier).
__device__ __forceinline__ bool consumer_sync_or(int flag) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(flag), "n"(kConsumers)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Partial dot products of NR rows (1 or 2; row addresses w[]) for this lane:
// J chunks, MT tokens, one accumulator per row, token and field (scaled by
// 4^s), folded to one int per row and token.  With two rows their
// accumulations alternate, so consecutive dp4a never feed each other.
template <int MT, int J, int NR>
__device__ __forceinline__ void row_partials(const uint32_t (&w)[NR], int valid_j,
                                             const uint4 (&xr)[MT][J][4], int (&v)[NR][MT]) {
  int acc[NR][MT][4];
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int s = 0; s < 4; ++s) acc[r][m][s] = 0;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if (j < valid_j) {
      uint32_t q[NR][4];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const uint4 pk = lds128(w[r] + 512 * j);
        q[r][0] = pk.x;
        q[r][1] = pk.y;
        q[r][2] = pk.z;
        q[r][3] = pk.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint4 xv = xr[m][j][s];
            const uint32_t xw = i == 0 ? xv.x : i == 1 ? xv.y : i == 2 ? xv.z : xv.w;
            const uint32_t mask = 0x03030303u << (2 * s);
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[r][m][s] = dp4a_us(q[r][i] & mask, xw, acc[r][m][s]);
          }
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m)
      v[r][m] = acc[r][m][0] + (acc[r][m][1] >> 2) + (acc[r][m][2] >> 4) + (acc[r][m][3] >> 6);
}

}  // namespace dec
}  // namespace bitnet
