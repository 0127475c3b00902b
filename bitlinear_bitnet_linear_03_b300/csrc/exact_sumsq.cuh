// exact_sumsq.cuh — the subln RMSNorm's sum of squares, exactly.
//
// "Microsoft BitNet b1.58 ... 1-bit AI model" (communeify), "Meet BitNet
// b1.58 2B4T", names subln normalisation and no formula; the library's
// reading is: t_k = x_k * x_k (one binary32 product), ss = the exact sum of
// the t_k rounded once to binary32 (ties to even), r = 1 / sqrt(ss / H + eps)
// in four binary32 operations.  The sum is exact and so independent of the
// order of the additions: every finite binary32 value is an integer multiple
// of 2^-149 below 2^277, so a sum of up to 2^16 squares is an integer below
// 2^293 in those units, held here in five 64-bit limbs and added with carry
// chains.  A NaN square makes ss NaN; otherwise an infinite square makes it
// +Inf.  No binary64 arithmetic is involved.
#pragma once

#include <stdint.h>

namespace bitnet {
namespace sumsq {

struct Acc {
  uint64_t w[5];
  uint32_t nan_, inf_;
};

__device__ __forceinline__ void zero(Acc& a) {
#pragma unroll
  for (int j = 0; j < 5; ++j) a.w[j] = 0;
  a.nan_ = a.inf_ = 0;
}

__device__ __forceinline__ void add5(Acc& s, uint64_t a0, uint64_t a1, uint64_t a2, uint64_t a3,
                                     uint64_t a4) {
  asm("add.cc.u64 %0, %0, %5;\n\t"
      "addc.cc.u64 %1, %1, %6;\n\t"
      "addc.cc.u64 %2, %2, %7;\n\t"
      "addc.cc.u64 %3, %3, %8;\n\t"
      "addc.u64 %4, %4, %9;"
      : "+l"(s.w[0]), "+l"(s.w[1]), "+l"(s.w[2]), "+l"(s.w[3]), "+l"(s.w[4])
      : "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(a4));
}

// Adds the binary32 value t (>= 0 or NaN/Inf) exactly.
__device__ __forceinline__ void add_term(Acc& s, float t) {
  const uint32_t u = __float_as_uint(t);
  const uint32_t e = (u >> 23) & 0xffu, f = u & 0x7fffffu;
  if (e == 255u) {
    if (f) s.nan_ = 1;
    else s.inf_ = 1;
    return;
  }
  const uint64_t m = e ? (uint64_t)(f | 0x800000u) : (uint64_t)f;
  const int o = e ? (int)e - 1 : 0;  // t = m * 2^(o - 149)
  const int i = o >> 6, sh = o & 63;
  const uint64_t lo = m << sh;
  const uint64_t hi = sh > 40 ? (m >> (64 - sh)) : 0ull;  // m < 2^24
  add5(s, i == 0 ? lo : 0ull, i == 1 ? lo : (i == 0 ? hi : 0ull),
       i == 2 ? lo : (i == 1 ? hi : 0ull), i == 3 ? lo : (i == 2 ? hi : 0ull),
       i == 3 ? hi : 0ull);
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int off, unsigned mask) {
  const uint32_t lo = __shfl_xor_sync(mask, (uint32_t)v, off);
  const uint32_t hi = __shfl_xor_sync(mask, (uint32_t)(v >> 32), off);
  return ((uint64_t)hi << 32) | lo;
}

// Butterfly over the lanes l ^ off for off = first .. 1 (powers of two): every
// participating lane ends with the sum of its group.
__device__ __forceinline__ void warp_reduce(Acc& s, int first) {
  for (int off = first; off >= 1; off >>= 1) {
    uint64_t o[5];
#pragma unroll
    for (int j = 0; j < 5; ++j) o[j] = shfl_xor_u64(s.w[j], off, 0xffffffffu);
    add5(s, o[0], o[1], o[2], o[3], o[4]);
    s.nan_ |= __shfl_xor_sync(0xffffffffu, s.nan_, off);
    s.inf_ |= __shfl_xor_sync(0xffffffffu, s.inf_, off);
  }
}

__device__ __forceinline__ int bit_at(const Acc& s, int pos) {
  if (pos < 0) return 0;
  const int L = pos >> 6, b = pos & 63;
  uint64_t w = 0;
#pragma unroll
  for (int j = 0; j < 5; ++j)
    if (j == L) w = s.w[j];
  return (int)((w >> b) & 1u);
}

// True if any bit below position pos is set.
__device__ __forceinline__ bool any_below(const Acc& s, int pos) {
  bool any = false;
#pragma unroll
  for (int j = 0; j < 5; ++j) {
    const int lo = 64 * j;
    if (pos >= lo + 64) any |= s.w[j] != 0;
    else if (pos > lo) any |= (s.w[j] & ((1ull << (pos - lo)) - 1ull)) != 0;
  }
  return any;
}

// The nearest binary32 (ties to even) to the exact sum.
__device__ __forceinline__ float round_to_f32(const Acc& s) {
  if (s.nan_) return __uint_as_float(0x7fc00000u);
  if (s.inf_) return __uint_as_float(0x7f800000u);
  int bl = 0;
#pragma unroll
  for (int j = 0; j < 5; ++j)
    if (s.w[j]) bl = 64 * j + 64 - __clzll((long long)s.w[j]);
  if (bl == 0) return 0.0f;
  int drop = bl > 24 ? bl - 24 : 0;
  // bits [drop, drop + 24) of the sum
  uint64_t lo = 0, hi = 0;
  const int L = drop >> 6, b = drop & 63;
#pragma unroll
  for (int j = 0; j < 5; ++j) {
    if (j == L) lo = s.w[j];
    if (j == L + 1) hi = s.w[j];
  }
  uint64_t mant = (lo >> b) | (b ? (hi << (64 - b)) : 0ull);
  mant &= 0xffffffull;
  const int round_bit = bit_at(s, drop - 1);
  const bool sticky = any_below(s, drop - 1);
  if (round_bit && (sticky || (mant & 1u))) mant += 1;
  if (mant == (1ull << 24)) {
    mant >>= 1;
    drop += 1;
  }
  // value = mant * 2^(drop - 149)
  if (mant < (1ull << 23)) return __uint_as_float((uint32_t)mant);  // subnormal (drop == 0)
  const int e8 = drop + 1;
  if (e8 >= 255) return __uint_as_float(0x7f800000u);
  return __uint_as_float(((uint32_t)e8 << 23) | ((uint32_t)mant & 0x7fffffu));
}

// ---- The common case in 128 bits.  With o_max the largest offset of any
// square (t = m * 2^(o - 149), m < 2^24), the sum is taken in units of
// 2^(anchor - 149), anchor = max(o_max - 88, 0): every term is then below
// 2^112 and the sum of up to 2^16 of them below 2^128.  A term with nonzero
// bits below the anchor (a square 2^88 times smaller than the largest) sets
// `lost`; the caller then redoes the row with the five-limb sum above.  (A
// caller may anchor each warp's terms at that warp's own largest square and
// bring the warp sums to the common anchor with shift_right128, again
// flagging any nonzero bit that falls below it.)
struct Acc128 {
  uint64_t lo, hi;
  uint32_t nan_, inf_, lost;
};

__device__ __forceinline__ void zero(Acc128& a) {
  a.lo = a.hi = 0;
  a.nan_ = a.inf_ = a.lost = 0;
}

__device__ __forceinline__ void add2(Acc128& a, uint64_t l, uint64_t h) {
  asm("add.cc.u64 %0, %0, %2;\n\taddc.u64 %1, %1, %3;" : "+l"(a.lo), "+l"(a.hi) : "l"(l), "l"(h));
}

// Offset o of a finite nonzero square (-1 for zero or non-finite).
__device__ __forceinline__ int term_offset(float t) {
  const uint32_t u = __float_as_uint(t);
  const uint32_t e = (u >> 23) & 0xffu, f = u & 0x7fffffu;
  if (e == 255u || (e == 0u && f == 0u)) return -1;
  return e ? (int)e - 1 : 0;
}

__device__ __forceinline__ void add_term(Acc128& a, float t, int anchor) {
  const uint32_t u = __float_as_uint(t);
  const uint32_t e = (u >> 23) & 0xffu, f = u & 0x7fffffu;
  const uint64_t m = e ? (uint64_t)(f | 0x800000u) : (uint64_t)f;
  const int sh = (e ? (int)e - 1 : 0) - anchor;  // <= 88 by the choice of anchor
  if (e == 255u) {
    a.nan_ |= f != 0u;
    a.inf_ |= f == 0u;
  } else if (sh >= 0) {
    const uint64_t l = sh < 64 ? m << sh : 0ull;
    const uint64_t h = sh >= 64 ? m << (sh - 64) : (sh > 40 ? m >> (64 - sh) : 0ull);
    add2(a, l, h);
  } else if (m != 0ull) {
    if (-sh >= 24 || (m & ((1ull << -sh) - 1ull))) a.lost = 1;
    if (-sh < 24) add2(a, m >> -sh, 0ull);
  }
}

__device__ __forceinline__ void warp_reduce(Acc128& a, int first) {
  for (int off = first; off >= 1; off >>= 1) {
    const uint64_t ol = shfl_xor_u64(a.lo, off, 0xffffffffu), oh = shfl_xor_u64(a.hi, off, 0xffffffffu);
    add2(a, ol, oh);
    a.nan_ |= __shfl_xor_sync(0xffffffffu, a.nan_, off);
    a.inf_ |= __shfl_xor_sync(0xffffffffu, a.inf_, off);
    a.lost |= __shfl_xor_sync(0xffffffffu, a.lost, off);
  }
}

// ---- Lean accumulation of finite squares for one lane.  A term t = m *
// 2^(o - 149) with sh = o - anchor in [0, 88] is m * 2^sh in units of
// 2^(anchor - 149); with sh = 32 q + s it goes into accumulator q as
// m * 2^s, one 32 x 32 -> 64-bit multiply-add (2^s for the two other
// accumulators is 0: a 32-bit shift of 1 by 32 or more, or by a negative
// count read as unsigned, gives 0).  Each accumulator receives terms below
// 2^56, so 32 terms stay below 2^61.  A nonzero term with sh < 0 (2^88 below
// the anchor's square) is not added and sets `lost`; the caller then takes
// the five-limb sum.
struct Lean {
  uint64_t a0, a1, a2;
  uint32_t lost;
};

__device__ __forceinline__ uint32_t shl1(int n) {
  uint32_t r;
  asm("shl.b32 %0, 1, %1;" : "=r"(r) : "r"(n));
  return r;
}
__device__ __forceinline__ uint64_t mad_wide(uint32_t a, uint32_t b, uint64_t c) {
  uint64_t r;
  asm("mad.wide.u32 %0, %1, %2, %3;" : "=l"(r) : "r"(a), "r"(b), "l"(c));
  return r;
}

// t: a finite square (>= 0).
__device__ __forceinline__ void lean_add(Lean& s, float t, int anchor) {
  const uint32_t u = __float_as_uint(t);
  const int o = max((int)(u >> 23), 1) - 1;  // subnormal or zero: o = 0
  const uint32_t m = u - ((uint32_t)o << 23);  // significand with its leading bit
  const int sh = o - anchor;
  s.a0 = mad_wide(m, shl1(sh), s.a0);
  s.a1 = mad_wide(m, shl1(sh - 32), s.a1);
  s.a2 = mad_wide(m, shl1(sh - 64), s.a2);
  s.lost |= (uint32_t)(sh < 0 && m != 0u);
}

// a0 + a1 * 2^32 + a2 * 2^64 as (lo, hi).
__device__ __forceinline__ void lean_total(const Lean& s, uint64_t& lo, uint64_t& hi) {
  const unsigned __int128 v =
      (unsigned __int128)s.a0 + ((unsigned __int128)s.a1 << 32) + ((unsigned __int128)s.a2 << 64);
  lo = (uint64_t)v;
  hi = (uint64_t)(v >> 64);
}

// The 128-bit values (lo, hi) of the 32 lanes summed exactly, every lane
// receiving the sum, when each value is below 2^122 (so the sum is below
// 2^127).  Each value is cut into five 26-bit limbs; one hardware warp
// reduction per limb adds 32 of them below 2^31, with no carry lost, and the
// five limb sums are put back together in 128 bits.
__device__ __forceinline__ void warp_sum128(uint64_t& lo, uint64_t& hi) {
  constexpr uint32_t M = (1u << 26) - 1u;
  const uint32_t l0 = __reduce_add_sync(0xffffffffu, (uint32_t)lo & M);
  const uint32_t l1 = __reduce_add_sync(0xffffffffu, (uint32_t)(lo >> 26) & M);
  const uint32_t l2 = __reduce_add_sync(0xffffffffu, (uint32_t)((lo >> 52) | (hi << 12)) & M);
  const uint32_t l3 = __reduce_add_sync(0xffffffffu, (uint32_t)(hi >> 14) & M);
  const uint32_t l4 = __reduce_add_sync(0xffffffffu, (uint32_t)(hi >> 40));
  const unsigned __int128 S = (unsigned __int128)l0 + ((unsigned __int128)l1 << 26) +
                              ((unsigned __int128)l2 << 52) + ((unsigned __int128)l3 << 78) +
                              ((unsigned __int128)l4 << 104);
  lo = (uint64_t)S;
  hi = (uint64_t)(S >> 64);
}

// (lo, hi) >>= d (d >= 0); true if a nonzero bit was shifted out.
__device__ __forceinline__ bool shift_right128(uint64_t& lo, uint64_t& hi, int d) {
  if (d <= 0) return false;
  if (d >= 128) {
    const bool lost = (lo | hi) != 0ull;
    lo = hi = 0ull;
    return lost;
  }
  if (d >= 64) {
    const int e = d - 64;
    const bool lost = lo != 0ull || (e > 0 && (hi & ((1ull << e) - 1ull)) != 0ull);
    lo = hi >> e;
    hi = 0ull;
    return lost;
  }
  const bool lost = (lo & ((1ull << d) - 1ull)) != 0ull;
  lo = (lo >> d) | (hi << (64 - d));
  hi >>= d;
  return lost;
}

// Nearest binary32 (ties to even) to S * 2^(anchor - 149), S = hi * 2^64 + lo.
__device__ __forceinline__ float round_to_f32(const Acc128& a, int anchor) {
  if (a.nan_) return __uint_as_float(0x7fc00000u);
  if (a.inf_) return __uint_as_float(0x7f800000u);
  const unsigned __int128 S = ((unsigned __int128)a.hi << 64) | a.lo;
  if (S == 0) return 0.0f;
  const int bl = a.hi ? 128 - __clzll((long long)a.hi) : 64 - __clzll((long long)a.lo);
  int drop = bl - 24 > -anchor ? bl - 24 : -anchor;  // never keep a bit below 2^-149
  uint64_t mant;
  if (drop <= 0) {
    mant = (uint64_t)(S << (-drop));  // exact
  } else {
    mant = (uint64_t)(S >> drop) & 0xffffffull;
    const bool round_bit = (uint64_t)(S >> (drop - 1)) & 1u;
    const bool sticky = drop > 1 && (S << (128 - (drop - 1))) != 0;
    if (round_bit && (sticky || (mant & 1u))) mant += 1;
    if (mant == (1ull << 24)) {
      mant >>= 1;
      drop += 1;
    }
  }
  const int d5 = drop + anchor;  // value = mant * 2^(d5 - 149)
  if (mant < (1ull << 23)) return __uint_as_float((uint32_t)mant);  // subnormal (d5 == 0)
  const int e8 = d5 + 1;
  if (e8 >= 255) return __uint_as_float(0x7f800000u);
  return __uint_as_float(((uint32_t)e8 << 23) | ((uint32_t)mant & 0x7fffffu));
}

// r = 1 / sqrt(ss / H + eps), four binary32 operations.
__device__ __forceinline__ float rms_scale(float ss, int H, float eps) {
  const float q = __fdiv_rn(ss, (float)H);
  const float t = __fadd_rn(q, eps);
  return __fdiv_rn(1.0f, __fsqrt_rn(t));
}

}  // namespace sumsq
}  // namespace bitnet
