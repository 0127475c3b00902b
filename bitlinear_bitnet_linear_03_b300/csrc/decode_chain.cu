// decode_chain.cu — the BitLinear phases of a decode step in one persistent
// kernel (one CTA per SM), with the data flow between phases carried by
// tagged values instead of grid-wide barriers.
//
// Each phase is a decode BitLinear ("BitNet.cpp deep dive" (dashen-tech),
// §3.1: acc = sum_pos - sum_neg; y = (float)acc * (x_scale * w_scale)) of a
// per-token int8 quantised input ("Microsoft BitNet b1.58 ... 1-bit AI
// model" (communeify), "Meet BitNet b1.58 2B4T": W1.58A8), optionally
// preceded by the subln RMSNorm and optionally gated, h = relu(gate)^2 * up
// (same page: subln, ReLU^2).  The weights do not depend on any phase, so the
// weight rows of every phase stream, in order, into a deep shared-memory ring
// while the consumers are still on earlier phases ("BitNet - 1-bit LLM
// inference framework" (news.hada.io), HN comment: memory bandwidth is the
// bottleneck).  There is no producer warp: the CTA's whole sequence of bulk
// copies is listed in the chain's table when the chain is built, thread 0
// issues the first ring-full, and the warp that releases a slot last (the
// eighth to finish its stage) issues the copy S stages ahead into it.  With
// eight warps (two per SM sub-partition) a thread may hold up to 255
// registers, which the in-register activations and input staging need.
//
// Data flow.  A phase input that is an output of an earlier phase (a link)
// is read through link words in the chain's table: every value is stored
// together with a tag, (run * nphases + phase + 1), in one naturally aligned
// 4-byte (bf16 value + low 16 bits of the tag) or 8-byte (binary32 value +
// the tag) word, which a single store writes and a single load reads whole.
// The writer needs no fence and there is no barrier: a consumer polls the
// words it needs until every tag is the current one, so each CTA waits
// exactly for the values it reads.  Inputs that are not links are never
// written by the chain (checked when the chain is built), so they need no
// ordering at all.  The run number comes from a counter in the table that
// every CTA increments once at its start (run = old value / CTAs).
//
// Work split: phase rows (gated: row pairs up n / gate n) are divided evenly
// over the CTAs; a stage is a run of whole rows of at most two targets (two
// copies into one slot; gated: the same rows of up, then of gate), up to
// ~62 KB, so a CTA's share of a phase is one stage even where it crosses a
// target boundary: every stage costs a release and a refill, and on B300
// those latencies, not the dot products, bound a phase.  Consumer lane l of a warp owns the 64-weight chunks l, l + 32, ...
// of its K part: their int8 activations sit in registers for the whole
// phase, and a row costs one 16-byte shared load, 16 ANDs and 16 dp4a per
// chunk (decode_common.cuh).  When several warps split K, their parts meet in
// shared-memory atomics that also count the parts; the last part writes the
// row.
//
// A thread loads all of its input groups at once, checks their tags and
// loads again only the groups still stale.  (Waiting on one word of a stale
// group before reloading, to spare L2 the full reloads, measured no faster.)
//
// The subln sum of squares is exact (exact_sumsq.cuh): each warp adds its
// squares with 32 x 32 -> 64-bit multiply-adds in 128 bits anchored 88 bits
// below its own largest square, the eight warp sums meet after one barrier
// (hardware warp reductions on 26-bit limbs), and the total is rounded once;
// a row whose squares span more than the window takes five limbs, out of
// line.  The quantisers round with a full-rate float add instead of the
// float-to-integer conversion units.  Rarely run code stays out of line and
// the row loops are not unrolled, to keep the kernel's code small.
//
// Every wait is bounded (a second by default): on time-out the kernel records
// an error bit, every warp stops at the next uniform point, the CTA waits for
// its copies in flight and returns.
#include <algorithm>
#include <vector>

#include "decode_chain.cuh"
#include "decode_common.cuh"
#include "exact_sumsq.cuh"

namespace bitnet {

__device__ int g_chain_error;

namespace {
using namespace dec;

constexpr int kMaxStages = 10;
constexpr int kChainWarps = 8;  // all consumers; no producer warp
constexpr int kChainThreads = 32 * kChainWarps;
constexpr int kMaxChainCtas = 1024;
constexpr int kListMax = 512;  // copies of a CTA's sequence held in shared memory
constexpr int kRingBudget = 192 * 1024;
constexpr int kStageTarget = 62 * 1024;  // about one stage per phase per CTA
// Groups of 8 inputs a thread keeps in registers (all of K <= 8192), and how
// many of them have their loads in flight together.
constexpr int kHold = 8192 / (8 * 32 * kChainWarps);
constexpr int kPipe = kHold;
// Stage rows whose K parts meet in shared memory (when several warps split K).
constexpr int kAccRows = kMaxRowsPerWarp * kChainWarps / 2;
constexpr int kMaxPhases = 16384;
constexpr int kErrLinkWait = 1, kErrFullWait = 2, kErrEmptyWait = 4, kErrDrain = 8;
constexpr int kTargets = kDecodeMaxTargets;

enum : int { kInBf16 = 0, kInF32 = 1, kInLinkBf16 = 2, kInLinkF32 = 3 };

struct CTarget {
  const uint8_t* Wq;
  const float* w_scale;
  float* y;
  uint16_t* y_bf16;
  int32_t* acc_out;
  uint32_t* link16;            // bf16 link words [M, N], or null
  unsigned long long* link32;  // binary32 link words [M, N], or null
  int row0;                    // first row in the phase's row space
  int N;
};

struct CPhase {
  CTarget t[kTargets];
  const void* x;                // external bf16 / binary32 input, or link words
  const float* g;               // RMSNorm gain, or null
  float* h;                     // gated: h [M, N]
  unsigned long long* h_link;   // gated: binary32 link words of h, or null
  int8_t* xq_out;
  float* xs_out;
  float eps;
  int in_kind;
  int in_phase;  // producing phase of a linked input
  int gated;
  int count;
  int rows_total;  // rows (gated: row pairs) of the phase
  int rows_q, rows_rem;  // even split over the CTAs: q rows each, one more for the first rem
  int K, wk, kpart, rows_per_stage;
  int pad;
};

// One entry of the CTA's copy sequence: a stage of whole weight rows, in one
// or two bulk copies placed one after the other in the slot (rows of one
// target, then of the next; gated: the same rows of up, then of gate).
struct StageCopy {
  const uint8_t* src0;
  const uint8_t* src1;  // second piece, or null
  uint32_t bytes0;
  uint32_t bytes1;
};

struct Args {
  const CPhase* phases;
  unsigned long long* counter;
  const StageCopy* copies;    // every CTA's copy sequence, one after another
  const uint32_t* cta_first;  // [ctas + 1]: where each CTA's sequence starts
  int nphases, M, stages, slot_bytes, xs_stride;
  long long wait;
};

// This CTA's rows [r0, r1) of a phase: q rows each, one more for the first
// rem CTAs (the host's copy lists follow the same rule).
__device__ __forceinline__ void cta_rows(const CPhase& ph, int& r0, int& r1) {
  const int b = (int)blockIdx.x;
  r0 = b * ph.rows_q + min(b, ph.rows_rem);
  r1 = r0 + ph.rows_q + (b < ph.rows_rem ? 1 : 0);
}

// The CTA's stage sequence within one phase, in order: f(r, n, t, b) for the
// stage of phase rows [r, r + n), whose rows [r, b) belong to target t and
// [b, r + n) to target t + 1 (a stage holds rows of at most two targets, so
// a CTA whose share crosses a target boundary still takes one stage); false
// if f stopped it.  Gated: rows are row pairs, t = 0, b = r + n.
template <typename F>
__device__ __forceinline__ bool for_each_stage(const CPhase& ph, F&& f) {
  int r_begin, r_end;
  cta_rows(ph, r_begin, r_end);
  if (ph.gated) {
    for (int r = r_begin; r < r_end; r += ph.rows_per_stage) {
      const int n = min(ph.rows_per_stage, r_end - r);
      if (!f(r, n, 0, r + n)) return false;
    }
    return true;
  }
  int t = 0;
  for (int r = r_begin; r < r_end;) {
    while (t + 1 < ph.count && ph.t[t + 1].row0 <= r) ++t;
    const int b = t + 1 < ph.count ? ph.t[t + 1].row0 : r_end;
    const int b2 = t + 2 < ph.count ? ph.t[t + 2].row0 : r_end;
    const int n = min(min(ph.rows_per_stage, r_end - r), b2 - r);
    if (!f(r, n, t, min(b, r + n))) return false;
    r += n;
  }
  return true;
}

__device__ __forceinline__ void copy_phase(const CPhase& src, CPhase* dst, int lane) {
  static_assert(sizeof(CPhase) % 8 == 0, "phase descriptor is copied in 8-byte words");
  const unsigned long long* s = reinterpret_cast<const unsigned long long*>(&src);
  unsigned long long* d = reinterpret_cast<unsigned long long*>(dst);
  for (int i = lane; i < (int)(sizeof(CPhase) / 8); i += 32) d[i] = s[i];
}

// Named barrier 1 over the CTA's warps, optionally ORing a flag (every warp
// leaves with the same answer).
__device__ __forceinline__ void chain_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kChainThreads) : "memory");
}
__device__ __forceinline__ bool chain_sync_or(int flag) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(flag), "n"(kChainThreads)
      : "memory");
  return r != 0;
}

// ---- link words
__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void ld_relaxed_v2u64(const void* p, unsigned long long& a,
                                                 unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Group g (8 consecutive inputs) of token m as binary32 values.  A linked
// input is polled until all 8 tags equal `tag`; false on time-out or when
// another warp has given up.
__device__ __forceinline__ bool load_group(const CPhase& ph, int m, int g, uint32_t tag,
                                           long long limit, const int* abort_flag, float (&v)[8]) {
  const int64_t base = (int64_t)m * ph.K + 8 * (int64_t)g;
  if (ph.in_kind == kInBf16) {
    const uint4 q = ld_nc_v4(static_cast<const uint16_t*>(ph.x) + base);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
      v[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
    return true;
  }
  if (ph.in_kind == kInF32) {
    const float* p = static_cast<const float*>(ph.x) + base;
    const uint4 a = ld_nc_v4(p), b = ld_nc_v4(p + 4);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(w[i]);
    return true;
  }
  long long t0 = 0;
  for (int tries = 0;; ++tries) {
    bool ok = true;
    if (ph.in_kind == kInLinkBf16) {
      const uint32_t* p = static_cast<const uint32_t*>(ph.x) + base;
      const uint4 a = ld_relaxed_v4(p), b = ld_relaxed_v4(p + 4);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      const uint32_t t16 = tag & 0xffffu;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ok &= (w[i] >> 16) == t16;
        v[i] = bf16_bits_to_float(w[i] & 0xffffu);
      }
    } else {
      const unsigned long long* p = static_cast<const unsigned long long*>(ph.x) + base;
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        unsigned long long a, b;
        ld_relaxed_v2u64(p + i, a, b);
        ok &= (uint32_t)(a >> 32) == tag && (uint32_t)(b >> 32) == tag;
        v[i] = __uint_as_float((uint32_t)a);
        v[i + 1] = __uint_as_float((uint32_t)b);
      }
    }
    if (ok) return true;
    if (tries == 0) t0 = clock64();
    else if (clock64() - t0 > limit || *(volatile const int*)abort_flag) return false;
  }
}

__device__ __forceinline__ void load_gain8(const float* g, int grp, float (&gv)[8]) {
  const uint4 a = ld_nc_v4(g + 8 * grp), b = ld_nc_v4(g + 8 * grp + 4);
  gv[0] = __uint_as_float(a.x); gv[1] = __uint_as_float(a.y);
  gv[2] = __uint_as_float(a.z); gv[3] = __uint_as_float(a.w);
  gv[4] = __uint_as_float(b.x); gv[5] = __uint_as_float(b.y);
  gv[6] = __uint_as_float(b.z); gv[7] = __uint_as_float(b.w);
}

// The raw words of group g (8 consecutive inputs) of token m, loaded without
// waiting for them: 4 (bf16), 8 (binary32 or bf16 link) or 16 (binary32
// link) words.  decode_group turns them into binary32 values and tells
// whether every tag of a linked group is the current one.  Issuing the loads
// of all of a thread's groups before looking at any keeps one memory round
// trip on the critical path instead of one per group.
struct Raw {
  uint32_t w[16];
};
__device__ __forceinline__ void issue_group(const CPhase& ph, int m, int g, Raw& r) {
  const int64_t base = (int64_t)m * ph.K + 8 * (int64_t)g;
  if (ph.in_kind == kInBf16) {
    const uint4 q = ld_nc_v4(static_cast<const uint16_t*>(ph.x) + base);
    r.w[0] = q.x; r.w[1] = q.y; r.w[2] = q.z; r.w[3] = q.w;
  } else if (ph.in_kind == kInF32) {
    const float* f = static_cast<const float*>(ph.x) + base;
    const uint4 a = ld_nc_v4(f), b = ld_nc_v4(f + 4);
    r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
    r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
  } else if (ph.in_kind == kInLinkBf16) {
    const uint32_t* q = static_cast<const uint32_t*>(ph.x) + base;
    const uint4 a = ld_relaxed_v4(q), b = ld_relaxed_v4(q + 4);
    r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
    r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
  } else {
    const unsigned long long* q = static_cast<const unsigned long long*>(ph.x) + base;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      unsigned long long a, b;
      ld_relaxed_v2u64(q + i, a, b);
      r.w[2 * i] = (uint32_t)a;
      r.w[2 * i + 1] = (uint32_t)(a >> 32);
      r.w[2 * i + 2] = (uint32_t)b;
      r.w[2 * i + 3] = (uint32_t)(b >> 32);
    }
  }
}
__device__ __forceinline__ bool decode_group(const CPhase& ph, const Raw& r, uint32_t tag,
                                             float (&v)[8]) {
  bool ok = true;
  if (ph.in_kind == kInBf16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_bits_to_float(r.w[i] & 0xffffu);
      v[2 * i + 1] = bf16_bits_to_float(r.w[i] >> 16);
    }
  } else if (ph.in_kind == kInF32) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r.w[i]);
  } else if (ph.in_kind == kInLinkBf16) {
    const uint32_t t16 = tag & 0xffffu;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ok &= (r.w[i] >> 16) == t16;
      v[i] = bf16_bits_to_float(r.w[i] & 0xffffu);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ok &= r.w[2 * i + 1] == tag;
      v[i] = __uint_as_float(r.w[2 * i]);
    }
  }
  return ok;
}

// Layout of the quantised input in shared memory: 64-weight chunk c takes 64
// bytes, its 16-byte quarter s at slot (s + c/2) mod 4, so that the 8 lanes of
// a quarter-warp reading quarter s of 8 consecutive chunks hit 8 distinct
// 16-byte bank groups.
__device__ __forceinline__ int xs_chunk_offset(int c, int s) { return 64 * c + 16 * ((s + (c >> 1)) & 3); }
// Group g (8 inputs): chunk g/8, quarter (g/2) mod 4, half g mod 2.
__device__ __forceinline__ int xs_offset(int g) {
  return xs_chunk_offset(g >> 3, (g >> 1) & 3) + 8 * (g & 1);
}

// One finished output value of a (non-gated) target: every requested form.
__device__ __forceinline__ void store_out(const CTarget& T, int64_t o, float y, int acc,
                                          uint32_t tag) {
  if (T.y) T.y[o] = y;
  const uint16_t b = (T.y_bf16 || T.link16) ? f32_to_bf16_rn(y) : (uint16_t)0;
  if (T.y_bf16) T.y_bf16[o] = b;
  if (T.acc_out) T.acc_out[o] = acc;
  if (T.link16) st_relaxed_u32(T.link16 + o, (uint32_t)b | (tag << 16));
  if (T.link32)
    st_relaxed_u64(T.link32 + o, (unsigned long long)__float_as_uint(y) |
                                     ((unsigned long long)tag << 32));
}

// ---- Out of line: inputs wider than the held groups, and the five-limb
// sum of squares.  They run rarely (K > 8192 at one token, or a row whose
// squares span more than 2^88), so they stay out of the kernel's hot code.

// Largest |x| (r == 0) or |(x * r) * g| (normalised) over the groups of token
// m this thread owns beyond the held ones.
__device__ __noinline__ float wide_absmax(const CPhase& ph, int m, int tid, uint32_t tag,
                                          long long limit, const int* abort_flag, float r,
                                          bool* bad) {
  float mx = 0.0f;
  const int ngroups = ph.K >> 3;
  for (int g = tid + kHold * kChainThreads; g < ngroups; g += kChainThreads) {
    float v[8];
    if (!load_group(ph, m, g, tag, limit, abort_flag, v)) {
      *bad = true;
      break;
    }
    if (ph.g) {
      float gv[8];
      load_gain8(ph.g, g, gv);
      for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(__fmul_rn(v[e], r), gv[e]);
    }
    for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(v[e]));
  }
  return mx;
}

// Quantises those groups into xs (and xq_out when given).
__device__ __noinline__ void wide_quantize(const CPhase& ph, int m, int tid, uint32_t tag,
                                           long long limit, const int* abort_flag, float r,
                                           float inv, int8_t* xs_row, int8_t* xq_out) {
  const int ngroups = ph.K >> 3;
  for (int g = tid + kHold * kChainThreads; g < ngroups; g += kChainThreads) {
    float v[8];
    load_group(ph, m, g, tag, limit, abort_flag, v);
    if (ph.g) {
      float gv[8];
      load_gain8(ph.g, g, gv);
      for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(__fmul_rn(v[e], r), gv[e]);
    }
    int q[8];
    for (int e = 0; e < 8; ++e) q[e] = quant_i8(__fmul_rn(v[e], inv));
    const uint2 packed = make_uint2(pack_i8x4(q[0], q[1], q[2], q[3]), pack_i8x4(q[4], q[5], q[6], q[7]));
    *reinterpret_cast<uint2*>(xs_row + xs_offset(g)) = packed;
    if (xq_out) *reinterpret_cast<uint2*>(xq_out + (int64_t)m * ph.K + 8 * g) = packed;
  }
}

// The exact sum of the squares of token m's inputs in five 64-bit limbs,
// rounded once (every thread of the CTA calls it; it synchronises them).
__device__ __noinline__ float exact_row_sumsq(const CPhase& ph, int m, int tid, uint32_t tag,
                                              long long limit, const int* abort_flag,
                                              unsigned long long* s_sum, uint32_t* s_flag) {
  const int warp = tid >> 5, lane = tid & 31;
  sumsq::Acc acc;
  sumsq::zero(acc);
  const int ngroups = ph.K >> 3;
  for (int g = tid; g < ngroups; g += kChainThreads) {
    float v[8];
    load_group(ph, m, g, tag, limit, abort_flag, v);  // already produced: returns at once
    for (int e = 0; e < 8; ++e) sumsq::add_term(acc, __fmul_rn(v[e], v[e]));
  }
  sumsq::warp_reduce(acc, 16);
  if (lane == 0) {
    for (int j = 0; j < 5; ++j) s_sum[warp * 5 + j] = acc.w[j];
    s_flag[warp] = acc.nan_ | (acc.inf_ << 1);
  }
  chain_sync();
  sumsq::Acc tot;
  sumsq::zero(tot);
  if (lane < kChainWarps) {
    for (int j = 0; j < 5; ++j) tot.w[j] = s_sum[lane * 5 + j];
    tot.nan_ = s_flag[lane] & 1u;
    tot.inf_ = s_flag[lane] >> 1;
  }
  sumsq::warp_reduce(tot, kChainWarps / 2);
  const float ss = __shfl_sync(0xffffffffu, sumsq::round_to_f32(tot), 0);
  chain_sync();  // s_sum is free again
  return ss;
}

template <int MT, int J>
__global__ void __launch_bounds__(kChainThreads, 1) k_decode_chain(const __grid_constant__ Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(16) CPhase s_ph[2];
  __shared__ float s_max[MT][kChainWarps];
  __shared__ unsigned long long s_sum128[MT][kChainWarps][2];
  __shared__ uint32_t s_sumflag[MT][kChainWarps];
  __shared__ unsigned long long s_sum5[kChainWarps][5];  // the five-limb path
  __shared__ uint32_t s_sumflag5[kChainWarps];
  // K-part merge per ring slot, stage row and token: count in bits 48.., the
  // parts' biased sums below; gated: the gate's biased sums in s_accv.
  __shared__ unsigned long long s_acc[kMaxStages][kAccRows][MT];
  __shared__ unsigned long long s_accv[kMaxStages][kAccRows][MT];
  __shared__ StageCopy s_copies[kListMax];  // the start of the CTA's copy sequence
  __shared__ int s_rel[kMaxStages];     // warps that have released the slot's stage
  __shared__ int s_issued[kMaxStages];  // copies issued into the slot
  __shared__ int s_abort;
  __shared__ uint32_t s_run;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = smem_addr(smem);
  int8_t* xs = reinterpret_cast<int8_t*>(smem + a.stages * a.slot_bytes);
  const int S = a.stages;
  const uint32_t c_first = a.cta_first[blockIdx.x];
  const int n_copies = (int)(a.cta_first[blockIdx.x + 1] - c_first);

  for (int q = threadIdx.x; q < kMaxStages * kAccRows * MT; q += kChainThreads) {
    (&s_acc[0][0][0])[q] = 0ull;
    (&s_accv[0][0][0])[q] = 0ull;
  }
  if (threadIdx.x < 32) copy_phase(a.phases[0], &s_ph[0], lane);
  for (int i = threadIdx.x; i < n_copies && i < kListMax; i += kChainThreads)
    s_copies[i] = a.copies[c_first + i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kChainWarps);
      s_rel[s] = 0;
      s_issued[s] = 0;
    }
    mbar_fence_init();
    s_abort = 0;
    const unsigned long long old = atomicAdd(a.counter, 1ull);
    s_run = (uint32_t)(old / gridDim.x);
    // The first ring-full of weight stages.
    for (int k = 0; k < S && k < n_copies; ++k) {
      const StageCopy c = a.copies[c_first + k];  // (s_copies is not yet complete)
      const uint32_t fb = smem_addr(&full_bar[k]);
      const uint32_t dst = ring + k * a.slot_bytes;
      mbar_arrive_expect_tx(fb, c.bytes0 + c.bytes1);
      bulk_copy_g2s(dst, c.src0, c.bytes0, fb);
      if (c.src1) bulk_copy_g2s(dst + c.bytes0, c.src1, c.bytes1, fb);
      s_issued[k] = 1;
    }
  }
  __syncthreads();
  // tag of phase p's outputs in this run: tag0 + p
  const uint32_t tag0 = s_run * (uint32_t)a.nphases + 1u;

  // ------------------------------------------------------------ consumers
  const int tid = threadIdx.x;  // 0 .. kChainThreads-1
  int c_slot = 0;
  uint32_t c_parity = 0;
  int c_k = 0;  // stages of the CTA's sequence consumed so far
  constexpr int kDescWords = (int)(sizeof(CPhase) / 8);
  constexpr int kDescPerLane = (kDescWords + 31) / 32;
  for (int p = 0; p < a.nphases; ++p) {
    // Every consumer has finished phase p-1, so s_ph[p & 1] (written during
    // phase p-1) is complete and s_ph[(p+1) & 1] is free.
    if (p > 0 && chain_sync_or(*(volatile int*)&s_abort)) break;
    const CPhase& ph = s_ph[p & 1];
    // Loads whose latency overlaps the wait for the input: the next phase's
    // descriptor (warp 0; stored once the input is quantised), the matrices'
    // scales and, for a normalised input, the gains of this thread's groups.
    unsigned long long desc[kDescPerLane];
    if (warp == 0 && p + 1 < a.nphases) {
      const unsigned long long* src = reinterpret_cast<const unsigned long long*>(&a.phases[p + 1]);
#pragma unroll
      for (int i = 0; i < kDescPerLane; ++i)
        if (lane + 32 * i < kDescWords) desc[i] = src[lane + 32 * i];
    }
    auto store_desc = [&]() {
      if (warp == 0 && p + 1 < a.nphases) {
        unsigned long long* dst = reinterpret_cast<unsigned long long*>(&s_ph[(p + 1) & 1]);
#pragma unroll
        for (int i = 0; i < kDescPerLane; ++i)
          if (lane + 32 * i < kDescWords) dst[lane + 32 * i] = desc[i];
      }
    };
    int r_begin, r_end;
    cta_rows(ph, r_begin, r_end);
    if (r_begin >= r_end) {  // no rows of this phase here: its input is not needed
      store_desc();
      continue;
    }
    const bool reporter = r_begin == 0;  // the one CTA with rows that starts at row 0
    const float ws_lane = lane < ph.count ? *ph.t[lane].w_scale : 0.0f;

    // ---- prologue: the phase input, (normalised,) quantised into xs
    const int K = ph.K;
    const int ngroups = K >> 3;
    const bool norm = ph.g != nullptr;
    const uint32_t in_tag = tag0 + (uint32_t)ph.in_phase;
    float gh[kHold][8];
    if (norm) {
#pragma unroll
      for (int i = 0; i < kHold; ++i)
        if (tid + i * kChainThreads < ngroups) load_gain8(ph.g, tid + i * kChainThreads, gh[i]);
    }
    float xscale[MT];
    bool stop = false;
    // Inputs beyond the held groups (K > 8 * kHold * kChainThreads) take the
    // out-of-line paths below.
    const bool wide = ngroups > kHold * kChainThreads;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      xscale[m] = 0.0f;
      if (m >= a.M || stop) continue;
      float hv[kHold][8];
      bool bad = false;
      // The held groups (tid + i * kChainThreads, i < kHold), kPipe at a
      // time: their loads first, then the tags; a linked group not yet
      // produced is polled again.
#pragma unroll
      for (int c = 0; c < kHold; c += kPipe) {
        if (bad || tid + c * kChainThreads >= ngroups) break;
        Raw raw[kPipe];
        uint32_t pend = 0;
#pragma unroll
        for (int i = 0; i < kPipe; ++i)
          if (tid + (c + i) * kChainThreads < ngroups)
            issue_group(ph, m, tid + (c + i) * kChainThreads, raw[i]);
#pragma unroll
        for (int i = 0; i < kPipe; ++i)
          if (tid + (c + i) * kChainThreads < ngroups && !decode_group(ph, raw[i], in_tag, hv[c + i]))
            pend |= 1u << i;
        if (pend) {
          const long long t0 = clock64();
          // Spin without sleeping: a sleeping poller can wake microseconds
          // after its input has landed (measured on B300).
          while (pend) {
#pragma unroll
            for (int i = 0; i < kPipe; ++i)
              if ((pend >> i) & 1u) issue_group(ph, m, tid + (c + i) * kChainThreads, raw[i]);
#pragma unroll
            for (int i = 0; i < kPipe; ++i)
              if (((pend >> i) & 1u) && decode_group(ph, raw[i], in_tag, hv[c + i]))
                pend &= ~(1u << i);
            if (pend && (clock64() - t0 > a.wait || *(volatile int*)&s_abort)) {
              bad = true;
              break;
            }
          }
        }
      }
      float mx = 0.0f;
      if (!norm) {
#pragma unroll
        for (int i = 0; i < kHold; ++i)
          if (tid + i * kChainThreads < ngroups)
#pragma unroll
            for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(hv[i][e]));
        if (wide && !bad) mx = fmaxf(mx, wide_absmax(ph, m, tid, in_tag, a.wait, &s_abort, 0.0f, &bad));
      }
      if (bad) {
        atomicOr(&g_chain_error, kErrLinkWait);
        *(volatile int*)&s_abort = 1;
      }
      float r = 0.0f;
      if (norm) {
        // ss = exact sum of the squares (exact_sumsq.cuh): each warp sums its
        // squares t = x * x (binary32) in 128 bits anchored 88 bits below its
        // largest square; after one barrier every warp brings the eight warp
        // sums to the common anchor and adds them (hardware warp reductions,
        // every lane gets the total).  A row whose squares span more than that
        // window (a nonzero square falls below the anchor), or a wide row,
        // takes the five-limb sum.  The largest square comes from the bit
        // patterns (t >= 0; a NaN square, of either sign, or +Inf has an
        // exponent field of 255 or more).
        uint32_t tb = 0u;
#pragma unroll
        for (int i = 0; i < kHold; ++i)
          if (tid + i * kChainThreads < ngroups)
#pragma unroll
            for (int e = 0; e < 8; ++e) tb = max(tb, __float_as_uint(__fmul_rn(hv[i][e], hv[i][e])));
        const uint32_t tb_w = __reduce_max_sync(0xffffffffu, tb);
        sumsq::Acc128 acc;
        sumsq::zero(acc);
        int aw = 0;
        if ((tb_w >> 23) >= 255u) {  // warp-uniform: ss is NaN or +Inf, no sum needed
#pragma unroll
          for (int i = 0; i < kHold; ++i)
            if (tid + i * kChainThreads < ngroups)
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float t = __fmul_rn(hv[i][e], hv[i][e]);
                acc.nan_ |= t != t;
                acc.inf_ |= t == __uint_as_float(0x7f800000u);
              }
        } else {
          aw = max(max((int)(tb_w >> 23), 1) - 1 - 88, 0);
          sumsq::Lean ln = {0ull, 0ull, 0ull, 0u};
#pragma unroll
          for (int i = 0; i < kHold; ++i)
            if (tid + i * kChainThreads < ngroups)
#pragma unroll
              for (int e = 0; e < 8; ++e) sumsq::lean_add(ln, __fmul_rn(hv[i][e], hv[i][e]), aw);
          sumsq::lean_total(ln, acc.lo, acc.hi);
          acc.lost = ln.lost;
          sumsq::warp_sum128(acc.lo, acc.hi);
        }
        const uint32_t fl_w =
            __reduce_or_sync(0xffffffffu, acc.nan_ | (acc.inf_ << 1) | (acc.lost << 2));
        if (lane == 0) {
          s_sum128[m][warp][0] = acc.lo;
          s_sum128[m][warp][1] = acc.hi;
          s_sumflag[m][warp] = fl_w | ((uint32_t)aw << 8);
        }
        if (chain_sync_or(*(volatile int*)&s_abort)) {
          stop = true;
          continue;
        }
        uint64_t lo = 0ull, hi = 0ull;
        uint32_t fl = 0u;
        int aj = 0;
        if (lane < kChainWarps) {
          lo = s_sum128[m][lane][0];
          hi = s_sum128[m][lane][1];
          fl = s_sumflag[m][lane] & 0xffu;
          aj = (int)(s_sumflag[m][lane] >> 8);
        }
        const int anchor = __reduce_max_sync(0xffffffffu, aj);
        if (sumsq::shift_right128(lo, hi, anchor - aj)) fl |= 4u;
        sumsq::warp_sum128(lo, hi);
        fl = __reduce_or_sync(0xffffffffu, fl);
        float ss;
        if ((fl & 4u) || wide) {  // uniform over the CTA
          ss = exact_row_sumsq(ph, m, tid, in_tag, a.wait, &s_abort, &s_sum5[0][0], &s_sumflag5[0]);
        } else {
          sumsq::Acc128 tot;
          tot.lo = lo;
          tot.hi = hi;
          tot.nan_ = fl & 1u;
          tot.inf_ = (fl >> 1) & 1u;
          tot.lost = 0u;
          ss = sumsq::round_to_f32(tot, anchor);
        }
        r = sumsq::rms_scale(ss, K, ph.eps);
        // n = (x * r) * g, then its largest magnitude
#pragma unroll
        for (int i = 0; i < kHold; ++i)
          if (tid + i * kChainThreads < ngroups)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              hv[i][e] = __fmul_rn(__fmul_rn(hv[i][e], r), gh[i][e]);
              mx = fmaxf(mx, fabsf(hv[i][e]));
            }
        if (wide) mx = fmaxf(mx, wide_absmax(ph, m, tid, in_tag, a.wait, &s_abort, r, &bad));
      }
      // mx >= 0 and never NaN, so its bit pattern orders like its value
      mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx)));
      if (lane == 0) s_max[m][warp] = mx;
      if (chain_sync_or(*(volatile int*)&s_abort)) {
        stop = true;
        continue;
      }
      float amax = s_max[m][0];
#pragma unroll
      for (int w = 1; w < kChainWarps; ++w) amax = fmaxf(amax, s_max[m][w]);
      const ActScale sc = act_scale_from_absmax(amax);
      xscale[m] = sc.scale;
      int8_t* xs_row = xs + (int64_t)m * a.xs_stride;
#pragma unroll
      for (int i = 0; i < kHold; ++i) {
        const int g = tid + i * kChainThreads;
        if (g >= ngroups) break;
        int q[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = quant_i8(__fmul_rn(hv[i][e], sc.inv));
        const uint2 packed = make_uint2(pack_i8x4(q[0], q[1], q[2], q[3]),
                                        pack_i8x4(q[4], q[5], q[6], q[7]));
        *reinterpret_cast<uint2*>(xs_row + xs_offset(g)) = packed;
        if (reporter && ph.xq_out)
          *reinterpret_cast<uint2*>(ph.xq_out + (int64_t)m * K + 8 * g) = packed;
      }
      if (wide)
        wide_quantize(ph, m, tid, in_tag, a.wait, &s_abort, r, sc.inv, xs_row,
                      reporter ? ph.xq_out : nullptr);
      if (reporter && tid == 0 && ph.xs_out) ph.xs_out[m] = sc.scale;
    }
    if (stop || chain_sync_or(*(volatile int*)&s_abort)) break;
    store_desc();

    // ---- this warp's K part and its activations in registers
    const int wk = ph.wk;
    const int kw = warp % wk, wr = warp / wk, nwr = kChainWarps / wk;
    const int nch = K >> 6;
    const int k_lo = kw * ph.kpart, k_hi = min(nch, k_lo + ph.kpart);
    int valid_j = 0;
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (k_lo + lane + 32 * j < k_hi) valid_j = j + 1;
    uint4 xr[MT][J][4];
    int lsum[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int ls[4] = {0, 0, 0, 0};  // four independent sums (short dependency chains)
#pragma unroll
      for (int j = 0; j < J; ++j) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (m < a.M && j < valid_j)
            v = *reinterpret_cast<const uint4*>(xs + (int64_t)m * a.xs_stride +
                                                xs_chunk_offset(k_lo + lane + 32 * j, s));
          xr[m][j][s] = v;
          ls[0] = dp4a_ss(v.x, 0x01010101u, ls[0]);
          ls[1] = dp4a_ss(v.y, 0x01010101u, ls[1]);
          ls[2] = dp4a_ss(v.z, 0x01010101u, ls[2]);
          ls[3] = dp4a_ss(v.w, 0x01010101u, ls[3]);
        }
      }
      lsum[m] = (ls[0] + ls[1]) + (ls[2] + ls[3]);
    }
    const int64_t rb = K >> 2;
    const uint32_t out_tag = tag0 + (uint32_t)p;

    // ---- the stages of this phase
    for_each_stage(ph, [&](int r_st, int nrows, int t_st, int b_st) {
      const int slot = c_slot;
      const uint32_t parity = c_parity;
      const int k = c_k++;
      if (++c_slot == S) {
        c_slot = 0;
        c_parity ^= 1u;
      }
      // The copy that will refill this slot (stage k + S): from shared
      // memory, or (past the held start of the sequence) fetched now so that
      // whichever warp releases the slot last can issue it at once.
      StageCopy next = {nullptr, nullptr, 0u, 0u};
      if (lane == 0 && k + S < n_copies)
        next = k + S < kListMax ? s_copies[k + S] : a.copies[c_first + k + S];
      auto release = [&]() {
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_addr(&empty_bar[slot]));
          if (atomicAdd(&s_rel[slot], 1) == kChainWarps - 1) {
            // The last warp to release the slot refills it.  Its wait on the
            // slot's empty barrier (every warp arrived, with release semantics)
            // orders all warps' reads of the slot, and what they saw of
            // s_abort, before the new copy; a warp that skipped its wait for
            // the stage's data had seen s_abort set, so no copy is issued then.
            s_rel[slot] = 0;
            bool free_slot = next.src0 != nullptr;
            if (free_slot && !mbar_wait(smem_addr(&empty_bar[slot]), (uint32_t)((k / S) & 1), a.wait)) {
              atomicOr(&g_chain_error, kErrEmptyWait);
              *(volatile int*)&s_abort = 1;
              free_slot = false;
            }
            if (free_slot && *(volatile int*)&s_abort) free_slot = false;
            if (free_slot) {
              const uint32_t fb = smem_addr(&full_bar[slot]);
              const uint32_t dst = ring + slot * a.slot_bytes;
              mbar_arrive_expect_tx(fb, next.bytes0 + next.bytes1);
              bulk_copy_g2s(dst, next.src0, next.bytes0, fb);
              if (next.src1) bulk_copy_g2s(dst + next.bytes0, next.src1, next.bytes1, fb);
              ++s_issued[slot];
            }
          }
        }
      };
      if (*(volatile int*)&s_abort) {
        release();
        return true;
      }
      if (!mbar_wait(smem_addr(&full_bar[slot]), parity, a.wait)) {
        if (lane == 0) atomicOr(&g_chain_error, kErrFullWait);
        *(volatile int*)&s_abort = 1;
        release();
        return true;
      }
      const uint32_t sbase = ring + slot * a.slot_bytes + 16 * (k_lo + lane);
      const int my_rows = nrows > wr ? (nrows - wr + nwr - 1) / nwr : 0;
      // Lane q*MT + m keeps the (warp-uniform) sums of row q for token m.
      int tot = 0, totv = 0;
      // (Row loops are not unrolled: one copy of the dot-product code keeps
      // the kernel small enough for the instruction cache.)
      if (!ph.gated) {
#pragma unroll 1
        for (int q = 0; q < kMaxRowsPerWarp; q += 2) {
          if (q + 1 < my_rows) {
            const uint32_t w[2] = {sbase + (uint32_t)((wr + q * nwr) * rb),
                                   sbase + (uint32_t)((wr + (q + 1) * nwr) * rb)};
            int v[2][MT];
            row_partials<MT, J, 2>(w, valid_j, xr, v);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const int s0 = __reduce_add_sync(0xffffffffu, v[0][m] - lsum[m]);
              const int s1 = __reduce_add_sync(0xffffffffu, v[1][m] - lsum[m]);
              if (lane == q * MT + m) tot = s0;
              if (lane == (q + 1) * MT + m) tot = s1;
            }
          } else if (q < my_rows) {
            const uint32_t w[1] = {sbase + (uint32_t)((wr + q * nwr) * rb)};
            int v[1][MT];
            row_partials<MT, J, 1>(w, valid_j, xr, v);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const int s0 = __reduce_add_sync(0xffffffffu, v[0][m] - lsum[m]);
              if (lane == q * MT + m) tot = s0;
            }
          }
        }
      } else {
        // row pair q: up row at q, gate row at nrows + q (the slot's second copy)
#pragma unroll 1
        for (int q = 0; q < kMaxRowsPerWarp; ++q) {
          if (q < my_rows) {
            const uint32_t w[2] = {sbase + (uint32_t)((wr + q * nwr) * rb),
                                   sbase + (uint32_t)((nrows + wr + q * nwr) * rb)};
            int v[2][MT];
            row_partials<MT, J, 2>(w, valid_j, xr, v);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const int s0 = __reduce_add_sync(0xffffffffu, v[0][m] - lsum[m]);
              const int s1 = __reduce_add_sync(0xffffffffu, v[1][m] - lsum[m]);
              if (lane == q * MT + m) {
                tot = s0;
                totv = s1;
              }
            }
          }
        }
      }
      // the row this lane reports (q = lane / MT) and its target
      const int row_l = wr + (lane / MT) * nwr;
      const int t_l = r_st + row_l < b_st ? t_st : t_st + 1;
      const float ws_t = __shfl_sync(0xffffffffu, ws_lane, ph.gated ? 0 : min(t_l, kTargets - 1));
      const float ws_g = __shfl_sync(0xffffffffu, ws_lane, 1);
      {
        const int q = lane / MT, m = lane % MT;
        if (q < my_rows && q < kMaxRowsPerWarp && m < a.M) {
          float xsc = xscale[0];
#pragma unroll
          for (int mm = 1; mm < MT; ++mm)
            if (mm == m) xsc = xscale[mm];
          const int row = wr + q * nwr;
          bool last = true;
          if (wk > 1) {
            // Merge the K parts: each part adds 1 << 48 (the count) plus its
            // value biased by 2^31 (non-negative, below 2^32), so at most 8
            // parts never carry out of the low 48 bits.  Gated: the gate's
            // part goes in first, then the counted up part, so the part that
            // completes the count sees every gate part.
            if (ph.gated) {
              atomicAdd(&s_accv[slot][row][m], (unsigned long long)((long long)totv + 2147483648ll));
              __threadfence_block();
            }
            const unsigned long long add =
                (1ull << 48) + (unsigned long long)((long long)tot + 2147483648ll);
            const unsigned long long old = atomicAdd(&s_acc[slot][row][m], add);
            last = (int)(old >> 48) == wk - 1;
            if (last) {
              const long long sum = (long long)((old + add) & 0xffffffffffffull);
              tot = (int)(sum - (long long)wk * 2147483648ll);
              s_acc[slot][row][m] = 0ull;
              if (ph.gated) {
                __threadfence_block();
                const long long sv = (long long)atomicExch(&s_accv[slot][row][m], 0ull);
                totv = (int)(sv - (long long)wk * 2147483648ll);
              }
            }
          }
          if (last) {
            if (!ph.gated) {
              const CTarget& T = ph.t[t_l];
              const int64_t o = (int64_t)m * T.N + (r_st + row - T.row0);
              store_out(T, o, __fmul_rn(__int2float_rn(tot), __fmul_rn(xsc, ws_t)), tot, out_tag);
            } else {
              const int64_t o = (int64_t)m * ph.t[0].N + r_st + row;
              const float u = __fmul_rn(__int2float_rn(tot), __fmul_rn(xsc, ws_t));
              const float v = __fmul_rn(__int2float_rn(totv), __fmul_rn(xsc, ws_g));
              const float tr = v > 0.0f ? v : 0.0f;
              const float h = __fmul_rn(__fmul_rn(tr, tr), u);
              store_out(ph.t[0], o, u, tot, out_tag);
              store_out(ph.t[1], o, v, totv, out_tag);
              ph.h[o] = h;
              if (ph.h_link)
                st_relaxed_u64(ph.h_link + o, (unsigned long long)__float_as_uint(h) |
                                                  ((unsigned long long)out_tag << 32));
            }
          }
        }
      }
      release();
      return true;
    });
  }
  // Never leave the CTA with a copy in flight: wait for the last copy issued
  // into every slot (already landed unless a wait ran out).
  chain_sync();
  if (tid == 0)
    for (int s = 0; s < S; ++s)
      if (s_issued[s] > 0 &&
          !mbar_wait(smem_addr(&full_bar[s]), (uint32_t)((s_issued[s] - 1) & 1), kDrainCycles)) {
        atomicOr(&g_chain_error, kErrDrain);
        break;
      }
}

// ---------------------------------------------------------------- host side
struct PhasePlan {
  int wk, kpart, rows_per_stage, stage_bytes;
};

int tokens_per_pass(int64_t M) { return M <= 1 ? 1 : M <= 2 ? 2 : 4; }

// Smallest J (chunks per lane) for which 8 warps can split K.
int min_j(int mt, int64_t K) {
  const int nch = (int)(K / 64);
  const int jopts[2] = {mt == 4 ? 1 : 2, mt == 1 ? 4 : 0};
  for (int o = 0; o < 2; ++o)
    if (jopts[o] && (nch + 7) / 8 <= 32 * jopts[o]) return jopts[o];
  return 0;
}

bool plan_phase(int64_t K, int j, bool gated, PhasePlan* pp) {
  if (K < 64 || K % 64 != 0 || K > 65536) return false;
  const int nch = (int)(K / 64);
  int wk = 0;
  for (int w = 1; w <= kChainWarps; w *= 2)
    if ((nch + w - 1) / w <= 32 * j) {
      wk = w;
      break;
    }
  if (!wk) return false;
  const int nwr = kChainWarps / wk;
  const int64_t row_bytes = K / 4 * (gated ? 2 : 1);  // per stage row (gated: a row pair)
  int64_t R = kStageTarget / row_bytes / nwr * nwr;
  if (R < nwr) R = nwr;
  if (R > (int64_t)kMaxRowsPerWarp * nwr) R = (int64_t)kMaxRowsPerWarp * nwr;
  pp->wk = wk;
  pp->kpart = (nch + wk - 1) / wk;
  pp->rows_per_stage = (int)R;
  pp->stage_bytes = (int)(R * row_bytes);
  return true;
}

size_t round256(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t kHeader = 256;  // run counter, padded

struct Range {
  uintptr_t lo, hi;
};
Range rng(const void* p, size_t bytes) {
  return Range{reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + bytes};
}
bool overlap(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }

// What validating a chain description yields: per phase the input kind and
// producing phase, where each link buffer sits in the table, and every CTA's
// sequence of weight copies.
struct ChainLayout {
  std::vector<int> in_kind, in_phase;
  std::vector<size_t> in_off;                  // table offset of a linked input's words
  std::vector<std::vector<size_t>> link16_off;  // per phase, per target (0 = none)
  std::vector<std::vector<size_t>> link32_off;
  std::vector<size_t> hlink_off;
  std::vector<PhasePlan> plan;
  std::vector<uint32_t> cta_first;  // [ctas + 1]
  std::vector<StageCopy> copies;
  size_t phases_off, first_off, copies_off, total;
  int ctas, mt, j, slot, stages, xs_stride;
  size_t smem;
};

// CTA c's rows of a phase with `rows` rows split over `ctas` CTAs (the rule
// of the kernel's cta_rows).
void split_rows(int64_t rows, int ctas, int c, int64_t* r0, int64_t* r1) {
  const int64_t q = rows / ctas, rem = rows % ctas;
  *r0 = c * q + std::min<int64_t>(c, rem);
  *r1 = *r0 + q + (c < rem ? 1 : 0);
}

// Every CTA's copy sequence, in the order of the kernel's for_each_stage.
void list_copies(const bitnet_decode_phase* ph, int np, ChainLayout* L) {
  L->cta_first.assign((size_t)L->ctas + 1, 0);
  L->copies.clear();
  for (int c = 0; c < L->ctas; ++c) {
    L->cta_first[(size_t)c] = (uint32_t)L->copies.size();
    for (int i = 0; i < np; ++i) {
      const bitnet_decode_phase& p = ph[i];
      const bool gated = (p.flags & BITNET_PHASE_GATED) != 0;
      const int64_t rb = p.K / 4, R = L->plan[(size_t)i].rows_per_stage;
      int64_t rows = 0;
      for (int t = 0; t < p.count; ++t) rows += p.targets[t].N;
      if (gated) rows = p.targets[0].N;
      int64_t r0, r1;
      split_rows(rows, L->ctas, c, &r0, &r1);
      if (gated) {
        for (int64_t r = r0; r < r1; r += R) {
          const int64_t n = std::min(R, r1 - r);
          L->copies.push_back({p.targets[0].Wq + r * rb, p.targets[1].Wq + r * rb,
                               (uint32_t)(n * rb), (uint32_t)(n * rb)});
        }
        continue;
      }
      // the kernel's for_each_stage: at most two targets' rows per stage
      std::vector<int64_t> start((size_t)p.count + 1, 0);
      for (int t = 0; t < p.count; ++t) start[(size_t)t + 1] = start[(size_t)t] + p.targets[t].N;
      int t = 0;
      for (int64_t r = r0; r < r1;) {
        while (t + 1 < p.count && start[(size_t)t + 1] <= r) ++t;
        const int64_t b = t + 1 < p.count ? start[(size_t)t + 1] : r1;
        const int64_t b2 = t + 2 < p.count ? start[(size_t)t + 2] : r1;
        const int64_t n = std::min(std::min(R, r1 - r), b2 - r);
        const int64_t split = std::min(b, r + n);
        StageCopy sc = {p.targets[t].Wq + (r - start[(size_t)t]) * rb, nullptr,
                        (uint32_t)((split - r) * rb), 0u};
        if (split < r + n) {
          sc.src1 = p.targets[t + 1].Wq;
          sc.bytes1 = (uint32_t)((r + n - split) * rb);
        }
        L->copies.push_back(sc);
        r += n;
      }
    }
  }
  L->cta_first[(size_t)L->ctas] = (uint32_t)L->copies.size();
}

// Checks the description and lays out the table.  BITNET_ERR_* on failure.
// max_dyn_smem: the dynamic shared memory a CTA of the chain kernel may use;
// ctas: the grid (one CTA per SM).
bitnet_status layout_chain(const bitnet_decode_phase* ph, int np, int64_t M, size_t max_dyn_smem,
                           int ctas, ChainLayout* L) {
  if (!ph) return BITNET_ERR_NULL;
  if (np < 1 || np > kMaxPhases || M < 1 || M > kDecodeMaxM) return BITNET_ERR_SHAPE;
  if (ctas < 1 || ctas > kMaxChainCtas) return BITNET_ERR_SHAPE;
  L->ctas = ctas;
  L->mt = tokens_per_pass(M);
  L->j = 0;
  int64_t max_k = 0;
  for (int i = 0; i < np; ++i) {
    const bitnet_decode_phase& p = ph[i];
    if (!p.targets) return BITNET_ERR_NULL;
    if ((p.x == nullptr) == (p.x_f32 == nullptr)) return p.x ? BITNET_ERR_SHAPE : BITNET_ERR_NULL;
    if (p.flags & ~(unsigned)BITNET_PHASE_GATED) return BITNET_ERR_SHAPE;
    const bool gated = (p.flags & BITNET_PHASE_GATED) != 0;
    if (p.count < 1 || p.count > kTargets || (gated && p.count != 2)) return BITNET_ERR_SHAPE;
    if (p.K < 64 || p.K % 64 != 0 || p.K > 65536) return BITNET_ERR_SHAPE;
    if (p.norm_gain && !p.x) return BITNET_ERR_SHAPE;  // the norm takes a bf16 input
    if (gated && !p.h) return BITNET_ERR_NULL;
    const int jj = min_j(L->mt, p.K);
    if (!jj) return BITNET_ERR_SHAPE;
    L->j = std::max(L->j, jj);
    max_k = std::max<int64_t>(max_k, p.K);
    int64_t rows = 0;
    for (int t = 0; t < p.count; ++t) {
      const bitnet_linear_target& g = p.targets[t];
      if (!g.Wq || !g.w_scale) return BITNET_ERR_NULL;
      if (!gated && !g.y && !g.y_bf16) return BITNET_ERR_NULL;
      if (g.N < 1 || g.N > (1 << 30)) return BITNET_ERR_SHAPE;
      rows += g.N;
    }
    if (gated && p.targets[0].N != p.targets[1].N) return BITNET_ERR_SHAPE;
    if (rows > (1 << 30)) return BITNET_ERR_SHAPE;
  }
  // Work split, ring and shared memory.
  L->plan.resize(np);
  int slot = 0;
  for (int i = 0; i < np; ++i) {
    if (!plan_phase(ph[i].K, L->j, (ph[i].flags & BITNET_PHASE_GATED) != 0, &L->plan[i]))
      return BITNET_ERR_SHAPE;
    slot = std::max(slot, L->plan[i].stage_bytes);
  }
  L->slot = slot;
  L->xs_stride = (int)max_k;
  int stages = kRingBudget / slot;
  stages = std::max(2, std::min(kMaxStages, stages));
  while (stages > 2 && (size_t)stages * slot + (size_t)L->mt * max_k > max_dyn_smem) --stages;
  L->stages = stages;
  L->smem = (size_t)stages * slot + (size_t)L->mt * max_k;
  if (L->smem > max_dyn_smem) return BITNET_ERR_SHAPE;

  // Outputs (written by the chain) and external inputs (read only).
  struct Out {
    Range r;
    int phase, kind;  // kind: 0 y, 1 y_bf16, 2 h, 3 other
    int target;
  };
  std::vector<Out> outs;
  for (int i = 0; i < np; ++i) {
    const bitnet_decode_phase& p = ph[i];
    for (int t = 0; t < p.count; ++t) {
      const bitnet_linear_target& g = p.targets[t];
      const size_t n = (size_t)(M * g.N);
      if (g.y) outs.push_back({rng(g.y, 4 * n), i, 0, t});
      if (g.y_bf16) outs.push_back({rng(g.y_bf16, 2 * n), i, 1, t});
      if (g.acc_out) outs.push_back({rng(g.acc_out, 4 * n), i, 3, t});
    }
    if (p.flags & BITNET_PHASE_GATED)
      outs.push_back({rng(p.h, 4 * (size_t)(M * p.targets[0].N)), i, 2, 0});
    if (p.xq_out) outs.push_back({rng(p.xq_out, (size_t)(M * p.K)), i, 3, 0});
    if (p.x_scale_out) outs.push_back({rng(p.x_scale_out, 4 * (size_t)M), i, 3, 0});
  }
  for (size_t u = 0; u < outs.size(); ++u)
    for (size_t v = u + 1; v < outs.size(); ++v)
      if (overlap(outs[u].r, outs[v].r)) return BITNET_ERR_ALIAS;

  L->in_kind.assign(np, 0);
  L->in_phase.assign(np, 0);
  L->in_off.assign(np, 0);
  L->link16_off.assign(np, std::vector<size_t>(kTargets, 0));
  L->link32_off.assign(np, std::vector<size_t>(kTargets, 0));
  L->hlink_off.assign(np, 0);
  list_copies(ph, np, L);
  L->phases_off = kHeader;
  L->first_off = round256(kHeader + (size_t)np * sizeof(CPhase));
  L->copies_off = round256(L->first_off + L->cta_first.size() * sizeof(uint32_t));
  size_t off = round256(L->copies_off + L->copies.size() * sizeof(StageCopy));
  for (int i = 0; i < np; ++i) {
    const bitnet_decode_phase& p = ph[i];
    const bool bf = p.x != nullptr;
    const Range in = bf ? rng(p.x, 2 * (size_t)(M * p.K)) : rng(p.x_f32, 4 * (size_t)(M * p.K));
    int match = -1;
    for (size_t u = 0; u < outs.size(); ++u) {
      if (!overlap(in, outs[u].r)) continue;
      const Out& o = outs[u];
      const bool exact = o.r.lo == in.lo && o.r.hi == in.hi && o.phase < i &&
                         ((bf && o.kind == 1) || (!bf && (o.kind == 0 || o.kind == 2)));
      if (!exact) return BITNET_ERR_ALIAS;
      match = (int)u;
    }
    if (match < 0) {
      L->in_kind[i] = bf ? kInBf16 : kInF32;
      continue;
    }
    const Out& o = outs[match];
    L->in_phase[i] = o.phase;
    L->in_kind[i] = bf ? kInLinkBf16 : kInLinkF32;
    size_t* slot_off = o.kind == 2   ? &L->hlink_off[o.phase]
                       : o.kind == 1 ? &L->link16_off[o.phase][o.target]
                                     : &L->link32_off[o.phase][o.target];
    if (*slot_off == 0) {  // one link buffer per linked output
      *slot_off = off;
      off = round256(off + (size_t)(M * p.K) * (bf ? 4 : 8));
    }
    L->in_off[i] = *slot_off;
  }
  // Every other array the chain reads must not overlap what it writes.
  for (int i = 0; i < np; ++i) {
    const bitnet_decode_phase& p = ph[i];
    std::vector<Range> ins;
    if (L->in_kind[i] == kInBf16) ins.push_back(rng(p.x, 2 * (size_t)(M * p.K)));
    if (L->in_kind[i] == kInF32) ins.push_back(rng(p.x_f32, 4 * (size_t)(M * p.K)));
    if (p.norm_gain) ins.push_back(rng(p.norm_gain, 4 * (size_t)p.K));
    for (int t = 0; t < p.count; ++t) {
      ins.push_back(rng(p.targets[t].Wq, (size_t)(p.targets[t].N * (p.K / 4))));
      ins.push_back(rng(p.targets[t].w_scale, 4));
    }
    for (const Range& r : ins)
      for (const Out& o : outs)
        if (overlap(r, o.r)) return BITNET_ERR_ALIAS;
  }
  L->total = off;
  return BITNET_OK;
}

int g_sm_count[64];

cudaError_t sm_count(int* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_sm_count[dev]) {
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_sm_count[dev] = v;
  }
  *n = g_sm_count[dev];
  return cudaSuccess;
}

// J of a chain: the largest any phase needs (0 if some K is not supported).
int chain_j(const bitnet_decode_phase* ph, int np, int64_t M) {
  int j = 0;
  for (int i = 0; i < np; ++i) {
    if (!ph || M < 1 || M > kDecodeMaxM) return 0;
    const int jj = min_j(tokens_per_pass(M), ph[i].K);
    if (!jj) return 0;
    j = std::max(j, jj);
  }
  return j;
}

// The dynamic shared memory one CTA of variant (mt, j) may take: the SM's
// opt-in maximum less the kernel's static arrays.
template <int MT, int J>
cudaError_t max_dyn_t(size_t* out) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, k_decode_chain<MT, J>);
  int dev = 0, optin = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  *out = (size_t)optin > fa.sharedSizeBytes ? (size_t)optin - fa.sharedSizeBytes : 0;
  return cudaSuccess;
}

cudaError_t max_dynamic_smem(int mt, int j, size_t* out) {
  *out = 0;
  if (mt == 1 && j == 2) return max_dyn_t<1, 2>(out);
  if (mt == 1 && j == 4) return max_dyn_t<1, 4>(out);
  if (mt == 2 && j == 2) return max_dyn_t<2, 2>(out);
  if (mt == 4 && j == 1) return max_dyn_t<4, 1>(out);
  return cudaSuccess;  // an unsupported shape: the layout check reports it
}

template <int MT, int J>
cudaError_t configure(int smem, int* resident) {
  cudaError_t e = cudaFuncSetAttribute(k_decode_chain<MT, J>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(resident, k_decode_chain<MT, J>, kChainThreads,
                                                       smem);
}

cudaError_t configure_variant(int mt, int j, int smem, int* resident) {
  if (mt == 1 && j == 2) return configure<1, 2>(smem, resident);
  if (mt == 1 && j == 4) return configure<1, 4>(smem, resident);
  if (mt == 2 && j == 2) return configure<2, 2>(smem, resident);
  if (mt == 4 && j == 1) return configure<4, 1>(smem, resident);
  return cudaErrorNotSupported;
}

template <int MT, int J>
cudaError_t launch_coop(const Args& a, int ctas, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kChainThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_chain<MT, J>, a);
}

}  // namespace

// The grid of a chain on the current device (one CTA per SM); 148 when no
// device answers (host-only checks).
int chain_ctas() {
  int n = 0;
  return sm_count(&n) == cudaSuccess && n > 0 ? n : 148;
}

bitnet_status check_decode_chain(const bitnet_decode_phase* phases, int nphases, int64_t M,
                                 size_t* table_bytes) {
  ChainLayout L;  // the table layout does not depend on the ring depth
  const bitnet_status st = layout_chain(phases, nphases, M, (size_t)1 << 30, chain_ctas(), &L);
  *table_bytes = st == BITNET_OK ? L.total : 0;
  return st;
}

bitnet_status build_decode_chain(const bitnet_decode_phase* phases, int nphases, int64_t M,
                                 void* table, size_t table_bytes, bitnet_decode_chain* chain,
                                 cudaError_t* cuda_err) {
  *cuda_err = cudaSuccess;
  ChainLayout L;
  size_t max_dyn = 0;
  int ctas = 0;
  cudaError_t e = sm_count(&ctas);
  if (e == cudaSuccess)
    e = max_dynamic_smem(tokens_per_pass(M), chain_j(phases, nphases, M), &max_dyn);
  if (e != cudaSuccess) {
    *cuda_err = e;
    return BITNET_ERR_CUDA;
  }
  bitnet_status st = layout_chain(phases, nphases, M, max_dyn, ctas, &L);
  if (st != BITNET_OK) return st;
  if (table_bytes < L.total) return BITNET_ERR_WORKSPACE;
  int resident = 0;
  e = configure_variant(L.mt, L.j, (int)L.smem, &resident);
  if (e != cudaSuccess) {
    *cuda_err = e;
    return BITNET_ERR_CUDA;
  }
  if (resident < 1) {
    *cuda_err = cudaErrorCooperativeLaunchTooLarge;
    return BITNET_ERR_CUDA;
  }
  uint8_t* base = static_cast<uint8_t*>(table);
  std::vector<CPhase> host((size_t)nphases);
  for (int i = 0; i < nphases; ++i) {
    const bitnet_decode_phase& p = phases[i];
    CPhase& c = host[(size_t)i];
    c = CPhase{};
    const bool gated = (p.flags & BITNET_PHASE_GATED) != 0;
    int64_t rows = 0;
    for (int t = 0; t < p.count; ++t) {
      const bitnet_linear_target& g = p.targets[t];
      CTarget& T = c.t[t];
      T.Wq = g.Wq;
      T.w_scale = g.w_scale;
      T.y = g.y;
      T.y_bf16 = g.y_bf16;
      T.acc_out = g.acc_out;
      T.link16 = L.link16_off[i][t] ? reinterpret_cast<uint32_t*>(base + L.link16_off[i][t]) : nullptr;
      T.link32 = L.link32_off[i][t]
                     ? reinterpret_cast<unsigned long long*>(base + L.link32_off[i][t])
                     : nullptr;
      T.row0 = gated ? 0 : (int)rows;
      T.N = (int)g.N;
      rows += g.N;
    }
    c.in_kind = L.in_kind[i];
    c.in_phase = L.in_phase[i];
    if (c.in_kind == kInLinkBf16 || c.in_kind == kInLinkF32) c.x = base + L.in_off[i];
    else c.x = p.x ? static_cast<const void*>(p.x) : static_cast<const void*>(p.x_f32);
    c.g = p.norm_gain;
    c.eps = p.norm_eps;
    c.gated = gated ? 1 : 0;
    c.h = p.h;
    c.h_link = L.hlink_off[i] ? reinterpret_cast<unsigned long long*>(base + L.hlink_off[i]) : nullptr;
    c.xq_out = p.xq_out;
    c.xs_out = p.x_scale_out;
    c.count = p.count;
    c.rows_total = gated ? (int)p.targets[0].N : (int)rows;
    c.rows_q = c.rows_total / ctas;
    c.rows_rem = c.rows_total % ctas;
    c.K = (int)p.K;
    c.wk = L.plan[i].wk;
    c.kpart = L.plan[i].kpart;
    c.rows_per_stage = L.plan[i].rows_per_stage;
  }
  // Clear the header (run counter) and every link word, then the phases and
  // the copy lists.
  e = cudaMemset(base, 0, L.total);
  if (e == cudaSuccess)
    e = cudaMemcpy(base + L.phases_off, host.data(), host.size() * sizeof(CPhase),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(base + L.first_off, L.cta_first.data(), L.cta_first.size() * sizeof(uint32_t),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !L.copies.empty())
    e = cudaMemcpy(base + L.copies_off, L.copies.data(), L.copies.size() * sizeof(StageCopy),
                   cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    *cuda_err = e;
    return BITNET_ERR_CUDA;
  }
  chain->table = table;
  chain->M = M;
  chain->nphases = nphases;
  chain->cfg[0] = L.mt;
  chain->cfg[1] = L.j;
  chain->cfg[2] = L.stages;
  chain->cfg[3] = L.slot;
  chain->cfg[4] = L.xs_stride;
  chain->cfg[5] = (int)L.smem;
  chain->cfg[6] = ctas;
  chain->cfg[7] = (int)(L.first_off / 256);
  chain->cfg[8] = (int)(L.copies_off / 256);
  for (int i = 9; i < 12; ++i) chain->cfg[i] = 0;
  return BITNET_OK;
}

cudaError_t launch_decode_chain(const bitnet_decode_chain* chain, long long wait_cycles,
                                cudaStream_t s) {
  Args a = {};
  uint8_t* t = static_cast<uint8_t*>(chain->table);
  a.phases = reinterpret_cast<const CPhase*>(t + kHeader);
  a.counter = reinterpret_cast<unsigned long long*>(t);
  a.cta_first = reinterpret_cast<const uint32_t*>(t + (size_t)chain->cfg[7] * 256);
  a.copies = reinterpret_cast<const StageCopy*>(t + (size_t)chain->cfg[8] * 256);
  a.nphases = chain->nphases;
  a.M = (int)chain->M;
  a.stages = chain->cfg[2];
  a.slot_bytes = chain->cfg[3];
  a.xs_stride = chain->cfg[4];
  a.wait = wait_cycles;
  const int mt = chain->cfg[0], j = chain->cfg[1], ctas = chain->cfg[6];
  const size_t smem = (size_t)chain->cfg[5];
  if (a.stages < 2 || a.stages > kMaxStages || ctas < 1) return cudaErrorInvalidValue;
  if (mt == 1 && j == 2) return launch_coop<1, 2>(a, ctas, smem, s);
  if (mt == 1 && j == 4) return launch_coop<1, 4>(a, ctas, smem, s);
  if (mt == 2 && j == 2) return launch_coop<2, 2>(a, ctas, smem, s);
  if (mt == 4 && j == 1) return launch_coop<4, 1>(a, ctas, smem, s);
  return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_chain_error(int* code, cudaStream_t s) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_chain_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_chain_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e;
}

}  // namespace bitnet
