// gemm_tc.cu — tensor-core BitLinear for blocks of tokens.
//
// The product is the BitLinear contraction of "BitNet.cpp deep dive"
// (dashen-tech), §3.1 (acc = sum_pos - sum_neg = sum_k q[n,k] x[m,k]) over a
// whole block of tokens, with the rescale y = (float)acc * (x_scale *
// w_scale).  sm_103a has no integer tensor-core MMA (ptxas rejects
// tcgen05.mma .kind::i8 for this target), so the contraction runs on exact
// stand-ins: bf16 operands under kind::f16 (ternary weights and int8
// activations are integers of magnitude <= 256, exact in bf16), or the e4m3
// digit forms below.  Every product is exact and every partial sum is an
// integer of magnitude <= 128 K < 2^24 for K <= 65536, so the binary32
// accumulator is exact and independent of the order of the additions; the
// epilogue rescales that binary32 integer directly (and forms int32 only for
// the optional accumulator output).
// The exact e4m3 digit form (kind::f8f6f4) replaces bf16 wherever K >= 128
// and M is not in 65..256: x = 16 hi + lo with hi in [-8, 7] and lo in
// [0, 15], both exact in e4m3, as are the ternary weights.
//  * M <= 64 (Kind<2>): each token's two digit rows are stacked in
//    one 128-row A tile, so one MMA covers 32 K instead of 16;
//  * M > 256 (Kind<4>): the digits hi' = 16 hi and lo are two A tiles of the
//    same tokens, both multiplied into one accumulator.  The tensor time
//    equals bf16's, and the operands of a 128 x 256 tile move 64 KB per 128
//    K instead of 96 KB (prefill is bound by L2 -> SM traffic).
//
// Pipeline (one CTA per SM, persistent over work items of 128 x BN output
// tiles, BN = 256, or 128 for narrow N):
//  * M <= 256 (fused): the TMA brings the A tile (bf16, or e4m3 digits) and
//    the packed 2-bit codes of the B tile (16 or 32 bytes per row per
//    stage); four converter warps expand the codes into the
//    128-byte-swizzled B tile in shared memory (bf16: one multiply-add and
//    two byte permutes per four weights; e4m3: one byte permute per four)
//    and signal the MMA.  When the output has fewer tiles than half the SMs,
//    K is split over CTAs: each split adds its exact partial sums into a
//    zeroed fp32 workspace (red.global.add.v4.f32; all values are integers
//    below 2^24) and the last split of a tile to finish writes the outputs;
//  * M > 256: a pre-pass expands the packed weights once per call into a
//    K-major e4m3 operand B [N, K] and the int8 activations into the digit
//    operand A [2M, K] (hi' rows, then lo rows), both in the workspace and
//    largely in L2 during the GEMM (bf16 copies when K < 128);
//  * warp 0, one lane: TMA (cp.async.bulk.tensor.2d, 128-byte swizzle) loads
//    the tiles of each 128-byte K step into a 192 KB ring;
//  * warp 1: allocates 512 TMEM columns (two 256-column fp32
//    accumulators) and one lane issues tcgen05.mma for each stage, releasing
//    the stage with tcgen05.commit;
//  * warps 2-5: tcgen05.ld the finished accumulator (one TMEM lane = one
//    output row per thread), rescale, store; the other accumulator takes the
//    next tile meanwhile.
// Every mbarrier wait is bounded; on time-out the kernel records an error in
// g_device_error, drains what it issued and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "gemm_tc.cuh"

namespace bitnet {

__device__ int g_device_error;

namespace {

constexpr int kBM = 128;
constexpr int kRowBytes = 128;  // K bytes of one row per stage (one swizzle atom)
constexpr int kATileBytes = kBM * kRowBytes;
constexpr int kThreads = 192;       // TMA, MMA, 4 epilogue warps
constexpr int kThreadsFused = 320;  // + 4 warps expanding the packed weights
constexpr uint32_t kTmemCols = 512;
constexpr int kRingBytes = 192 * 1024;
// Tile N = BN (256 or 128): B tile, stage size, ring depth and shared memory.
// Unfused: a TMA stage holds the A and B tiles (the prefill digit form: the
// hi' and lo A tiles and the B tile, 64 KB at BN = 256).  FUSED: a TMA stage holds the
// A tile and the packed 2-bit codes of the B tile (16 bytes per row), and
// the codes are expanded into one of two bf16 B buffers after the ring, so
// the TMA ring is deep (6 stages) while the expanded tiles are only double
// buffered.
// GATED (unfused only): a stage holds the A tile and two B tiles (up and
// gate rows of the same output columns).
// KIND 2 (e4m3 digits, fused only): a stage row holds 128 weights, so the
// packed codes are 32 bytes per row per stage, and three e4m3 B buffers
// follow a 4-stage ring.
template <int BN, bool FUSED = false, bool GATED = false, int KIND = 1>
struct Tile {
  static constexpr int kBTileBytes = BN * kRowBytes;
  static constexpr int kPackedBytes = FUSED ? BN * (KIND == 2 ? 32 : 16) : 0;
  // A bytes per stage: one 128-row tile, two for the prefill digit form
  // (KIND 4: 16 hi and lo digit tiles of the same tokens)
  static constexpr int kABytes = KIND == 4 ? 2 * kATileBytes : kATileBytes;
  static constexpr int kStageBytes =
      kABytes + (FUSED ? kPackedBytes : (GATED ? 2 : 1) * kBTileBytes);
  // expanded B buffers: two (bf16), three (digits: expansion runs on while
  // the MMAs of the two previous stages are in flight)
  static constexpr int kNB = KIND == 2 ? 3 : 2;
  static constexpr int kBBufBytes = FUSED ? kNB * kBTileBytes : 0;
  static constexpr int kStages = (kRingBytes - kBBufBytes) / kStageBytes;  // 4, 6 fused, 4 digits, 3 prefill digits
  static_assert(!FUSED || kStages > kNB, "a ring slot is reused only after its B buffer");
  static constexpr int kSmemBytes = kStages * kStageBytes + kBBufBytes + 1024;  // + alignment
};
constexpr long long kDrainCycles = 2000000000ll;  // bound of the final drains (~1 s)
constexpr int kErrProducer = 1 << 4, kErrMma = 1 << 5, kErrEpilogue = 1 << 6, kErrDrain = 1 << 7;

// Operand element: bf16 (2 bytes), 64 elements of K per 128-byte stage row.
template <int KIND>
struct Kind;
template <>
struct Kind<1> {
  static constexpr int kElem = 2;
  static constexpr int kKStage = kRowBytes / kElem;  // 64 elements per stage
  // Instruction descriptor: D f32 (bits 4-5 = 1), A bf16 (bits 7-9 = 1),
  // B bf16 (bits 10-12 = 1), K-major A and B (bits 15, 16 = 0), M/16 at
  // bits 24-28; N/8 at bits 17-22 is added per tile shape.
  static constexpr uint32_t kIdescBase =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBM >> 4) << 24);
  template <int BN>
  static constexpr uint32_t idesc() { return kIdescBase | ((uint32_t)(BN >> 3) << 17); }
};
// Operand element: e4m3 (1 byte), 128 elements of K per 128-byte stage row
// (the exact digit form, fused path with M <= 64 only).  B holds the ternary
// weights (-1, 0, +1: 0xB8, 0x00, 0x38); the A tile stacks two digit rows
// per token, hi = x >> 4 in [-8, 7] in rows 0-63 and lo = x & 15 in [0, 15]
// in rows 64-127.  Every value is exact in e4m3 and every product and
// partial sum is an integer of magnitude <= 15 K, so the binary32
// accumulators are exact; the epilogue forms acc = 16 D[m] + D[64 + m] in
// int32, which is x . q exactly.
template <>
struct Kind<2> {
  static constexpr int kElem = 1;
  static constexpr int kKStage = kRowBytes / kElem;  // 128 elements per stage
  // Instruction descriptor: D f32 (bits 4-5 = 1), A and B e4m3 (bits 7-9 and
  // 10-12 = 0), K-major, M/16 at bits 24-28; N/8 at bits 17-22 per tile.
  static constexpr uint32_t kIdescBase = (1u << 4) | ((uint32_t)(kBM >> 4) << 24);
  template <int BN>
  static constexpr uint32_t idesc() { return kIdescBase | ((uint32_t)(BN >> 3) << 17); }
};
// The prefill digit form (M > 256): the same e4m3 operands, with the A digits
// hi' = 16 (x >> 4) in [-128, 112] and lo = x & 15 as two 128-row tiles of the
// same tokens, both multiplied into one accumulator, so that it holds
// sum (16 hi + lo) q = sum x q exactly (|partial sums| <= 128 K < 2^24).
template <>
struct Kind<4> : Kind<2> {};
// Every tcgen05.mma consumes 32 bytes of K per row (16 bf16 or 32 e4m3).
constexpr int kMmaKBytes = 32;
// Digit rows: the lo digits of token m sit in A-tile row kDigitRows + m.
constexpr int kDigitRows = 64;

struct Args {
  int M, N, K;
  int m_tiles, n_tiles, k_stages;
  // Split K.  Items below full_tiles are whole tiles (item = tile).  The
  // other tiles, rest = tiles - full_tiles of them, are split: item
  // full_tiles + j is tile full_tiles + j % rest, K stages [s * kps,
  // (s + 1) * kps) of split s = j / rest.  Every split adds its exact partial
  // sums into acc_ws (zeroed by the pre-pass) and the last split of a tile to
  // finish (counted in tile_cnt[tile - full_tiles]) writes the outputs.
  // acc_ws is [M, N] when full_tiles == 0 (every tile split: few output
  // tiles), else one 128 x BN block per split tile (only the tiles of a last,
  // partly filled wave are split, so that the wave keeps every SM busy).
  int splits, kps, full_tiles;
  float* acc_ws;
  int* tile_cnt;
  const float* x_scale;
  const float* w_scale;
  float* y;          // binary32 output, or null (gated: u, optional)
  uint16_t* y_bf16;  // bf16 output, or null
  int32_t* acc_out;
  long long wait;    // bound of every wait but the final drains, in clocks
  // gated (the FFN's up and gate products on one A tile): the gate's scale,
  // its optional binary32 output v, and h = relu(v)^2 * u (required)
  const float* w_scale2;
  float* y2;
  float* h;
  // optional: the bits of each row's max |h| (fmaxf from 0, so never NaN;
  // the non-negative binary32 values order as their bit patterns), combined
  // over the tiles with atomicMax; zeroed before the launch
  unsigned* hmax;
};

// Work item -> tile and K-stage range.
__device__ __forceinline__ void item_range(const Args& a, int item, int& tile, int& ks0, int& ks1) {
  if (item < a.full_tiles) {
    tile = item;
    ks0 = 0;
    ks1 = a.k_stages;
    return;
  }
  const int j = item - a.full_tiles, rest = a.m_tiles * a.n_tiles - a.full_tiles;
  tile = a.full_tiles + j % rest;
  ks0 = (j / rest) * a.kps;
  ks1 = min(a.k_stages, ks0 + a.kps);
}
__device__ __forceinline__ int item_count(const Args& a) {
  return a.full_tiles + (a.m_tiles * a.n_tiles - a.full_tiles) * a.splits;
}

// ---- PTX wrappers (PTX ISA: mbarrier, cp.async.bulk.tensor, tcgen05)
__device__ __forceinline__ uint32_t saddr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
template <int KIND, int BN>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t accumulate) {
  if (KIND == 2 || KIND == 4)
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(Kind<KIND>::template idesc<BN>()), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(Kind<KIND>::template idesc<BN>()), "r"(accumulate)
        : "memory");
}
// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart
// (stride byte offset), start address advanced by 32 bytes per K step inside
// the swizzle atom.  Bits: [0,14) start >> 4, [16,30) leading offset >> 4
// (unused for swizzled K-major), [32,46) stride offset >> 4, [46,48) = 1,
// [61,64) = 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Epilogue warps (2-5): named barrier 2 over their 128 threads, optionally
// OR-reducing a flag (uniform result).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_sync_or(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 2, 128, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)flag)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void red_add_v4(float* p, uint32_t a, uint32_t b, uint32_t c,
                                           uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(__uint_as_float(a)),
               "f"(__uint_as_float(b)), "f"(__uint_as_float(c)), "f"(__uint_as_float(d))
               : "memory");
}
// y = acc * c (binary32 and/or bf16) and the accumulators for 32 consecutive
// outputs of one row.  f holds the accumulators as binary32: exact integers
// below 2^24 in magnitude, so f + 0 (which turns a -0 sum into +0) is the
// binary32 value of the integer, and y = (f + 0) * c is the rescale of it;
// the int32 accumulators are formed only when asked for.  vec4: the 32
// outputs are in range and 16-byte aligned as binary32; vec8: also as bf16.
__device__ __forceinline__ void store_row32(float* yrow, uint16_t* brow, int32_t* arow, int nb,
                                            const float (&f)[32], float c, bool vec4, bool vec8,
                                            int N) {
  if (vec4) {
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      float o[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) o[t] = __fmul_rn(__fadd_rn(f[j + t], 0.0f), c);
      if (yrow) {
        *reinterpret_cast<float4*>(yrow + nb + j) = make_float4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<float4*>(yrow + nb + j + 4) = make_float4(o[4], o[5], o[6], o[7]);
      }
      if (brow) {
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          w[t] = (uint32_t)f32_to_bf16_rn(o[2 * t]) | ((uint32_t)f32_to_bf16_rn(o[2 * t + 1]) << 16);
        if (vec8) {
          *reinterpret_cast<uint4*>(brow + nb + j) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) brow[nb + j + t] = (uint16_t)(w[t >> 1] >> (16 * (t & 1)));
        }
      }
      if (arow) {
        *reinterpret_cast<int4*>(arow + nb + j) =
            make_int4(__float2int_rn(f[j]), __float2int_rn(f[j + 1]), __float2int_rn(f[j + 2]),
                      __float2int_rn(f[j + 3]));
        *reinterpret_cast<int4*>(arow + nb + j + 4) =
            make_int4(__float2int_rn(f[j + 4]), __float2int_rn(f[j + 5]),
                      __float2int_rn(f[j + 6]), __float2int_rn(f[j + 7]));
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (nb + j < N) {
        const float o = __fmul_rn(__fadd_rn(f[j], 0.0f), c);
        if (yrow) yrow[nb + j] = o;
        if (brow) brow[nb + j] = f32_to_bf16_rn(o);
        if (arow) arow[nb + j] = __float2int_rn(f[j]);
      }
  }
}

// Four bf16 values (two words, in order) from four 2-bit codes held in the
// low bits of the bytes of u: code 0, 1, 2 -> q = -1, 0, +1 -> 0xBF80, 0x0000,
// 0x3F80 (exact).  Each code c becomes the byte selectors 4 + c (low byte,
// from the table 0x80, 0x00, 0x80) and c (high byte, from 0xBF, 0x00, 0x3F)
// of one byte permute: u * 0x11 puts c in both nibbles of its byte (no
// carries, c <= 2) and + 0x04 sets the low nibble's table bit.
__device__ __forceinline__ void bf16x4_from_codes(uint32_t u, uint32_t& lo, uint32_t& hi) {
  const uint32_t sel = u * 0x11u + 0x04040404u;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0x003F00BFu), "r"(0x00800080u), "r"(sel));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(0x003F00BFu), "r"(0x00800080u), "r"(sel >> 16));
}

// Expands the packed 2-bit codes of one stage (BN rows x 64 weights, 16
// bytes per row) into the bf16 B tile in the 128-byte-swizzled K-major
// layout the MMA descriptor reads: row r at (r/8)*1024 + (r%8)*128, 16-byte
// chunk c (weights 8c .. 8c+7) at slot c ^ (r%8).  Thread t of 128 takes rows
// t, t+128, ...
template <int BN>
__device__ __forceinline__ void expand_b_tile(uint32_t packed, uint32_t btile, int t) {
  for (int r = t; r < BN; r += 128) {
    uint4 w;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                 : "r"(packed + 16 * r));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    const uint32_t rowbase = btile + (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int sft = 2 * (c >> 1), h = c & 1;
      uint32_t o0, o1, o2, o3;
      bf16x4_from_codes((ww[2 * h] >> sft) & 0x03030303u, o0, o1);
      bf16x4_from_codes((ww[2 * h + 1] >> sft) & 0x03030303u, o2, o3);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(rowbase + 16u * (uint32_t)(c ^ (r & 7))),
                   "r"(o0), "r"(o1), "r"(o2), "r"(o3)
                   : "memory");
    }
  }
}

// Digit form, B side.  Masking a packed word with 0x33333333 leaves one code
// per nibble, and one byte permute over the table {0xB8, 0x00, 0x38} (e4m3 of
// q = -1, 0, +1, selected by code 0, 1, 2) turns four nibbles into four
// weights.  Packed word j of block h (bytes 4j .. 4j+3; byte t holds the
// weights t, 16+t, 32+t, 48+t of the block in bits 0-1, 2-3, 4-5, 6-7)
// becomes the 16-byte chunk c = 4h + j of the stage row, in this order:
// chunk byte 4o + i (o = 0..3, i = 0..3) holds block weight 16g + 4j + b with
// b = 2 (o & 1) + (i >> 1), g = 2 (i & 1) + (o >> 1).  This permutes K inside
// each 64-weight block; the digit pre-pass writes the activations in the same
// order, so every product still pairs x[k] with q[k].
constexpr uint32_t kE4m3Ternary = 0x003800B8u;
__device__ __forceinline__ uint32_t e4m3_lookup(uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(kE4m3Ternary), "r"(0u), "r"(sel));
  return d;
}

// Expands the packed codes of one digit-form stage (BN rows x 128 weights,
// two packed blocks = 32 bytes per row) into the e4m3 B tile in the
// 128-byte-swizzled K-major layout: row r at (r/8)*1024 + (r%8)*128, chunk c
// at slot c ^ (r%8).  Thread t of 128 takes rows t, t+128, ...
template <int BN>
__device__ __forceinline__ void expand_b_tile_e4m3(uint32_t packed, uint32_t btile, int t) {
  for (int r = t; r < BN; r += 128) {
    uint32_t ww[8];
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(ww[0]), "=r"(ww[1]), "=r"(ww[2]), "=r"(ww[3])
                 : "r"(packed + 32 * r));
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(ww[4]), "=r"(ww[5]), "=r"(ww[6]), "=r"(ww[7])
                 : "r"(packed + 32 * r + 16));
    const uint32_t rowbase = btile + (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t u = ww[c] & 0x33333333u, v = (ww[c] >> 2) & 0x33333333u;
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(rowbase + 16u * (uint32_t)(c ^ (r & 7))),
                   "r"(e4m3_lookup(u)), "r"(e4m3_lookup(u >> 16)), "r"(e4m3_lookup(v)),
                   "r"(e4m3_lookup(v >> 16))
                   : "memory");
    }
  }
}

// h = relu(v)^2 * u with t = max(v, 0) taken as v > 0 ? v : 0 (binary32).
__device__ __forceinline__ float relu2_mul(float u, float v) {
  const float t = v > 0.0f ? v : 0.0f;
  return __fmul_rn(__fmul_rn(t, t), u);
}

// 32 consecutive binary32 values of one row; vec4: in range and 16-byte
// aligned.
__device__ __forceinline__ void store_f32_32(float* row, int nb, const float (&v)[32], bool vec4,
                                             int N) {
  if (vec4) {
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      *reinterpret_cast<float4*>(row + nb + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (nb + j < N) row[nb + j] = v[j];
  }
}

template <int KIND, int BN, bool FUSED, bool GATED = false>
__global__ void __launch_bounds__(FUSED ? kThreadsFused : kThreads, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
          const __grid_constant__ CUtensorMap mapB2, const __grid_constant__ Args a) {
  static_assert(!(GATED && FUSED), "the gated form reads expanded bf16 weights");
  static_assert(!GATED || 4 * BN <= (int)kTmemCols, "two accumulators per tile, double buffered");
  static_assert(KIND == 1 || (KIND == 2 && FUSED && !GATED) || (KIND == 4 && !FUSED),
                "digit forms: fused (2) or unfused (4)");
  extern __shared__ uint8_t smem_raw[];
  using T = Tile<BN, FUSED, GATED, KIND>;
  constexpr int kStages = T::kStages;
  constexpr int kStageBytes = T::kStageBytes;
  constexpr int kBTileBytesT = T::kBTileBytes;
  constexpr int kPackedX = Kind<KIND>::kKStage / 4;  // packed bytes of K per stage
  // digit form: the lo digits' sums (TMEM rows 64-127) handed to the threads
  // of rows 0-63, 32 columns at a time (row stride 33: no bank conflicts)
  __shared__ float xbuf[KIND == 2 ? kDigitRows * 33 : 1];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  constexpr int kNB = T::kNB;
  __shared__ __align__(8) uint64_t bready_bar[kNB];  // fused: B buffer expanded
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int s_abort;

  const uint32_t smem0 = (saddr(smem_raw) + 1023u) & ~1023u;  // 1024-byte aligned tiles
  const uint32_t bbuf0 = smem0 + kStages * kStageBytes;        // fused: expanded B buffers
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = item_count(a);
  __shared__ int s_last;
  __shared__ float s_rowscale[kBM];  // split K: the last split's row scales

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(saddr(&full_bar[s]), 1);
      // fused: the four converter warps (packed codes read) and the MMA commit
      mbar_init(saddr(&empty_bar[s]), FUSED ? 5 : 1);
    }
    for (int b = 0; b < kNB; ++b) mbar_init(saddr(&bready_bar[b]), 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(saddr(&acc_full[b]), 1);
      mbar_init(saddr(&acc_empty[b]), 4);
    }
    mbar_init(saddr(&drain_bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_abort = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(&tmem_base_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_slot;
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0, issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
        int t, ks0, ks1;
        item_range(a, item, t, ks0, ks1);
        const int m0 = (t % a.m_tiles) * kBM, n0 = (t / a.m_tiles) * BN;
        for (int ks = ks0; ks < ks1; ++ks, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !mbar_wait(saddr(&empty_bar[s]), ((it / kStages) - 1) & 1, a.wait)) {
            atomicOr(&g_device_error, kErrProducer);
            *(volatile int*)&s_abort = 1;
            ok = false;
            break;
          }
          if (*(volatile int*)&s_abort) {
            ok = false;
            break;
          }
          const uint32_t fb = saddr(&full_bar[s]);
          const uint32_t sa = smem0 + s * kStageBytes;
          if (FUSED) {
            // A tile and the packed codes of the B tile (kPackedX bytes per
            // row = the stage's weights).  bf16: 128 token rows.  Digits
            // (M <= 64, one row tile): the operand is [2M, K], hi digits in
            // rows 0..M-1 and lo digits in rows M..2M-1; a 64-row box from
            // row 0 fills tile rows 0-63 and one from row M fills rows
            // 64-127 (rows past a token's own are padding: their outputs are
            // never stored, and rows past 2M read as zero).
            mbar_expect_tx(fb, kATileBytes + T::kPackedBytes);
            if (KIND == 2) {
              tma_load_2d(sa, &mapA, ks * Kind<KIND>::kKStage, 0, fb);
              tma_load_2d(sa + kDigitRows * kRowBytes, &mapA, ks * Kind<KIND>::kKStage, a.M, fb);
            } else {
              tma_load_2d(sa, &mapA, ks * Kind<KIND>::kKStage, m0, fb);
            }
            tma_load_2d(sa + kATileBytes, &mapB, ks * kPackedX, n0, fb);
          } else {
            // prefill digits: the operand is [2M, K] (hi' rows, then lo
            // rows); the hi' box's rows past M and the lo box's rows past
            // 2M only feed outputs that are never stored
            mbar_expect_tx(fb, kStageBytes);
            tma_load_2d(sa, &mapA, ks * Kind<KIND>::kKStage, m0, fb);
            if (KIND == 4) tma_load_2d(sa + kATileBytes, &mapA, ks * Kind<KIND>::kKStage, a.M + m0, fb);
            tma_load_2d(sa + T::kABytes, &mapB, ks * Kind<KIND>::kKStage, n0, fb);
            if (GATED)
              tma_load_2d(sa + T::kABytes + kBTileBytesT, &mapB2, ks * Kind<KIND>::kKStage, n0, fb);
          }
          issued = it + 1;
        }
      }
      // Never return with a copy in flight.
      for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
        if (!mbar_wait(saddr(&full_bar[j % kStages]), (j / kStages) & 1, kDrainCycles)) {
          atomicOr(&g_device_error, kErrDrain);
          break;
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++lt) {
        int t, ks0, ks1;
        item_range(a, item, t, ks0, ks1);
        (void)t;
        const int ab = lt & 1;
        if (lt >= 2 && !mbar_wait(saddr(&acc_empty[ab]), ((lt >> 1) - 1) & 1, a.wait)) {
          atomicOr(&g_device_error, kErrMma);
          *(volatile int*)&s_abort = 1;
          break;
        }
        tc_fence_after();
        // gated: the tile's u accumulator, its v accumulator BN columns on
        const uint32_t d = tmem + (uint32_t)(ab * (GATED ? 2 : 1) * BN);
        for (int ks = ks0; ks < ks1; ++ks, ++it) {
          const int s = it % kStages, b = it % kNB;
          // fused: the expanded B buffer (and the A tile of the stage, whose
          // landing the converters waited for and which is checked again)
          bool ready = mbar_wait(saddr(&full_bar[s]), (it / kStages) & 1, a.wait);
          if (FUSED && ready) ready = mbar_wait(saddr(&bready_bar[b]), (it / kNB) & 1, a.wait);
          if (!ready || *(volatile int*)&s_abort) {
            atomicOr(&g_device_error, kErrMma);
            *(volatile int*)&s_abort = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem0 + s * kStageBytes;
          const uint32_t sb = FUSED ? bbuf0 + b * kBTileBytesT : sa + T::kABytes;
#pragma unroll
          for (int kk = 0; kk < kRowBytes / kMmaKBytes; ++kk) {
            const uint64_t ad = sw128_desc(sa + kk * kMmaKBytes);
            const uint64_t bd = sw128_desc(sb + kk * kMmaKBytes);
            tc_mma<KIND, BN>(d, ad, bd, (ks != ks0 || kk != 0) ? 1u : 0u);
            if (KIND == 4) tc_mma<KIND, BN>(d, sw128_desc(sa + kATileBytes + kk * kMmaKBytes), bd, 1u);
            if (GATED) {
              const uint64_t bd2 = sw128_desc(sb + kBTileBytesT + kk * kMmaKBytes);
              tc_mma<KIND, BN>(d + (uint32_t)BN, ad, bd2, (ks != ks0 || kk != 0) ? 1u : 0u);
              if (KIND == 4)
                tc_mma<KIND, BN>(d + (uint32_t)BN, sw128_desc(sa + kATileBytes + kk * kMmaKBytes),
                                 bd2, 1u);
            }
          }
          // frees the stage, and (fused) the expanded B buffer, when these
          // MMAs finish: one commit per stage
          tc_commit(saddr(&empty_bar[s]));
        }
        if (!ok) break;
        tc_commit(saddr(&acc_full[ab]));    // accumulator ready for the epilogue
      }
      // All MMAs issued by this thread have finished before TMEM is freed.
      tc_commit(saddr(&drain_bar));
      if (!mbar_wait(saddr(&drain_bar), 0, kDrainCycles)) atomicOr(&g_device_error, kErrDrain);
    }
  } else if (FUSED && warp >= 6) {
    // ------------------------------------------------------------ B expansion
    const int ct = threadIdx.x - 6 * 32;  // 0 .. 127
    int it = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
      int t, ks0, ks1;
      item_range(a, item, t, ks0, ks1);
      (void)t;
      bool ok = true;
      for (int ks = ks0; ks < ks1; ++ks, ++it) {
        const int s = it % kStages, b = it % kNB;
        bool ready = mbar_wait(saddr(&full_bar[s]), (it / kStages) & 1, a.wait);
        // the MMAs of kNB stages ago (which read buffer b) have finished: that
        // stage's ring slot was released, by them and by these warps (the slot
        // cannot have been released again since: kStages > kNB, and the next
        // use of it needs these warps' arrival at a later stage)
        if (ready && it >= kNB)
          ready = mbar_wait(saddr(&empty_bar[(it - kNB) % kStages]), ((it - kNB) / kStages) & 1,
                            a.wait);
        if (!ready || *(volatile int*)&s_abort) {
          if (lane == 0) atomicOr(&g_device_error, kErrProducer);
          *(volatile int*)&s_abort = 1;
          ok = false;
          break;
        }
        const uint32_t sa = smem0 + s * kStageBytes;
        if (KIND == 2)
          expand_b_tile_e4m3<BN>(sa + kATileBytes, bbuf0 + b * kBTileBytesT, ct);
        else
          expand_b_tile<BN>(sa + kATileBytes, bbuf0 + b * kBTileBytesT, ct);
        // make the generic-proxy stores visible to the tensor core's reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(saddr(&bready_bar[b]));
          mbar_arrive(saddr(&empty_bar[s]));  // the packed codes are read
        }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const float ws = *a.w_scale;
    const float ws2 = GATED ? *a.w_scale2 : 0.0f;
    int lt = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x, ++lt) {
      int t, ks0, ks1;
      item_range(a, item, t, ks0, ks1);
      const int ab = lt & 1;
      const bool bad =
          !mbar_wait(saddr(&acc_full[ab]), (lt >> 1) & 1, a.wait) || *(volatile int*)&s_abort;
      if (epi_sync_or(bad)) {  // uniform over the epilogue warps
        if (lane == 0) atomicOr(&g_device_error, kErrEpilogue);
        *(volatile int*)&s_abort = 1;
        break;
      }
      tc_fence_after();
      const int m0 = (t % a.m_tiles) * kBM, n0 = (t / a.m_tiles) * BN;
      const int m = m0 + row;
      const bool mrow = m < a.M;
      const float c = mrow ? __fmul_rn(a.x_scale[m], ws) : 0.0f;
      float* yrow = a.y ? a.y + (int64_t)m * a.N : nullptr;
      uint16_t* brow = a.y_bf16 ? a.y_bf16 + (int64_t)m * a.N : nullptr;
      int32_t* arow = a.acc_out ? a.acc_out + (int64_t)m * a.N : nullptr;
      const bool split_tile = a.splits > 1 && t >= a.full_tiles;
      // (acc_ws + row * BN - n0 + nb) addresses the tile's own block
      float* wrow = a.full_tiles > 0
                        ? a.acc_ws + ((int64_t)(t - a.full_tiles) * kBM + row) * BN - n0
                        : a.acc_ws + (int64_t)m * a.N;
      const bool vec = (a.N & 3) == 0;
      const bool vec8 = (a.N & 7) == 0;
      if (GATED) {
        // u = f32(acc_u) * (sx * s_up), v = f32(acc_v) * (sx * s_gate),
        // h = relu(v)^2 * u; the accumulators are exact integers (adding +0
        // turns a -0 sum into the +0 of the integer's conversion)
        const float cv = mrow ? __fmul_rn(a.x_scale[m], ws2) : 0.0f;
        float* vrow = a.y2 ? a.y2 + (int64_t)m * a.N : nullptr;
        float* hrow = a.h + (int64_t)m * a.N;
        float hm = 0.0f;
        for (int cb = 0; cb < BN; cb += 32) {
          uint32_t ru[32], rv[32];
          const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ab * 2 * BN + cb);
          tmem_ld32(ta, ru);
          tmem_ld32(ta + (uint32_t)BN, rv);
          if (!mrow) continue;
          const int nb = n0 + cb;
          float uf[32], vf[32], hf[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            uf[j] = __fmul_rn(__fadd_rn(__uint_as_float(ru[j]), 0.0f), c);
            vf[j] = __fmul_rn(__fadd_rn(__uint_as_float(rv[j]), 0.0f), cv);
            hf[j] = relu2_mul(uf[j], vf[j]);
          }
          const bool v4 = vec && nb + 32 <= a.N;
          if (yrow) store_f32_32(yrow, nb, uf, v4, a.N);
          if (vrow) store_f32_32(vrow, nb, vf, v4, a.N);
          store_f32_32(hrow, nb, hf, v4, a.N);
          if (a.hmax) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (nb + j < a.N) hm = fmaxf(hm, fabsf(hf[j]));
          }
        }
        if (a.hmax && mrow) atomicMax(a.hmax + m, __float_as_uint(hm));
      }
      for (int cb = 0; cb < BN && !GATED; cb += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ab * BN + cb), r);
        if (KIND == 2) {
          // acc = 16 * (hi digits' sum, row m) + (lo digits' sum, row 64 + m):
          // exact integers in binary32, combined in int32.  Rows >= 64 (and
          // so >= M) only hand their sums over.
          float* xb = xbuf + (row & (kDigitRows - 1)) * 33;
          if (row >= kDigitRows) {
#pragma unroll
            for (int j = 0; j < 32; ++j) xb[j] = __uint_as_float(r[j]);
          }
          epi_sync();
          if (row < kDigitRows) {
            // 16 D[m] + D[64 + m]: integers below 2^24, so the fused
            // multiply-add is exact
#pragma unroll
            for (int j = 0; j < 32; ++j)
              r[j] = __float_as_uint(__fmaf_rn(16.0f, __uint_as_float(r[j]), xb[j]));
          }
          epi_sync();
        }
        if (!mrow) continue;
        const int nb = n0 + cb;
        if (split_tile) {
          // Add this split's exact partial sums (integers below 2^24 in
          // magnitude, whatever the order: fp32 addition is exact here).
          if (vec && nb + 32 <= a.N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              red_add_v4(wrow + nb + j, r[j], r[j + 1], r[j + 2], r[j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (nb + j < a.N) atomicAdd(wrow + nb + j, __uint_as_float(r[j]));
          }
          continue;
        }
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]);  // exact integers
        store_row32(yrow, brow, arow, nb, f, c, vec && nb + 32 <= a.N, vec8, a.N);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(saddr(&acc_empty[ab]));
      if (split_tile) {
        // The last split of the tile to finish writes the outputs.
        __threadfence();
        epi_sync();
        if (threadIdx.x == 64) s_last = atomicAdd(&a.tile_cnt[t - a.full_tiles], 1) == a.splits - 1;
        epi_sync();
        if (s_last) {
          __threadfence();
          // The 128 epilogue threads sweep the tile's sums together, four
          // columns per step (16-byte loads and stores when N % 4 == 0), eight
          // steps' loads in flight per thread; the rows' scales are staged in
          // shared memory first.
          const int et = threadIdx.x - 64;  // epilogue warps 2-5
          const int rows = min(kBM, a.M - m0), cols = min(BN, a.N - n0);
          const int g4 = (cols + 3) >> 2, total = rows * g4;
          if (et < rows) s_rowscale[et] = __fmul_rn(a.x_scale[m0 + et], ws);
          epi_sync();
          for (int i0 = et; i0 < total; i0 += 128 * 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int i = i0 + 128 * u;
              v[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              if (i < total) {
                const int rr = i / g4, cc = (i - rr * g4) * 4;
                const float* src = a.full_tiles > 0
                                       ? a.acc_ws + ((int64_t)(t - a.full_tiles) * kBM + rr) * BN + cc
                                       : a.acc_ws + (int64_t)(m0 + rr) * a.N + n0 + cc;
                if (vec) {
                  v[u] = __ldcg(reinterpret_cast<const float4*>(src));
                } else {
                  v[u].x = __ldcg(src);
                  if (n0 + cc + 1 < a.N) v[u].y = __ldcg(src + 1);
                  if (n0 + cc + 2 < a.N) v[u].z = __ldcg(src + 2);
                  if (n0 + cc + 3 < a.N) v[u].w = __ldcg(src + 3);
                }
              }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int i = i0 + 128 * u;
              if (i >= total) break;
              const int rr = i / g4, cc = (i - rr * g4) * 4;
              const int mm = m0 + rr, n = n0 + cc;
              const float cm = s_rowscale[rr];
              const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
              float o[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) o[j] = __fmul_rn(__fadd_rn(f[j], 0.0f), cm);
              const int64_t off = (int64_t)mm * a.N + n;
              if (vec) {
                if (a.y) *reinterpret_cast<float4*>(a.y + off) = make_float4(o[0], o[1], o[2], o[3]);
                if (a.y_bf16)
                  *reinterpret_cast<uint2*>(a.y_bf16 + off) =
                      make_uint2((uint32_t)f32_to_bf16_rn(o[0]) | ((uint32_t)f32_to_bf16_rn(o[1]) << 16),
                                 (uint32_t)f32_to_bf16_rn(o[2]) | ((uint32_t)f32_to_bf16_rn(o[3]) << 16));
                if (a.acc_out)
                  *reinterpret_cast<int4*>(a.acc_out + off) =
                      make_int4(__float2int_rn(f[0]), __float2int_rn(f[1]), __float2int_rn(f[2]),
                                __float2int_rn(f[3]));
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  if (n + j < a.N) {
                    if (a.y) a.y[off + j] = o[j];
                    if (a.y_bf16) a.y_bf16[off + j] = f32_to_bf16_rn(o[j]);
                    if (a.acc_out) a.acc_out[off + j] = __float2int_rn(f[j]);
                  }
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// Two e4m3 bytes (a0 in the low byte) of two small integers, exact: the
// conversion instruction puts its first source in the high byte.
__device__ __forceinline__ uint32_t e4m3x2_of(int a0, int a1) {
  unsigned short d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(__int2float_rn(a1)),
      "f"(__int2float_rn(a0)));
  return d;
}
// The e4m3 digits hi = (x >> 4) * hs (hs = 1 or 16) and lo = x & 15 of the
// four int8 values in w.
__device__ __forceinline__ void digits4(uint32_t w, int hs, uint32_t& hi, uint32_t& lo) {
  int x[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) x[b] = (int)(int8_t)(w >> (8 * b));
  hi = e4m3x2_of((x[0] >> 4) * hs, (x[1] >> 4) * hs) |
       (e4m3x2_of((x[2] >> 4) * hs, (x[3] >> 4) * hs) << 16);
  lo = e4m3x2_of(x[0] & 15, x[1] & 15) | (e4m3x2_of(x[2] & 15, x[3] & 15) << 16);
}
// Four e4m3 weights (one word, in order) from the four 2-bit codes in bits
// 0-1 of the bytes of v (higher bits ignored): code 0, 1, 2 -> q = -1, 0,
// +1 -> 0xB8, 0x00, 0x38.  Bit 0 of a code is clear exactly when q != 0, and
// both bits are clear exactly when q = -1.
__device__ __forceinline__ uint32_t e4m3x4_from_codes(uint32_t v) {
  const uint32_t nz = ~v & 0x01010101u;
  const uint32_t neg = ~(v | (v >> 1)) & 0x01010101u;
  return nz * 0x38u + (neg << 7);
}

// ---- pre-pass kernel
// One launch.  Items, in order:
//  * B (nblk packed 64-weight blocks): bf16 mode, eight 16-byte chunks of 8
//    weights per block (chunk c = field c/2 of words 2(c%2), 2(c%2)+1); e4m3
//    mode, four 16-byte chunks of 16 weights (chunk c = field c of the
//    block's 16 bytes, in byte order).  Consecutive threads write
//    consecutive chunks.
//  * A (nx groups of 16 int8 activations):
//    - kABf16: 32 bytes of bf16;
//    - kADigitsFused: the e4m3 digits hi = x >> 4 (16 bytes at A[i]) and
//      lo = x & 15 (at A[digit_lo + i]), x = 16 hi + lo, in the K order of
//      the on-chip e4m3 expansion: chunk j of a 64-wide block takes the
//      activations 16g + 4j + b (g, b = 0..3) of that block, as four words
//      X_g of four, and places X_g byte b at chunk byte 4o + i with
//      b = 2 (o & 1) + (i >> 1), g = 2 (i & 1) + (o >> 1): the byte permutes
//      (X0, X2 | X1, X3 by 0x5140 | 0x7362);
//    - kADigitsPrefill: hi' = 16 (x >> 4) and lo = x & 15, in K order;
//    - kADigitsFromF32: the same digits of x = the per-token int8 codes of
//      the binary32 rows hf, quantised with the rule of the activation
//      quantiser (scale from the row's max |hf| in hmax, inv = 127 / a',
//      x = round_clip(hf * inv)); the item that starts a row writes its
//      scale, and the codes also go to hq when asked.
//  * nz 16-byte zero stores (split-K sums and tile counters).
enum AMode { kABf16 = 0, kADigitsFused = 1, kADigitsPrefill = 2, kADigitsFromF32 = 3 };
struct Prep {
  const uint4* Wq;
  int64_t nblk;
  uint4* B;
  const uint4* Wq2;  // optional second matrix of the same shape (into B2)
  uint4* B2;
  int b_e4m3;
  const uint4* xq;
  int64_t nx;
  uint4* A;
  int a_mode;
  int64_t digit_lo, K;
  uint4* zero;
  int64_t nz;
  // kADigitsFromF32
  const float4* hf;
  const unsigned* hmax;
  float* sh;
  uint4* hq;
};
__global__ void __launch_bounds__(256) k_prepass(const Prep p) {
  const int64_t per = (p.b_e4m3 ? 4 : 8) * p.nblk;
  const int64_t nbi = per * (p.Wq2 ? 2 : 1);
  const int64_t total = nbi + p.nx + p.nz;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (int64_t)gridDim.x * blockDim.x) {
    if (it < nbi) {
      const bool second = it >= per;
      const uint4* Wq = second ? p.Wq2 : p.Wq;
      uint4* B = second ? p.B2 : p.B;
      const int64_t jt = second ? it - per : it;
      if (p.b_e4m3) {
        const uint4 w = Wq[jt >> 2];  // the 4 threads of a block share this load
        const int sft = 2 * (int)(jt & 3);
        B[jt] = make_uint4(e4m3x4_from_codes(w.x >> sft), e4m3x4_from_codes(w.y >> sft),
                           e4m3x4_from_codes(w.z >> sft), e4m3x4_from_codes(w.w >> sft));
      } else {
        const uint4 w = Wq[jt >> 3];  // the 8 threads of a block share this load
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        const int c = (int)(jt & 7), sft = 2 * (c >> 1), h = c & 1;
        uint4 o;
        bf16x4_from_codes((ww[2 * h] >> sft) & 0x03030303u, o.x, o.y);
        bf16x4_from_codes((ww[2 * h + 1] >> sft) & 0x03030303u, o.z, o.w);
        B[jt] = o;
      }
    } else if (it >= nbi + p.nx) {
      p.zero[it - nbi - p.nx] = make_uint4(0, 0, 0, 0);
    } else if (p.a_mode == kADigitsFused) {
      const int64_t i = it - nbi;
      const int64_t f = 16 * i, off = f % p.K;  // flat start, offset in its row
      // word index of activation (f - off) + (off & ~63) + 4j, j = chunk in block
      const uint32_t* xw = reinterpret_cast<const uint32_t*>(p.xq) +
                           (f - off + (off & ~63ll)) / 4 + ((off >> 4) & 3);
      const uint32_t X0 = xw[0], X1 = xw[4], X2 = xw[8], X3 = xw[12];
      const uint32_t P[4] = {__byte_perm(X0, X2, 0x5140), __byte_perm(X0, X2, 0x7362),
                             __byte_perm(X1, X3, 0x5140), __byte_perm(X1, X3, 0x7362)};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) digits4(P[q], 1, hi[q], lo[q]);
      p.A[i] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      p.A[p.digit_lo + i] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else if (p.a_mode == kADigitsFromF32) {
      const int64_t i = it - nbi;
      const int64_t f = 16 * i, m = f / p.K;
      const ActScale sc = act_scale_from_absmax(__uint_as_float(p.hmax[m]));
      if (f - m * p.K == 0) p.sh[m] = sc.scale;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = p.hf[4 * i + q];
        w[q] = pack_i8x4(round_clip(__fmul_rn(v.x, sc.inv), -128.f, 127.f),
                         round_clip(__fmul_rn(v.y, sc.inv), -128.f, 127.f),
                         round_clip(__fmul_rn(v.z, sc.inv), -128.f, 127.f),
                         round_clip(__fmul_rn(v.w, sc.inv), -128.f, 127.f));
      }
      if (p.hq) p.hq[i] = make_uint4(w[0], w[1], w[2], w[3]);
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) digits4(w[q], 16, hi[q], lo[q]);
      p.A[i] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      p.A[p.digit_lo + i] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else if (p.a_mode == kADigitsPrefill) {
      const int64_t i = it - nbi;
      const uint4 v = p.xq[i];
      const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) digits4(vv[q], 16, hi[q], lo[q]);
      p.A[i] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      p.A[p.digit_lo + i] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else {
      const int64_t i = it - nbi;
      const uint4 v = p.xq[i];
      const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
      uint32_t h[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // |x| <= 128 has at most 8 significant bits: the binary32 value's
        // low 16 bits are zero and its top half is the exact bf16.
        const uint32_t b0 = __float_as_uint(__int2float_rn((int)(int8_t)(vv[q] & 0xffu))) >> 16;
        const uint32_t b1 = __float_as_uint(__int2float_rn((int)(int8_t)((vv[q] >> 8) & 0xffu))) >> 16;
        const uint32_t b2 = __float_as_uint(__int2float_rn((int)(int8_t)((vv[q] >> 16) & 0xffu))) >> 16;
        const uint32_t b3 = __float_as_uint(__int2float_rn((int)(int8_t)(vv[q] >> 24))) >> 16;
        h[2 * q] = b0 | (b1 << 16);
        h[2 * q + 1] = b2 | (b3 << 16);
      }
      p.A[2 * i] = make_uint4(h[0], h[1], h[2], h[3]);
      p.A[2 * i + 1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

// ---- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mutex;

cudaError_t get_encode() {
  std::lock_guard<std::mutex> lock(g_encode_mutex);
  if (g_encode) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

// Packed weights [N, K/4] bytes as a 2-D uint8 tensor, boxes of box_bytes
// (16 or 32: 64 or 128 weights) x box_rows, no swizzle.
cudaError_t encode_packed(CUtensorMap* map, const void* Wq, int64_t N, int64_t K, int box_bytes,
                          int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)(K / 4), (cuuint64_t)N};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 4)};
  cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(Wq), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D K-major operand [rows, K], boxes of (128 bytes of K) x box_rows.
cudaError_t encode_operand(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                           int elem_bytes, int box_rows) {
  const CUtensorMapDataType dt =
      elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(K * elem_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / elem_bytes), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Operand kind used for the tensor-core path (bf16; see the top of the file).
constexpr int kKind = 1;

size_t round1k(size_t v) { return (v + 1023) / 1024 * 1024; }

// Small batches expand the packed weights on chip (streaming 2 bits per
// weight from HBM); large ones expand them once into an e4m3 (or bf16) copy
// that stays largely in L2 across the many output-tile rows.
bool use_fused(int64_t M) { return M <= 256; }
// The exact e4m3 digit form (two digit rows per token in one 128-row tile)
// serves M <= 64 on the fused path: half the MMAs of the bf16 form and
// 128-deep K stages.
bool use_digits(int64_t M, int64_t K) { return M <= 64 && K >= 128; }
// The prefill digit form (M > 256): e4m3 weights and the two digit tiles of
// the activations move 64 KB per 128-deep K step of a 128 x 256 tile, where
// bf16 moves 96 KB, at the same tensor time.
bool use_prefill_digits(int64_t M, int64_t K) { return M > 256 && K >= 128; }

// Tile N.  128-wide tiles fill the last wave of 148 SMs better for some
// shapes, but they stream the bf16 A operand twice as often from L2; measured
// on B300 (M = 4096, K = 6912, N = 2560) they lose (237 us vs 192 us), so
// the 256-wide tile is used unless N itself is narrow (fused: always 256).
int pick_bn(int64_t N) { return N <= 128 ? 128 : 256; }

// Workspace of one call: [B bf16 N x K (unfused only)] [A bf16 M x K]
// [split-K sums] [tile counters], each 1 KB aligned.  Split K:
//  * fused path, when the output has fewer tiles than half the SMs: every
//    tile, in as many splits as fill the SMs (each at least 16 K stages of
//    64, or 4 of 128 in the digit form); sums M x N fp32;
//  * unfused path, when the output is at most three waves of whole tiles
//    plus a last wave that would fill less than half the SMs: only that
//    wave's tiles, in as many splits as fill the SMs (each at least 16 K
//    stages); one 128 x BN fp32 block per split tile.  Measured on B300:
//    M = 4096, K = 6912, N = 2560 (two waves + 24 tiles) 167 -> 161 us;
//    K = 14336, N = 4096 (three waves + 68 tiles) 410 -> 399 us; with twelve
//    waves + 16 tiles (K = 4096, N = 14336) splitting lost 3%.
struct WsLayout {
  size_t b, a, acc, cnt, end;
  int splits, kps, full_tiles;
};
WsLayout ws_layout(int64_t M, int64_t N, int64_t K) {
  WsLayout L = {};
  const bool fused = use_fused(M);
  const int bn = fused ? 256 : pick_bn(N);
  const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
  const bool digits = fused && use_digits(M, K);
  const bool pdigits = !fused && use_prefill_digits(M, K);
  const int k_stages = (int)((K + (digits || pdigits ? 127 : 63)) / (digits || pdigits ? 128 : 64));
  // fewest K stages per split: 4 (512 K) in the digit form, 16 (1024 K) in
  // bf16; measured on B300 (digit form, N x K = 2560 x 2560 .. 2560 x 6912,
  // M = 16 / 64): 4 stages 13-15 / 22-23 us, 16 stages 19-22 / 22-30 us
  const int min_split_stages = digits ? 4 : 16;
  int splits = 1;
  int64_t split_tiles = tiles;  // tiles that are split when splits > 1
  L.full_tiles = 0;
  if (fused && tiles < 74) {
    splits = (int)(148 / tiles);
    if (splits > k_stages / min_split_stages) splits = k_stages / min_split_stages;
    if (splits < 1) splits = 1;
  } else if (!fused && tiles > 148 && tiles < 4 * 148 && tiles % 148 < 74) {
    const int64_t rem = tiles % 148;
    const int min_stages = pdigits ? 8 : 16;  // 1024 K
    splits = (int)(148 / rem);
    if (splits > k_stages / min_stages) splits = k_stages / min_stages;
    if (splits < 2) splits = 1;
    if (splits > 1) {
      L.full_tiles = (int)(tiles - rem);
      split_tiles = rem;
    }
  }
  L.kps = (k_stages + splits - 1) / splits;
  L.splits = (k_stages + L.kps - 1) / L.kps;
  if (L.splits < 2) L.full_tiles = 0;
  L.b = 0;
  L.a = fused ? 0 : round1k((size_t)(N * K * (pdigits ? 1 : 2)));
  L.acc = L.a + round1k((size_t)(M * K * 2));
  const size_t sums = L.full_tiles > 0 ? (size_t)split_tiles * kBM * bn * 4 : (size_t)(M * N * 4);
  L.cnt = L.acc + (L.splits > 1 ? round1k(sums) : 0);
  L.end = L.cnt + (L.splits > 1 ? round1k((size_t)split_tiles * 4) : 0);
  return L;
}

// The activations as binary32 rows to quantise in the pre-pass (the FFN's h
// before the down projection), with their row maxima; the int8 codes (hq,
// optional) and scales (sh) are written there too.
struct FromF32 {
  const float* h;
  const unsigned* hmax;
  int8_t* hq;
  float* sh;
};

template <int KIND, int BN, bool FUSED>
cudaError_t launch_kind(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                        const float* x_scale, int64_t M, int64_t N, int64_t K, float* y,
                        uint16_t* y_bf16, int32_t* acc_out, void* ws, long long wait,
                        cudaStream_t s, const FromF32* ff = nullptr) {
  if (ff && KIND != 4) return cudaErrorInvalidValue;
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  const WsLayout L = ws_layout(M, N, K);
  uint8_t* w = static_cast<uint8_t*>(ws);
  void* B = w + L.b;
  void* A = w + L.a;
  float* acc_ws = reinterpret_cast<float*>(w + L.acc);
  int* tile_cnt = reinterpret_cast<int*>(w + L.cnt);
  const int64_t nblk = FUSED ? 0 : N * K / 64, nx = M * K / 16;
  const int64_t nz = L.splits > 1 ? (int64_t)(L.end - L.acc) / 16 : 0;
  Prep pp;
  pp.Wq = reinterpret_cast<const uint4*>(Wq);
  pp.nblk = nblk;
  pp.B = reinterpret_cast<uint4*>(B);
  pp.Wq2 = nullptr;
  pp.B2 = nullptr;
  pp.b_e4m3 = KIND == 4;
  pp.xq = reinterpret_cast<const uint4*>(xq);
  pp.nx = nx;
  pp.A = reinterpret_cast<uint4*>(A);
  pp.a_mode = KIND == 2 ? kADigitsFused : KIND == 4 ? kADigitsPrefill : kABf16;
  pp.digit_lo = nx;
  pp.K = K;
  pp.zero = reinterpret_cast<uint4*>(w + L.acc);
  pp.nz = nz;
  pp.hf = nullptr;
  pp.hmax = nullptr;
  pp.sh = nullptr;
  pp.hq = nullptr;
  if (ff) {
    pp.a_mode = kADigitsFromF32;
    pp.hf = reinterpret_cast<const float4*>(ff->h);
    pp.hmax = ff->hmax;
    pp.sh = ff->sh;
    pp.hq = reinterpret_cast<uint4*>(ff->hq);
    x_scale = ff->sh;
  }
  int64_t grid = ((KIND == 4 ? 4 : 8) * nblk + nx + nz + 255) / 256;
  if (grid > 148 * 16) grid = 148 * 16;
  k_prepass<<<(unsigned)grid, 256, 0, s>>>(pp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mapA, mapB;
  // digits: [2M, K] e4m3 (hi rows, then lo rows), 64-row boxes (fused) or
  // 128-row boxes (prefill)
  e = KIND == 2   ? encode_operand(&mapA, A, 2 * M, K, 1, kDigitRows)
      : KIND == 4 ? encode_operand(&mapA, A, 2 * M, K, 1, kBM)
                  : encode_operand(&mapA, A, M, K, Kind<KIND>::kElem, kBM);
  if (e == cudaSuccess)
    e = FUSED ? encode_packed(&mapB, Wq, N, K, Kind<KIND>::kKStage / 4, BN)
              : encode_operand(&mapB, B, N, K, Kind<KIND>::kElem, BN);
  if (e != cudaSuccess) return e;
  Args a;
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.m_tiles = (int)((M + kBM - 1) / kBM);
  a.n_tiles = (int)((N + BN - 1) / BN);
  a.k_stages = (int)((K + Kind<KIND>::kKStage - 1) / Kind<KIND>::kKStage);
  a.splits = L.splits;
  a.kps = L.kps;
  a.full_tiles = L.full_tiles;
  a.acc_ws = acc_ws;
  a.tile_cnt = tile_cnt;
  a.x_scale = x_scale;
  a.w_scale = w_scale;
  a.y = y;
  a.y_bf16 = y_bf16;
  a.acc_out = acc_out;
  a.wait = wait;
  a.w_scale2 = nullptr;
  a.y2 = nullptr;
  a.h = nullptr;
  a.hmax = nullptr;
  static bool configured[64] = {};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(k_gemm_tc<KIND, BN, FUSED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Tile<BN, FUSED, false, KIND>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int items = a.full_tiles + (a.m_tiles * a.n_tiles - a.full_tiles) * a.splits;
  const int ctas = items < 148 ? items : 148;
  return launch_pdl(k_gemm_tc<KIND, BN, FUSED>, dim3(ctas),
                    dim3(FUSED ? kThreadsFused : kThreads),
                    (size_t)Tile<BN, FUSED, false, KIND>::kSmemBytes, s, mapA, mapB, mapB, a);
}

// The FFN's up and gate products in one GEMM (M > 256): both weight matrices
// are expanded once per call (e4m3, or bf16 when K < 128) and the
// activations split into digits (or widened to bf16), and k_gemm_tc<..,
// GATED> runs 128 x 128 output tiles with two accumulators each (u and v on
// the same A tiles), writing h = relu(v)^2 * u, optionally each row's max
// |h|, and, when asked, u and v.  Workspace: [B up][B gate][A], each 1 KB
// aligned.
size_t gated_ws(int64_t M, int64_t N, int64_t K) {
  const size_t wb = use_prefill_digits(M, K) ? 1 : 2;
  return 2 * round1k((size_t)(N * K * wb)) + round1k((size_t)(M * K * 2));
}

template <int KIND>
cudaError_t launch_gated_t(const uint8_t* Wu, const float* su, const uint8_t* Wg, const float* sg,
                           const int8_t* xq, const float* x_scale, int64_t M, int64_t N,
                           int64_t K, float* u, float* v, float* h, unsigned* hmax, void* ws,
                           long long wait, cudaStream_t s) {
  constexpr int BN = 128;
  constexpr size_t kWb = KIND == 4 ? 1 : 2;  // bytes per expanded weight
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  uint8_t* w = static_cast<uint8_t*>(ws);
  void* Bu = w;
  void* Bg = w + round1k((size_t)(N * K) * kWb);
  void* A = w + 2 * round1k((size_t)(N * K) * kWb);
  const int64_t nblk = N * K / 64, nx = M * K / 16;
  // one pre-pass: both weight matrices, the activations, and (when asked)
  // the zeroed row maxima of h
  Prep pp = {};
  pp.Wq = reinterpret_cast<const uint4*>(Wu);
  pp.nblk = nblk;
  pp.B = reinterpret_cast<uint4*>(Bu);
  pp.Wq2 = reinterpret_cast<const uint4*>(Wg);
  pp.B2 = reinterpret_cast<uint4*>(Bg);
  pp.b_e4m3 = KIND == 4;
  pp.xq = reinterpret_cast<const uint4*>(xq);
  pp.nx = nx;
  pp.A = reinterpret_cast<uint4*>(A);
  pp.a_mode = KIND == 4 ? kADigitsPrefill : kABf16;
  pp.digit_lo = nx;
  pp.K = K;
  pp.zero = reinterpret_cast<uint4*>(hmax);
  pp.nz = hmax ? (M + 3) / 4 : 0;
  int64_t grid = (2 * (KIND == 4 ? 4 : 8) * nblk + nx + pp.nz + 255) / 256;
  if (grid > 148 * 16) grid = 148 * 16;
  k_prepass<<<(unsigned)grid, 256, 0, s>>>(pp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mapA, mapB, mapB2;
  e = KIND == 4 ? encode_operand(&mapA, A, 2 * M, K, 1, kBM)
                : encode_operand(&mapA, A, M, K, Kind<KIND>::kElem, kBM);
  if (e == cudaSuccess) e = encode_operand(&mapB, Bu, N, K, Kind<KIND>::kElem, BN);
  if (e == cudaSuccess) e = encode_operand(&mapB2, Bg, N, K, Kind<KIND>::kElem, BN);
  if (e != cudaSuccess) return e;
  Args a = {};
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.m_tiles = (int)((M + kBM - 1) / kBM);
  a.n_tiles = (int)((N + BN - 1) / BN);
  a.k_stages = (int)((K + Kind<KIND>::kKStage - 1) / Kind<KIND>::kKStage);
  a.splits = 1;
  a.kps = a.k_stages;
  a.full_tiles = 0;
  a.acc_ws = nullptr;
  a.tile_cnt = nullptr;
  a.x_scale = x_scale;
  a.w_scale = su;
  a.y = u;
  a.y_bf16 = nullptr;
  a.acc_out = nullptr;
  a.wait = wait;
  a.w_scale2 = sg;
  a.y2 = v;
  a.h = h;
  a.hmax = hmax;
  static bool configured[64] = {};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(k_gemm_tc<KIND, BN, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Tile<BN, false, true, KIND>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int items = a.m_tiles * a.n_tiles;
  const int ctas = items < 148 ? items : 148;
  return launch_pdl(k_gemm_tc<KIND, BN, false, true>, dim3(ctas), dim3(kThreads),
                    (size_t)Tile<BN, false, true, KIND>::kSmemBytes, s, mapA, mapB, mapB2, a);
}

}  // namespace

size_t gemm_tc_gated_workspace(int64_t M, int64_t N, int64_t K) { return gated_ws(M, N, K); }

cudaError_t launch_gemm_tc_gated(const uint8_t* Wu, const float* su, const uint8_t* Wg,
                                 const float* sg, const int8_t* xq, const float* x_scale,
                                 int64_t M, int64_t N, int64_t K, float* u, float* v, float* h,
                                 unsigned* hmax, void* ws, long long wait, cudaStream_t s) {
  if (use_prefill_digits(M, K))
    return launch_gated_t<4>(Wu, su, Wg, sg, xq, x_scale, M, N, K, u, v, h, hmax, ws, wait, s);
  return launch_gated_t<kKind>(Wu, su, Wg, sg, xq, x_scale, M, N, K, u, v, h, hmax, ws, wait, s);
}

bool gemm_tc_from_f32_supported(int64_t M, int64_t K) { return use_prefill_digits(M, K); }

cudaError_t launch_gemm_tc_from_f32(const uint8_t* Wq, const float* w_scale, const float* h,
                                    const unsigned* hmax, int64_t M, int64_t N, int64_t K,
                                    float* y, uint16_t* y_bf16, int32_t* acc_out, int8_t* hq,
                                    float* sh, void* ws, long long wait, cudaStream_t s) {
  if (!use_prefill_digits(M, K)) return cudaErrorInvalidValue;
  const FromF32 ff = {h, hmax, hq, sh};
  if (pick_bn(N) == 128)
    return launch_kind<4, 128, false>(Wq, w_scale, nullptr, nullptr, M, N, K, y, y_bf16, acc_out,
                                      ws, wait, s, &ff);
  return launch_kind<4, 256, false>(Wq, w_scale, nullptr, nullptr, M, N, K, y, y_bf16, acc_out, ws,
                                    wait, s, &ff);
}

// M >= 12, or M >= 5 on matrices of at least 16 Mi weights: measured on B300
// (same box, us, CUDA cores vs tensor cores): 2560 x 2560 at M = 5 / 8 / 12
// 10.0 / 10.4 / 14.0 vs 12.0 / 13.4 / 13.8; 6912 x 2560 and 2560 x 6912 at
// M = 5..12 15.2-27.9 vs 13.8-14.9; 100B shapes 113-216 vs 45-52.
bool gemm_tc_eligible(int64_t M, int64_t N, int64_t K) {
  if (N < 1 || K < 64 || K % 64 != 0) return false;
  return M >= 12 || (M >= 5 && N * K >= ((int64_t)16 << 20));
}

size_t gemm_tc_workspace(int64_t M, int64_t N, int64_t K) { return ws_layout(M, N, K).end; }

cudaError_t launch_gemm_tc(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                           const float* x_scale, int64_t M, int64_t N, int64_t K, float* y,
                           uint16_t* y_bf16, int32_t* acc_out, void* ws, long long wait,
                           cudaStream_t s) {
  if (use_fused(M) && use_digits(M, K))
    return launch_kind<2, 256, true>(Wq, w_scale, xq, x_scale, M, N, K, y, y_bf16, acc_out, ws,
                                     wait, s);
  if (use_fused(M))
    return launch_kind<kKind, 256, true>(Wq, w_scale, xq, x_scale, M, N, K, y, y_bf16, acc_out,
                                         ws, wait, s);
  if (use_prefill_digits(M, K)) {
    if (pick_bn(N) == 128)
      return launch_kind<4, 128, false>(Wq, w_scale, xq, x_scale, M, N, K, y, y_bf16, acc_out, ws,
                                        wait, s);
    return launch_kind<4, 256, false>(Wq, w_scale, xq, x_scale, M, N, K, y, y_bf16, acc_out, ws,
                                      wait, s);
  }
  if (pick_bn(N) == 128)
    return launch_kind<kKind, 128, false>(Wq, w_scale, xq, x_scale, M, N, K, y, y_bf16, acc_out,
                                          ws, wait, s);
  return launch_kind<kKind, 256, false>(Wq, w_scale, xq, x_scale, M, N, K, y, y_bf16, acc_out, ws,
                                        wait, s);
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
