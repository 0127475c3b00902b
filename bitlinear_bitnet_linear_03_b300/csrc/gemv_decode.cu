// gemv_decode.cu — decode BitLinear (one to four tokens) streamed from HBM.
//
// What is computed is the BitLinear product of "BitNet.cpp deep dive"
// (dashen-tech), §3.1: acc = sum_pos - sum_neg over the ternary weights of a
// row, then y = (float)acc * (x_scale * w_scale).  As in gemv.cu the stored
// code c = q + 1 is used directly, sum q x = sum c x - sum x, with one AND and
// one byte dot product (dp4a) per four weights; every sum is an integer, so
// the result is exact and order-free.
//
// Layout of the work (decode is bound by the packed-weight stream):
//  * One producer lane streams the CTA's weight rows into a ring of shared-
//    memory stages with bulk asynchronous copies (cp.async.bulk, completion
//    counted on an mbarrier per stage).  A stage is a block of 32 rows times
//    a K-slice of at most 48 64-weight chunks (24 KB); when the slice is the
//    whole row the block is one contiguous copy, otherwise one copy per row.
//  * Every one of the eight consumer warps takes part in every stage, in
//    order (so the parity of each mbarrier phase is unambiguous): warp w owns
//    rows 4w .. 4w+3 of each block, an 8-lane group owns a row and lane
//    (l % 8) reads 16-byte chunks l%8, l%8 + 8, ... of the slice (128
//    contiguous bytes per group per step); row sums carry across the
//    K-slices of a block in registers.  The
//    int8 activations sit in shared memory in a swizzled chunk layout; the
//    four groups read the same chunk, so each activation read is a broadcast
//    that touches every bank once.  The row sum is three shuffles.
//  * Before waiting on the previous kernel the CTA asks for its whole weight
//    range to be prefetched into L2 and lets its successor launch:
//    consecutive decode kernels overlap under programmatic dependent launch.
//    Weights are read after that wait, unless the caller declared them
//    static (not written by any work still in flight): then the producer
//    starts filling the ring at once, while the previous kernel finishes.
//  * Up to kDecodeMaxTargets matrices sharing the same input run in one
//    launch; their rows are concatenated, stages never straddle two matrices.
//  * The input is int8 with its scales, or bf16: then every CTA forms the
//    per-token absmax over all of K and quantises x with the rule of the
//    activation-quantisation kernel (bit-identical codes).
//  * Every mbarrier wait is bounded (about a second); on time-out the kernel
//    records an error code, stops issuing copies, waits (bounded) for the
//    copies it has in flight and returns.
#include "common.cuh"

namespace bitnet {

__device__ int g_decode_error;

namespace {

constexpr int kGroups = 1;                  // consumer warp groups, alternating row blocks
constexpr int kGroupWarps = 8;
constexpr int kConsumerWarps = kGroups * kGroupWarps;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxStages = 8;
constexpr int kRingBudget = 96 * 1024;
constexpr int kMaxSliceChunks = 48;        // 32 rows x 48 chunks x 16 B = 24 KB per stage
constexpr int kMaxSmem = 227 * 1024 - 1024;  // dynamic part; static barriers etc. fit in the rest
constexpr int kPrefetchMax = 1 << 16;
constexpr long long kWaitCycles = 2000000000ll;  // ~1 s at 2 GHz
constexpr int kErrFullWait = 1;
constexpr int kErrEmptyWait = 2;
constexpr int kErrDrainWait = 3;

struct Target {
  const uint8_t* Wq;
  const float* w_scale;
  float* y;
  int32_t* acc_out;
  int row0;
  int N;
};

struct Args {
  Target t[kDecodeMaxTargets];
  int count;
  int rows_total;
  int rows_per_cta;
  const uint16_t* xb;    // bf16 input, or null
  const int8_t* xq;      // int8 input, or null
  const float* x_scale;  // scales of xq
  int8_t* xq_out;        // optional copy of the quantised bf16 input
  float* xs_out;
  int M, K;
  int slice_chunks;  // 64-weight chunks per K-slice (one stage = one block x one slice)
  int nslices;
  int stages;
  int stage_bytes;   // ring slot size: kBlockRows x slice_chunks x 16 bytes
  int weights_early; // weights may be read before the previous kernel ends
};

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
// Bounded wait for the phase with the given parity; false on time-out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles) return false;
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
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Byte offset of field s (16 bytes) of chunk c in the swizzled activation
// row: field s sits in slot (s + c/2) & 3 of the chunk's 64 bytes, so the
// eight chunks a quarter-warp reads at once land on eight distinct 16-byte
// bank groups.
__device__ __forceinline__ int xs_offset(int c, int s) { return 64 * c + 16 * ((s + (c >> 1)) & 3); }

// The CTA's stage sequence.  Rows of each matrix overlapping the CTA's range
// are taken in blocks of kBlockRows (block b goes to consumer group b % 2);
// each block is streamed as `nslices` K-slices of slice_chunks 64-weight
// chunks (the last may be shorter).  Calls f(p, first_row, nrows, slice, b)
// in order; stops when f returns false.
constexpr int kBlockRows = 32;
template <typename F>
__device__ __forceinline__ void for_each_stage(const Args& a, int r_begin, int r_end, F&& f) {
  int b = 0;
  for (int p = 0; p < a.count; ++p) {
    const int lo = max(r_begin, a.t[p].row0);
    const int hi = min(r_end, a.t[p].row0 + a.t[p].N);
    for (int r = lo; r < hi; r += kBlockRows, ++b)
      for (int sl = 0; sl < a.nslices; ++sl)
        if (!f(p, r - a.t[p].row0, min(kBlockRows, hi - r), sl, b)) return;
  }
}

// Ring slot and phase of a stage: group g owns slots g*H .. g*H + H-1 and
// takes its stages in order, so each slot's mbarrier phases are consumed in
// sequence by one group.
struct SlotPhase {
  int slot;
  int use;  // how many times this slot was filled before
};
__device__ __forceinline__ SlotPhase slot_of(const Args& a, int b, int sl) {
  const int H = a.stages / kGroups;
  const int ig = (b / kGroups) * a.nslices + sl;  // stage index within the group
  SlotPhase r;
  r.slot = (b % kGroups) * H + ig % H;
  r.use = ig / H;
  return r;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, MT <= 2 ? 2 : 1)
k_gemv_decode(const __grid_constant__ Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ float s_max[kConsumerWarps][MT];
  __shared__ int s_sumx[MT];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r_begin = blockIdx.x * a.rows_per_cta;
  const int r_end = min(r_begin + a.rows_per_cta, a.rows_total);
  const int64_t row_bytes = a.K >> 2;
  const int nch = a.K >> 6;
  const uint32_t ring = smem_addr(smem);
  int8_t* xs = reinterpret_cast<int8_t*>(smem + a.stages * a.stage_bytes);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kGroupWarps);
    }
    mbar_fence_init();
    for (int m = 0; m < MT; ++m) s_sumx[m] = 0;
    // L2 prefetch hint for this CTA's weights (independent of the previous
    // kernel; no data is read before griddep_wait).
    for (int p = 0; p < a.count; ++p) {
      const int lo = max(r_begin, a.t[p].row0);
      const int hi = min(r_end, a.t[p].row0 + a.t[p].N);
      if (lo >= hi) continue;
      const uint8_t* base = a.t[p].Wq + (int64_t)(lo - a.t[p].row0) * row_bytes;
      const int64_t bytes = (int64_t)(hi - lo) * row_bytes;
      for (int64_t off = 0; off < bytes; off += kPrefetchMax)
        prefetch_l2_bulk(base + off, (uint32_t)(bytes - off < kPrefetchMax ? bytes - off
                                                                              : kPrefetchMax));
    }
  }
  griddep_launch_dependents();
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == kConsumerWarps) {
    if (lane != 0) return;
    // Weights the caller declared static may stream in while the previous
    // kernel on the stream is still running; otherwise wait for it first.
    // Either way every bounded wait below starts after the dependency wait.
    bool dep_done = !a.weights_early;
    if (dep_done) griddep_wait();
    int issued[kGroups] = {};
    for_each_stage(a, r_begin, r_end, [&](int p, int row, int nrows, int sl, int b) {
      const SlotPhase sp = slot_of(a, b, sl);
      if (sp.use > 0) {
        if (!dep_done) {
          griddep_wait();
          dep_done = true;
        }
        if (!mbar_wait(smem_addr(&empty_bar[sp.slot]), (sp.use - 1) & 1)) {
          atomicOr(&g_decode_error, 1 << kErrEmptyWait);
          return false;
        }
      }
      const int c0 = sl * a.slice_chunks;
      const int chunks = min(a.slice_chunks, nch - c0);
      const uint32_t slice_bytes = (uint32_t)chunks * 16u;
      const uint32_t fb = smem_addr(&full_bar[sp.slot]);
      const uint32_t dst = ring + sp.slot * a.stage_bytes;
      const uint8_t* src = a.t[p].Wq + (int64_t)row * row_bytes + c0 * 16;
      mbar_arrive_expect_tx(fb, slice_bytes * (uint32_t)nrows);
      if (a.nslices == 1) {
        // whole rows: the block is one contiguous span
        bulk_copy_g2s(dst, src, slice_bytes * (uint32_t)nrows, fb);
      } else {
        for (int r = 0; r < nrows; ++r)
          bulk_copy_g2s(dst + r * slice_bytes, src + (int64_t)r * row_bytes, slice_bytes, fb);
      }
      ++issued[b % kGroups];
      return true;
    });
    // Never leave the CTA with a copy in flight: wait for the last copy of
    // every slot of both groups to land.
    const int H = a.stages / kGroups;
    for (int g = 0; g < kGroups; ++g) {
      const int first = issued[g] > H ? issued[g] - H : 0;
      for (int j = first; j < issued[g]; ++j)
        if (!mbar_wait(smem_addr(&full_bar[g * H + j % H]), (j / H) & 1)) {
          atomicOr(&g_decode_error, 1 << kErrDrainWait);
          g = kGroups;
          break;
        }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  griddep_wait();
  const int tid = threadIdx.x;  // 0 .. kConsumers-1
  const int K = a.K;
  const int nitems = K >> 4;   // 16-byte fields per token row
  float xscale[MT];
  if (a.xb != nullptr && MT <= 2 && nitems <= 2 * kConsumers) {
    // One pass: each thread keeps its (at most two) 16-element items of x in
    // registers between the absmax and the quantisation.
    uint4 held[MT][2][2];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float mx = 0.0f;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int f = tid + j * kConsumers;
        held[m][j][0] = held[m][j][1] = make_uint4(0, 0, 0, 0);
        if (m < a.M && f < nitems) {
          const uint4* src = reinterpret_cast<const uint4*>(a.xb + (int64_t)m * K) + 2 * f;
          held[m][j][0] = ld_nc_v4(src);
          held[m][j][1] = ld_nc_v4(src + 1);
        }
        const uint32_t e[8] = {held[m][j][0].x, held[m][j][0].y, held[m][j][0].z,
                               held[m][j][0].w, held[m][j][1].x, held[m][j][1].y,
                               held[m][j][1].z, held[m][j][1].w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          mx = fmaxf(mx, fabsf(bf16_bits_to_float(e[t] & 0xffffu)));
          mx = fmaxf(mx, fabsf(bf16_bits_to_float(e[t] >> 16)));
        }
      }
      mx = warp_max_f32(mx);
      if (lane == 0) s_max[warp][m] = mx;
    }
    consumer_sync();
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float mx = s_max[0][m];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) mx = fmaxf(mx, s_max[w][m]);
      const ActScale sc = act_scale_from_absmax(mx);
      xscale[m] = sc.scale;
      int sum = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int f = tid + j * kConsumers;
        if (m < a.M && f < nitems) {
          const uint32_t e[8] = {held[m][j][0].x, held[m][j][0].y, held[m][j][0].z,
                                 held[m][j][0].w, held[m][j][1].x, held[m][j][1].y,
                                 held[m][j][1].z, held[m][j][1].w};
          uint32_t wd[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            int q[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int el = 4 * i + t;
              const uint32_t h = (el & 1) ? (e[el >> 1] >> 16) : (e[el >> 1] & 0xffffu);
              q[t] = round_clip(__fmul_rn(bf16_bits_to_float(h), sc.inv), -128.f, 127.f);
            }
            wd[i] = pack_i8x4(q[0], q[1], q[2], q[3]);
            sum = dp4a_ss(wd[i], 0x01010101u, sum);
          }
          const uint4 packed = make_uint4(wd[0], wd[1], wd[2], wd[3]);
          *reinterpret_cast<uint4*>(xs + (int64_t)m * K + xs_offset(f >> 2, f & 3)) = packed;
          if (blockIdx.x == 0 && a.xq_out != nullptr)
            *reinterpret_cast<uint4*>(a.xq_out + (int64_t)m * K + 16 * f) = packed;
        }
      }
      sum = warp_sum_i32(sum);
      if (lane == 0 && sum) atomicAdd(&s_sumx[m], sum);
      if (blockIdx.x == 0 && tid == 0 && a.xs_out != nullptr && m < a.M) a.xs_out[m] = xscale[m];
    }
  } else if (a.xb != nullptr) {
    const int nv = K >> 3;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float mx = 0.0f;
      if (m < a.M) {
        const uint4* xrow = reinterpret_cast<const uint4*>(a.xb + (int64_t)m * K);
        for (int v = tid; v < nv; v += kConsumers) {
          const uint4 q = ld_nc_v4(xrow + v);
          const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            mx = fmaxf(mx, fabsf(bf16_bits_to_float(w4[t] & 0xffffu)));
            mx = fmaxf(mx, fabsf(bf16_bits_to_float(w4[t] >> 16)));
          }
        }
      }
      mx = warp_max_f32(mx);
      if (lane == 0) s_max[warp][m] = mx;
    }
    consumer_sync();
    float inv[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float mx = s_max[0][m];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) mx = fmaxf(mx, s_max[w][m]);
      const ActScale sc = act_scale_from_absmax(mx);
      inv[m] = sc.inv;
      xscale[m] = sc.scale;
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int sum = 0;
      if (m < a.M) {
        const uint4* xrow = reinterpret_cast<const uint4*>(a.xb + (int64_t)m * K);
        for (int f = tid; f < nitems; f += kConsumers) {
          const uint4 p0 = ld_nc_v4(xrow + 2 * f), p1 = ld_nc_v4(xrow + 2 * f + 1);
          const uint32_t e[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          uint32_t wd[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            int q[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int el = 4 * i + t;
              const uint32_t h = (el & 1) ? (e[el >> 1] >> 16) : (e[el >> 1] & 0xffffu);
              q[t] = round_clip(__fmul_rn(bf16_bits_to_float(h), inv[m]), -128.f, 127.f);
            }
            wd[i] = pack_i8x4(q[0], q[1], q[2], q[3]);
            sum = dp4a_ss(wd[i], 0x01010101u, sum);
          }
          const uint4 packed = make_uint4(wd[0], wd[1], wd[2], wd[3]);
          *reinterpret_cast<uint4*>(xs + (int64_t)m * K + xs_offset(f >> 2, f & 3)) = packed;
          if (blockIdx.x == 0 && a.xq_out != nullptr)
            *reinterpret_cast<uint4*>(a.xq_out + (int64_t)m * K + 16 * f) = packed;
        }
      }
      sum = warp_sum_i32(sum);
      if (lane == 0 && sum) atomicAdd(&s_sumx[m], sum);
      if (blockIdx.x == 0 && tid == 0 && a.xs_out != nullptr && m < a.M) a.xs_out[m] = xscale[m];
    }
  } else {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int sum = 0;
      xscale[m] = 0.0f;
      if (m < a.M) {
        xscale[m] = a.x_scale[m];
        const uint4* xrow = reinterpret_cast<const uint4*>(a.xq + (int64_t)m * K);
        for (int f = tid; f < nitems; f += kConsumers) {
          const uint4 v = ld_nc_v4(xrow + f);
          sum = dp4a_ss(v.x, 0x01010101u, sum);
          sum = dp4a_ss(v.y, 0x01010101u, sum);
          sum = dp4a_ss(v.z, 0x01010101u, sum);
          sum = dp4a_ss(v.w, 0x01010101u, sum);
          *reinterpret_cast<uint4*>(xs + (int64_t)m * K + xs_offset(f >> 2, f & 3)) = v;
        }
      }
      sum = warp_sum_i32(sum);
      if (lane == 0 && sum) atomicAdd(&s_sumx[m], sum);
    }
  }
  consumer_sync();
  int sumx[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) sumx[m] = s_sumx[m];

  // Group g takes row blocks g, g+2, ...; its warp wl owns rows 4wl .. 4wl+3
  // of each block, 8-lane group grp row 4wl + grp, and lane sub chunks sub,
  // sub+8, ... of each slice.  Slices start at multiples of 8 chunks, so in
  // every chunk this lane reads, field s sits at the same slot
  // (s + sub/2) & 3: xo[s] is its byte offset within the chunk.  The eight
  // lanes of a quarter-warp then read eight distinct 16-byte bank groups.
  const int gw = warp / kGroupWarps, wl = warp % kGroupWarps;
  const int grp = lane >> 3, sub = lane & 7;
  const int r = wl * 4 + grp;
  uint32_t xo[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) xo[k] = 16u * (uint32_t)((k + (sub >> 1)) & 3);
  const uint32_t xs_base = smem_addr(xs);
  // acc[m][k][i]: independent dp4a chains per token (field k, word i % NI).
  // One token needs 16 chains to keep the issue slots busy; more tokens bring
  // their own chains.
  constexpr int NI = MT == 1 ? 4 : 1;
  int acc[MT][4][NI];
  for_each_stage(a, r_begin, r_end, [&](int p, int row0, int nrows, int sl, int b) {
    if (b % kGroups != gw) return true;
    const SlotPhase sp = slot_of(a, b, sl);
    if (!mbar_wait(smem_addr(&full_bar[sp.slot]), sp.use & 1)) {
      if (lane == 0) atomicOr(&g_decode_error, 1 << kErrFullWait);
      return false;
    }
    if (sl == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < NI; ++i) acc[m][k][i] = 0;
    }
    const bool valid = r < nrows;
    const int c0 = sl * a.slice_chunks;
    const int chunks = min(a.slice_chunks, nch - c0);
    if (valid && sub < chunks) {
      uint32_t wp = ring + sp.slot * a.stage_bytes + (uint32_t)(r * chunks * 16) + 16 * sub;
      uint32_t xp = xs_base + 64 * (c0 + sub);
      // Operands of the current chunk; the next chunk's are loaded before
      // the current one is consumed.
      uint4 wv = lds128(wp);
      uint4 xv[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) xv[m][k] = lds128(xp + m * K + xo[k]);
      // One token: the next chunk's operands are loaded before the current
      // one is consumed.  More tokens: enough independent loads already.
      constexpr int NB = MT == 1 ? MT : 1;
      for (int c = sub;;) {
        const bool more = c + 8 < chunks;
        uint4 wn = make_uint4(0, 0, 0, 0);
        uint4 xn[NB][4];
        if (MT == 1 && more) {
          wn = lds128(wp + 128);
#pragma unroll
          for (int k = 0; k < 4; ++k) xn[0][k] = lds128(xp + 512 + xo[k]);
        }
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t xw[4] = {xv[m][k].x, xv[m][k].y, xv[m][k].z, xv[m][k].w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
              acc[m][k][i % NI] =
                  dp4a_us(ww[i] & (0x03030303u << (2 * k)), xw[i], acc[m][k][i % NI]);
          }
        }
        if (!more) break;
        c += 8;
        wp += 128;
        xp += 512;
        if (MT == 1) {
          wv = wn;
#pragma unroll
          for (int k = 0; k < 4; ++k) xv[0][k] = xn[0][k];
        } else {
          wv = lds128(wp);
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int k = 0; k < 4; ++k) xv[m][k] = lds128(xp + m * K + xo[k]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[sp.slot]));
    if (sl == a.nslices - 1) {
      const Target& T = a.t[p];
      const float ws = *T.w_scale;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        int t = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
        {
          int u = 0;
#pragma unroll
          for (int i = 0; i < NI; ++i) u += acc[m][k][i];
          t += u >> (2 * k);
        }
        t += __shfl_xor_sync(0xffffffffu, t, 4);
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        t += __shfl_xor_sync(0xffffffffu, t, 1);
        if (sub == 0 && valid && m < a.M) {
          const int total = t - sumx[m];
          const int64_t o = (int64_t)m * T.N + row0 + r;
          T.y[o] = __fmul_rn(__int2float_rn(total), __fmul_rn(xscale[m], ws));
          if (T.acc_out) T.acc_out[o] = total;
        }
      }
    }
    return true;
  });
}

struct Plan {
  int mt, slice_chunks, nslices, stages, stage_bytes;
  size_t smem;
};

bool make_plan(int64_t M, int64_t K, Plan* pl) {
  if (M < 1 || M > kDecodeMaxM || K < 64 || K % 64 != 0 || K > 65536) return false;
  pl->mt = M <= 1 ? 1 : M <= 2 ? 2 : 4;
  const int nch = (int)(K / 64);
  if (nch <= kMaxSliceChunks) {
    pl->nslices = 1;
    pl->slice_chunks = nch;
  } else {
    // slices start on multiples of 8 chunks (see the consumer loop)
    int ns = (nch + kMaxSliceChunks - 1) / kMaxSliceChunks;
    int sc = ((nch + ns - 1) / ns + 7) / 8 * 8;
    pl->slice_chunks = sc;
    pl->nslices = (nch + sc - 1) / sc;
  }
  pl->stage_bytes = kBlockRows * pl->slice_chunks * 16;
  int S = kRingBudget / pl->stage_bytes;
  S = S / kGroups * kGroups;
  if (S < 2 * kGroups) S = 2 * kGroups;
  if (S > kMaxStages) S = kMaxStages;
  pl->stages = S;
  pl->smem = (size_t)S * pl->stage_bytes + (size_t)pl->mt * (size_t)K;
  return pl->smem <= (size_t)kMaxSmem;
}

template <int MT>
cudaError_t launch_t(const Args& a, int ctas, size_t smem, cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(k_gemv_decode<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return launch_pdl(k_gemv_decode<MT>, dim3(ctas), dim3(kThreads), smem, s, a);
}

}  // namespace

bool decode_supported(int64_t M, int64_t K) {
  Plan pl;
  return make_plan(M, K, &pl);
}

cudaError_t launch_decode(const DecodeTarget* targets, int count, const int8_t* xq,
                          const float* x_scale, const uint16_t* x_bf16, int64_t M, int64_t K,
                          int8_t* xq_out, float* x_scale_out, bool weights_static,
                          cudaStream_t s) {
  Plan pl;
  if (count < 1 || count > kDecodeMaxTargets || !make_plan(M, K, &pl))
    return cudaErrorNotSupported;
  Args a = {};
  int64_t rows = 0;
  for (int p = 0; p < count; ++p) {
    a.t[p].Wq = targets[p].Wq;
    a.t[p].w_scale = targets[p].w_scale;
    a.t[p].y = targets[p].y;
    a.t[p].acc_out = targets[p].acc_out;
    a.t[p].row0 = (int)rows;
    a.t[p].N = (int)targets[p].N;
    rows += targets[p].N;
  }
  if (rows > (1 << 30)) return cudaErrorNotSupported;
  a.count = count;
  a.rows_total = (int)rows;
  a.xb = x_bf16;
  a.xq = xq;
  a.x_scale = x_scale;
  a.xq_out = xq_out;
  a.xs_out = x_scale_out;
  a.M = (int)M;
  a.K = (int)K;
  a.slice_chunks = pl.slice_chunks;
  a.nslices = pl.nslices;
  a.stages = pl.stages;
  a.stage_bytes = pl.stage_bytes;
  a.weights_early = weights_static ? 1 : 0;
  int64_t ctas = (rows + 3) / 4;
  if (ctas > 148) ctas = 148;
  a.rows_per_cta = (int)((rows + ctas - 1) / ctas);
  ctas = (rows + a.rows_per_cta - 1) / a.rows_per_cta;
  const int c = (int)ctas;
  if (pl.mt == 1) return launch_t<1>(a, c, pl.smem, s);
  if (pl.mt == 2) return launch_t<2>(a, c, pl.smem, s);
  return launch_t<4>(a, c, pl.smem, s);
}

cudaError_t read_and_clear_decode_error(int* code, cudaStream_t s) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_decode_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_decode_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e;
}

}  // namespace bitnet
