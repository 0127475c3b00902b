// gemv_decode.cu — decode BitLinear (one to four tokens) streamed from HBM.
//
// What is computed is the BitLinear product of "BitNet.cpp deep dive"
// (dashen-tech), §3.1: acc = sum_pos - sum_neg over the ternary weights of a
// row, then y = (float)acc * (x_scale * w_scale).  The stored code c = q + 1
// is used directly, sum q x = sum c x - sum x: in a 16-byte block of the
// packed layout, word i masked with 0x03030303 << 2s holds 4^s times the
// codes of weights 16s + 4i + {0..3}, so one AND and one byte dot product
// (dp4a) cover four weights; field s keeps its own accumulator and the 4^s is
// removed by an exact shift.  Every sum is an integer: the result is exact
// and independent of order.
//
// Layout of the work (decode is bound by the packed-weight stream):
//  * One producer lane streams the CTA's weight rows into a ring of shared-
//    memory stages with bulk asynchronous copies (cp.async.bulk, completion
//    counted on an mbarrier per stage).  A stage is R whole rows of one
//    matrix, i.e. one contiguous copy of about 20-24 KB (the copy engine
//    sustains full HBM bandwidth only with large copies).
//  * Eight consumer warps take part in every stage, in order, so the parity
//    of each mbarrier phase is unambiguous.  The warps split K into `wk`
//    parts and the stage's rows into 8/wk groups.  Lane l of a warp owns the
//    64-weight chunks l, l+32, ... of its K part for the whole kernel: their
//    int8 activations are loaded into registers once, and a row costs the
//    lane one 16-byte shared load, 16 ANDs and 16 dp4a per chunk; the 32
//    lanes read 512 contiguous bytes of the row.  Rows go two at a time, their
//    dp4a chains interleaved.  A row's lane sums meet in one warp reduction
//    (redux.sync).
//  * Single launch: the consumers store each row's K-part result in shared
//    memory and release the slot; the producer warp, when it takes the slot
//    back for a new copy, sums the parts and writes the stage's outputs
//    (rows across its lanes, coalesced).  The consumers' per-stage work is
//    then only the dot products.
//  * Chain of phases (one CTA per SM, grid barrier between phases): the
//    consumers write the outputs themselves, so the barrier arrival follows
//    the last stage directly; with wk > 1 the K parts meet in a 64-bit
//    shared-memory atomic per row that also counts the parts, and the last
//    part to arrive writes the row.
//  * Before waiting on the previous kernel the CTA asks for its whole weight
//    range and its input to be prefetched into L2 and lets its successor
//    launch:
//    consecutive decode kernels overlap under programmatic dependent launch.
//    Weights are read after that wait, unless the caller declared them
//    static (not written by any work still in flight): then the producer
//    issues the first stage while the previous kernel finishes.  The rest
//    of a phase's stages wait until the consumers have read the phase's
//    input x, whose loads would otherwise queue behind the weight copies.
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

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxStages = 8;
constexpr int kRingBudget = 96 * 1024;
constexpr int kStageTarget = 24 * 1024;
constexpr int kMaxRowsPerWarp = 8;         // rows of one stage handled by one warp
// Stages of a phase the producer issues before the consumers have read that
// phase's input x, so that the input's loads do not queue behind a full ring
// of weight copies (measured on B300: 3-4% faster for a 58 MB matrix, neutral
// for the 2B-shape chain).
constexpr int kEarlyStages = 1;
constexpr int kMaxSmem = 227 * 1024 - 10 * 1024;  // dynamic part; the static arrays fit in the rest
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

// One decode BitLinear launch: up to kDecodeMaxTargets matrices sharing the
// input x, and the work split computed on the host.
struct Phase {
  Target t[kDecodeMaxTargets];
  int count;
  int rows_total;
  int rows_per_cta;
  const uint16_t* xb;    // bf16 input, or null
  const int8_t* xq;      // int8 input, or null
  const float* x_scale;  // scales of xq
  int8_t* xq_out;        // optional copy of the quantised bf16 input
  float* xs_out;
  int K;
  int wk;              // warps splitting K (1, 2, 4 or 8)
  int kpart;           // 64-weight chunks per K part
  int rows_per_stage;  // R: whole rows per ring slot
  int stage_bytes;     // R * K / 4 (<= the ring slot)
};

// A launch runs one phase (ph0), or a chain of phases from a device table with
// a grid-wide barrier between consecutive phases.
struct Args {
  Phase ph0;
  const Phase* phases;          // chain table in device memory, or null
  unsigned long long* barrier;  // chain: generation-counted barrier word
  int nphases;
  int M;
  int stages;
  int slot_bytes;
  int xs_bytes;                 // per-token bf16 staging (max K)
  int weights_early;            // weights may be read before the previous kernel ends
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

// The CTA's stage sequence within one phase: for each matrix overlapping the
// CTA's rows, the rows in pieces of at most rows_per_stage.  Calls
// f(p, first_row, nrows) in order; returns false if f stopped it.
template <typename F>
__device__ __forceinline__ bool for_each_stage(const Phase& ph, F&& f) {
  const int r_begin = blockIdx.x * ph.rows_per_cta;
  const int r_end = min(r_begin + ph.rows_per_cta, ph.rows_total);
  for (int p = 0; p < ph.count; ++p) {
    const int lo = max(r_begin, ph.t[p].row0);
    const int hi = min(r_end, ph.t[p].row0 + ph.t[p].N);
    for (int r = lo; r < hi; r += ph.rows_per_stage)
      if (!f(p, r - ph.t[p].row0, min(ph.rows_per_stage, hi - r))) return false;
  }
  return true;
}

// L2 prefetch hint for one phase's weight rows of this CTA.
__device__ __forceinline__ void prefetch_phase(const Phase& ph) {
  const int r_begin = blockIdx.x * ph.rows_per_cta;
  const int r_end = min(r_begin + ph.rows_per_cta, ph.rows_total);
  const int64_t row_bytes = ph.K >> 2;
  for (int p = 0; p < ph.count; ++p) {
    const int lo = max(r_begin, ph.t[p].row0);
    const int hi = min(r_end, ph.t[p].row0 + ph.t[p].N);
    if (lo >= hi) continue;
    const uint8_t* base = ph.t[p].Wq + (int64_t)(lo - ph.t[p].row0) * row_bytes;
    const int64_t bytes = (int64_t)(hi - lo) * row_bytes;
    for (int64_t off = 0; off < bytes; off += kPrefetchMax)
      prefetch_l2_bulk(base + off,
                       (uint32_t)(bytes - off < kPrefetchMax ? bytes - off : kPrefetchMax));
  }
}

// L2 prefetch hint for one phase's input x (bf16 or int8, M rows).
__device__ __forceinline__ void prefetch_x(const Phase& ph, int M) {
  const void* p = ph.xb != nullptr ? (const void*)ph.xb : (const void*)ph.xq;
  const int64_t bytes = (int64_t)M * ph.K * (ph.xb != nullptr ? 2 : 1);
  for (int64_t off = 0; off < bytes; off += kPrefetchMax)
    prefetch_l2_bulk(static_cast<const uint8_t*>(p) + off,
                     (uint32_t)(bytes - off < kPrefetchMax ? bytes - off : kPrefetchMax));
}

// Grid barrier of a chain: a 64-bit counter that every CTA increments once
// per barrier and that is never reset; barrier b of this launch completes
// when it reaches base + (b + 1) * gridDim.x.  Bounded wait.
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool grid_wait(const unsigned long long* ctr, unsigned long long target) {
  if (ld_acquire_u64(ctr) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_u64(ctr) < target) {
    __nanosleep(64);
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}

// Copies a phase descriptor with the 32 lanes of a warp.
__device__ __forceinline__ void copy_phase(const Phase& src, Phase* dst, int lane) {
  static_assert(sizeof(Phase) % 8 == 0, "phase descriptor is copied in 8-byte words");
  const unsigned long long* s = reinterpret_cast<const unsigned long long*>(&src);
  unsigned long long* d = reinterpret_cast<unsigned long long*>(dst);
  for (int i = lane; i < (int)(sizeof(Phase) / 8); i += 32) d[i] = s[i];
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

// What the producer records when it fills a ring slot of a single-phase
// launch, read back when the consumers release the slot and it writes the
// stage's outputs.
struct StageRec {
  int p, row0, nrows;
};

// CHAIN: a chain of phases (cooperative launch, grid barrier between phases);
// the consumers write the outputs of every stage (K parts merged through
// shared-memory atomics) and arrive at the barrier.  Otherwise one phase: the
// consumers leave each row's K-part results in shared memory and release the
// slot, and the producer warp writes the stage's outputs while the next
// stages are consumed.
// A chain runs one CTA per SM (all resident for the grid barrier): its
// registers are not shared with a second CTA.
template <int MT, int J, bool CHAIN>
__global__ void __launch_bounds__(kThreads, (MT <= 2 && !CHAIN) ? 2 : 1)
k_gemv_decode(const __grid_constant__ Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ float s_max[kConsumerWarps][MT];
  __shared__ int s_abort;
  __shared__ int s_xgate;  // phases whose input x the consumers have read
  // The consumers' copy of the current phase descriptor (read in the hot
  // loop; shared memory instead of a pointer into the parameter block or the
  // chain table).
  __shared__ __align__(16) Phase s_ph;
  // CHAIN: K-part merge per ring slot and stage row; the low 48 bits hold
  // the sum of the parts' biased partial dot products, bits 48.. count the
  // parts added.  Otherwise: each K part's row result (part kw of stage row
  // r at kw * R + r), the stage records and the activation scales.
  constexpr int kAccRows = CHAIN ? kConsumerWarps * kMaxRowsPerWarp / 2 : 1;
  constexpr int kPartRows = CHAIN ? 1 : kConsumerWarps * kMaxRowsPerWarp;
  __shared__ unsigned long long s_acc[kMaxStages][kAccRows][MT];
  __shared__ int s_part[kMaxStages][kPartRows][MT];
  __shared__ StageRec s_stage[kMaxStages];
  __shared__ float s_xscale[MT];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = smem_addr(smem);
  const Phase* phases = CHAIN ? a.phases : &a.ph0;

  if (CHAIN)
    for (int q = threadIdx.x; q < kMaxStages * kAccRows * MT; q += kThreads)
      (&s_acc[0][0][0])[q] = 0ull;
  if (threadIdx.x < 32) copy_phase(phases[0], &s_ph, threadIdx.x);
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kConsumerWarps);
    }
    mbar_fence_init();
    s_abort = 0;
    s_xgate = 0;
    // L2 prefetch hints for the first phase's input and weights (no data is
    // read before the dependency wait).
    prefetch_x(phases[0], a.M);
    prefetch_phase(phases[0]);
  }
  griddep_launch_dependents();
  __syncthreads();

  // ------------------------------------------------------------ producer
  // Lane 0 fills the ring with bulk copies.  Single phase: the whole warp
  // also writes the outputs of each stage the consumers have released
  // (y = acc * (x_scale * w_scale), rows across the lanes).
  if (warp == kConsumerWarps) {
    if (CHAIN && lane != 0) return;
    // Weights the caller declared static may stream in while the previous
    // kernel on the stream is still running (the first stage); otherwise
    // wait for it first.  Either way every bounded wait below starts after
    // the dependency wait.  In a chain the producer runs ahead across phase
    // boundaries (weights never depend on earlier phases), up to the first
    // stage of a phase whose input the consumers have not read yet.
    bool dep_done = !a.weights_early;
    if (dep_done) griddep_wait();
    const int S = a.stages;
    const float ws_lane = (!CHAIN && lane < s_ph.count) ? *s_ph.t[lane].w_scale : 0.0f;
    auto finish = [&](int slot) {
      const StageRec rec = s_stage[slot];
      const Target& T = s_ph.t[rec.p];
      const float wsc = __shfl_sync(0xffffffffu, ws_lane, rec.p);
      const int R = s_ph.rows_per_stage, wk = s_ph.wk;
      for (int m = 0; m < a.M; ++m) {
        const float c = __fmul_rn(s_xscale[m], wsc);
        for (int r = lane; r < rec.nrows; r += 32) {
          int tot = 0;
          for (int kw = 0; kw < wk; ++kw) tot += s_part[slot][kw * R + r][m];
          const int64_t o = (int64_t)m * T.N + rec.row0 + r;
          T.y[o] = __fmul_rn(__int2float_rn(tot), c);
          if (T.acc_out) T.acc_out[o] = tot;
        }
      }
    };
    int i = 0, done = 0;
    bool ok = true;
    for (int ph_i = 0; ph_i < a.nphases && ok; ++ph_i) {
      const Phase& ph = phases[ph_i];
      if (ph_i + 1 < a.nphases) {
        prefetch_x(phases[ph_i + 1], a.M);
        prefetch_phase(phases[ph_i + 1]);
      }
      const int64_t row_bytes = ph.K >> 2;
      int k_phase = 0;  // stages of this phase issued so far
      ok = for_each_stage(ph, [&](int p, int row, int nrows) {
        const int slot = i % S, use = i / S;
        if (k_phase++ == kEarlyStages) {
          // wait (bounded) until the consumers have this phase's input
          const long long t0 = clock64();
          while (*(volatile int*)&s_xgate <= ph_i) {
            if (*(volatile int*)&s_abort) return false;
            if (clock64() - t0 > kWaitCycles) {
              if (lane == 0) atomicOr(&g_decode_error, 1 << kErrEmptyWait);
              *(volatile int*)&s_abort = 1;
              return false;
            }
            __nanosleep(32);
          }
          if (!dep_done) {
            griddep_wait();
            dep_done = true;
          }
        }
        if (use > 0) {
          if (!dep_done) {
            griddep_wait();
            dep_done = true;
          }
          if (!mbar_wait(smem_addr(&empty_bar[slot]), (use - 1) & 1) ||
              *(volatile int*)&s_abort) {
            if (lane == 0) atomicOr(&g_decode_error, 1 << kErrEmptyWait);
            *(volatile int*)&s_abort = 1;
            return false;
          }
          if (!CHAIN) {
            finish(slot);
            ++done;
          }
        }
        if (lane == 0) {
          if (!CHAIN) s_stage[slot] = StageRec{p, row, nrows};
          const uint32_t bytes = (uint32_t)(nrows * row_bytes);
          const uint32_t fb = smem_addr(&full_bar[slot]);
          mbar_arrive_expect_tx(fb, bytes);
          bulk_copy_g2s(ring + slot * a.slot_bytes, ph.t[p].Wq + (int64_t)row * row_bytes,
                        bytes, fb);
        }
        if (!CHAIN) __syncwarp();
        ++i;
        return true;
      });
    }
    // Single phase: the stages still in the ring.
    if (!CHAIN)
      for (; ok && done < i; ++done) {
        const int slot = done % S;
        if (!mbar_wait(smem_addr(&empty_bar[slot]), (done / S) & 1) ||
            *(volatile int*)&s_abort) {
          if (lane == 0) atomicOr(&g_decode_error, 1 << kErrEmptyWait);
          *(volatile int*)&s_abort = 1;
          ok = false;
          break;
        }
        finish(slot);
      }
    // Never leave the CTA with a copy in flight: wait for the last copy of
    // every slot to land.
    if (lane == 0) {
      const int first = i > S ? i - S : 0;
      for (int j = first > done ? first : done; j < i; ++j)
        if (!mbar_wait(smem_addr(&full_bar[j % S]), (j / S) & 1)) {
          atomicOr(&g_decode_error, 1 << kErrDrainWait);
          break;
        }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  griddep_wait();
  const int tid = threadIdx.x;  // 0 .. kConsumers-1
  int8_t* xs = reinterpret_cast<int8_t*>(smem + a.stages * a.slot_bytes);
  unsigned long long bar_base = 0;
  if (CHAIN && tid == 0) bar_base = ld_acquire_u64(a.barrier) / gridDim.x * gridDim.x;
  // Ring position (slot and phase parity) of the next stage; the consumers
  // walk the same stage sequence as the producer.
  int c_slot = 0;
  uint32_t c_parity = 0;

  for (int ph_i = 0; ph_i < a.nphases; ++ph_i) {
    const Phase& ph = s_ph;
    if (ph_i > 0) {
      // Every CTA has finished phase ph_i - 1 before any reads phase ph_i's
      // input.  Meanwhile warp 1 copies the (static) descriptor of phase
      // ph_i.
      if (warp == 1) copy_phase(phases[ph_i], &s_ph, lane);
      if (tid == 0 && !grid_wait(a.barrier, bar_base + (unsigned long long)ph_i * gridDim.x)) {
        atomicOr(&g_decode_error, 1 << kErrFullWait);
        *(volatile int*)&s_abort = 1;
      }
      if (consumer_sync_or(*(volatile int*)&s_abort)) break;
    }
    const int K = ph.K;
    const int64_t row_bytes = K >> 2;
    // This warp: K part kw (chunks k_lo .. k_hi-1) and row group wr of 8/wk.
    // Lane l holds the int8 activations of chunks k_lo + l + 32j (j < J) in
    // registers and the sum of those codes, which it subtracts from every
    // row's partial (sum q x = sum c x - sum x, taken part by part).
    const int kw = warp % ph.wk, wr = warp / ph.wk, nwr = kConsumerWarps / ph.wk;
    const int nch = K >> 6;
    const int k_lo = kw * ph.kpart, k_hi = min(nch, k_lo + ph.kpart);
    // Matrix scales: lane p keeps w_scale of matrix p (read with a shuffle).
    const float ws_lane = lane < ph.count ? *ph.t[lane].w_scale : 0.0f;
    int valid_j = 0;
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (k_lo + lane + 32 * j < k_hi) valid_j = j + 1;
    uint4 xr[MT][J][4];
    int lsum[MT];
    float xscale[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      lsum[m] = 0;
      xscale[m] = 0.0f;
#pragma unroll
      for (int j = 0; j < J; ++j)
#pragma unroll
        for (int s = 0; s < 4; ++s) xr[m][j][s] = make_uint4(0, 0, 0, 0);
    }
    if (ph.xb != nullptr) {
      // bf16 input: the CTA quantises x once into shared memory (after the
      // ring), each thread taking 16-element pieces; the row absmax is shared
      // through s_max.  Then every lane picks up its chunks.
      const int nitems = K >> 4;
      const bool one_pass = nitems <= 2 * kConsumers;
      uint4 held[MT][2][2];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float mx = 0.0f;
        if (m < a.M) {
          const uint4* xrow = reinterpret_cast<const uint4*>(ph.xb + (int64_t)m * K);
          if (one_pass) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int f = tid + j * kConsumers;
              held[m][j][0] = held[m][j][1] = make_uint4(0, 0, 0, 0);
              if (f < nitems) {
                held[m][j][0] = ld_nc_v4(xrow + 2 * f);
                held[m][j][1] = ld_nc_v4(xrow + 2 * f + 1);
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
          } else {
            for (int v = tid; v < (K >> 3); v += kConsumers) {
              const uint4 q = ld_nc_v4(xrow + v);
              const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                mx = fmaxf(mx, fabsf(bf16_bits_to_float(w4[t] & 0xffffu)));
                mx = fmaxf(mx, fabsf(bf16_bits_to_float(w4[t] >> 16)));
              }
            }
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
        if (m >= a.M) continue;
        const uint4* xrow = reinterpret_cast<const uint4*>(ph.xb + (int64_t)m * K);
        for (int j = 0;; ++j) {
          const int f = tid + j * kConsumers;
          if (f >= nitems || (one_pass && j >= 2)) break;
          uint32_t e[8];
          if (one_pass) {
            const uint4 h0 = j == 0 ? held[m][0][0] : held[m][1][0];
            const uint4 h1 = j == 0 ? held[m][0][1] : held[m][1][1];
            e[0] = h0.x; e[1] = h0.y; e[2] = h0.z; e[3] = h0.w;
            e[4] = h1.x; e[5] = h1.y; e[6] = h1.z; e[7] = h1.w;
          } else {
            const uint4 h0 = ld_nc_v4(xrow + 2 * f), h1 = ld_nc_v4(xrow + 2 * f + 1);
            e[0] = h0.x; e[1] = h0.y; e[2] = h0.z; e[3] = h0.w;
            e[4] = h1.x; e[5] = h1.y; e[6] = h1.z; e[7] = h1.w;
          }
          uint32_t wd[4];
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) {
            int q[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int el = 4 * ii + t;
              const uint32_t h = (el & 1) ? (e[el >> 1] >> 16) : (e[el >> 1] & 0xffffu);
              q[t] = round_clip(__fmul_rn(bf16_bits_to_float(h), sc.inv), -128.f, 127.f);
            }
            wd[ii] = pack_i8x4(q[0], q[1], q[2], q[3]);
          }
          const uint4 packed = make_uint4(wd[0], wd[1], wd[2], wd[3]);
          *reinterpret_cast<uint4*>(xs + (int64_t)m * a.xs_bytes + 16 * f) = packed;
          if (blockIdx.x == 0 && ph.xq_out != nullptr)
            *reinterpret_cast<uint4*>(ph.xq_out + (int64_t)m * K + 16 * f) = packed;
        }
        if (blockIdx.x == 0 && tid == 0 && ph.xs_out != nullptr) ph.xs_out[m] = xscale[m];
      }
      consumer_sync();
      if (tid == 0) *(volatile int*)&s_xgate = ph_i + 1;  // x is read: the weights may stream
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= a.M) continue;
#pragma unroll
        for (int j = 0; j < J; ++j) {
          if (j >= valid_j) continue;
          const int c = k_lo + lane + 32 * j;
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint4 v =
                *reinterpret_cast<const uint4*>(xs + (int64_t)m * a.xs_bytes + 64 * c + 16 * s);
            xr[m][j][s] = v;
            lsum[m] = dp4a_ss(v.x, 0x01010101u, lsum[m]);
            lsum[m] = dp4a_ss(v.y, 0x01010101u, lsum[m]);
            lsum[m] = dp4a_ss(v.z, 0x01010101u, lsum[m]);
            lsum[m] = dp4a_ss(v.w, 0x01010101u, lsum[m]);
          }
        }
      }
    } else {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= a.M) continue;
        xscale[m] = ph.x_scale[m];
#pragma unroll
        for (int j = 0; j < J; ++j) {
          if (j >= valid_j) continue;
          const int c = k_lo + lane + 32 * j;
          const uint4* src = reinterpret_cast<const uint4*>(ph.xq + (int64_t)m * K + 64 * c);
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint4 v = ld_nc_v4(src + s);
            xr[m][j][s] = v;
            lsum[m] = dp4a_ss(v.x, 0x01010101u, lsum[m]);
            lsum[m] = dp4a_ss(v.y, 0x01010101u, lsum[m]);
            lsum[m] = dp4a_ss(v.z, 0x01010101u, lsum[m]);
            lsum[m] = dp4a_ss(v.w, 0x01010101u, lsum[m]);
          }
        }
      }
      consumer_sync();
      if (tid == 0) *(volatile int*)&s_xgate = ph_i + 1;  // x is read: the weights may stream
    }

    // On a time-out a warp sets s_abort and from then on every warp only
    // walks the stage sequence (no waits, no work) so that all of them reach
    // the same named barriers; the phase loop then ends uniformly.
    if (!CHAIN && tid == 0)
      for (int m = 0; m < MT; ++m) s_xscale[m] = xscale[m];
    const int full_rows = ph.rows_per_stage / nwr;  // rows of a full stage per warp
    for_each_stage(ph, [&](int p, int row0, int nrows) {
      const int slot = c_slot;
      const uint32_t parity = c_parity;
      if (++c_slot == a.stages) {
        c_slot = 0;
        c_parity ^= 1u;
      }
      if (*(volatile int*)&s_abort) return true;
      if (!mbar_wait(smem_addr(&full_bar[slot]), parity)) {
        if (lane == 0) atomicOr(&g_decode_error, 1 << kErrFullWait);
        *(volatile int*)&s_abort = 1;
        return true;
      }
      const float wsc = CHAIN ? __shfl_sync(0xffffffffu, ws_lane, p) : 0.0f;
      const uint32_t sbase = ring + slot * a.slot_bytes + 16 * (k_lo + lane);
      // Rows wr + q*nwr (q < my_rows <= kMaxRowsPerWarp) of the stage, two at
      // a time; their warp sums are uniform across the lanes.
      const int my_rows = nrows == ph.rows_per_stage
                              ? full_rows
                              : (nrows > wr ? (nrows - wr + nwr - 1) / nwr : 0);
      // Lane q*MT + m keeps the (warp-uniform) sum of row q for token m.
      int tot = 0;
#pragma unroll
      for (int q = 0; q < kMaxRowsPerWarp; q += 2) {
        if (q + 1 < my_rows) {
          const uint32_t w[2] = {sbase + (uint32_t)((wr + q * nwr) * row_bytes),
                                 sbase + (uint32_t)((wr + (q + 1) * nwr) * row_bytes)};
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
          const uint32_t w[1] = {sbase + (uint32_t)((wr + q * nwr) * row_bytes)};
          int v[1][MT];
          row_partials<MT, J, 1>(w, valid_j, xr, v);
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const int s0 = __reduce_add_sync(0xffffffffu, v[0][m] - lsum[m]);
            if (lane == q * MT + m) tot = s0;
          }
        }
      }
      // Lane q*MT + m finishes row q for token m: all rows of the stage at once.
      {
        const int q = lane / MT, m = lane % MT;
        if (!CHAIN) {
          // The producer sums the K parts and writes the row.
          if (q < my_rows && q < kMaxRowsPerWarp)
            s_part[slot][kw * ph.rows_per_stage + wr + q * nwr][m] = tot;
        } else if (q < my_rows && q < kMaxRowsPerWarp && m < a.M) {
          float xsc = xscale[0];
#pragma unroll
          for (int mm = 1; mm < MT; ++mm)
            if (mm == m) xsc = xscale[mm];
          const int row = wr + q * nwr;
          bool last = true;
          if (ph.wk > 1) {
            // Merge the K parts: the last part to arrive writes the row.  Each
            // part adds 1 << 48 (the count) plus its value biased by 2^31
            // (non-negative, below 2^32), so at most 8 parts never carry out
            // of the low 48 bits.
            const unsigned long long add =
                (1ull << 48) + (unsigned long long)((long long)tot + 2147483648ll);
            const unsigned long long old = atomicAdd(&s_acc[slot][row][m], add);
            last = (int)(old >> 48) == ph.wk - 1;
            if (last) {
              const long long sum = (long long)((old + add) & 0xffffffffffffull);
              tot = (int)(sum - (long long)ph.wk * 2147483648ll);
              s_acc[slot][row][m] = 0ull;
            }
          }
          if (last) {
            const Target& T = ph.t[p];
            const int64_t o = (int64_t)m * T.N + row0 + row;
            T.y[o] = __fmul_rn(__int2float_rn(tot), __fmul_rn(xsc, wsc));
            if (T.acc_out) T.acc_out[o] = tot;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[slot]));
      return true;
    });
    // This CTA's outputs of the phase are written.  In a chain: after the
    // CTA barrier one thread makes them visible GPU-wide (a fence is
    // cumulative over what the CTA barrier ordered) and arrives at the grid
    // barrier.
    if (consumer_sync_or(*(volatile int*)&s_abort)) break;
    if (CHAIN && ph_i + 1 < a.nphases && tid == 0) {
      __threadfence();
      atomicAdd(a.barrier, 1ull);
    }
  }
}

// Work split of one phase for MT tokens per pass and J chunks per lane.
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

bool plan_phase(int64_t K, int j, PhasePlan* pp) {
  if (K < 64 || K % 64 != 0 || K > 65536) return false;
  const int nch = (int)(K / 64);
  int wk = 0;
  for (int w = 1; w <= 8; w *= 2)
    if ((nch + w - 1) / w <= 32 * j) {
      wk = w;
      break;
    }
  if (!wk) return false;
  const int nwr = kConsumerWarps / wk;
  const int64_t row_bytes = K / 4;
  int64_t R = kStageTarget / row_bytes / nwr * nwr;
  if (R < nwr) R = nwr;
  if (R > (int64_t)kMaxRowsPerWarp * nwr) R = (int64_t)kMaxRowsPerWarp * nwr;
  pp->wk = wk;
  pp->kpart = (nch + wk - 1) / wk;
  pp->rows_per_stage = (int)R;
  pp->stage_bytes = (int)(R * row_bytes);
  return true;
}

// Ring depth and shared memory for a slot size and a staging width.
int ring_stages(int slot_bytes) {
  int S = kRingBudget / slot_bytes;
  if (S < 2) S = 2;
  if (S > kMaxStages) S = kMaxStages;
  return S;
}

struct Plan {
  int mt, j;
  PhasePlan pp;
  int stages;
  size_t smem;
};

bool make_plan(int64_t M, int64_t K, Plan* pl) {
  if (M < 1 || M > kDecodeMaxM) return false;
  pl->mt = tokens_per_pass(M);
  pl->j = min_j(pl->mt, K);
  if (!pl->j || !plan_phase(K, pl->j, &pl->pp)) return false;
  pl->stages = ring_stages(pl->pp.stage_bytes);
  pl->smem = (size_t)pl->stages * pl->pp.stage_bytes + (size_t)pl->mt * (size_t)K;
  return pl->smem <= (size_t)kMaxSmem;
}

template <int MT, int J, bool CHAIN>
cudaError_t configure(int smem_needed) {
  (void)smem_needed;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(k_gemv_decode<MT, J, CHAIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return cudaSuccess;
}

template <int MT, int J>
cudaError_t launch_t(const Args& a, int ctas, size_t smem, cudaStream_t s) {
  cudaError_t e = configure<MT, J, false>((int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_gemv_decode<MT, J, false>, dim3(ctas), dim3(kThreads), smem, s, a);
}

// Chains run as a cooperative launch (all CTAs resident: the grid barrier
// needs it).
template <int MT, int J>
cudaError_t launch_coop(const Args& a, int ctas, size_t smem, cudaStream_t s) {
  cudaError_t e = configure<MT, J, true>((int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemv_decode<MT, J, true>, a);
}

cudaError_t dispatch(int mt, int j, bool coop, const Args& a, int ctas, size_t smem,
                     cudaStream_t s) {
  if (mt == 1 && j == 2) return coop ? launch_coop<1, 2>(a, ctas, smem, s) : launch_t<1, 2>(a, ctas, smem, s);
  if (mt == 1 && j == 4) return coop ? launch_coop<1, 4>(a, ctas, smem, s) : launch_t<1, 4>(a, ctas, smem, s);
  if (mt == 2 && j == 2) return coop ? launch_coop<2, 2>(a, ctas, smem, s) : launch_t<2, 2>(a, ctas, smem, s);
  if (mt == 4 && j == 1) return coop ? launch_coop<4, 1>(a, ctas, smem, s) : launch_t<4, 1>(a, ctas, smem, s);
  return cudaErrorNotSupported;
}

// The fixed shared memory of one single-phase CTA (its static arrays plus the
// per-block reservation) and how many CTAs of the variant (mt, j) the
// registers allow per SM.
template <int MT, int J>
cudaError_t fixed_smem(size_t* fixed, int* reg_ctas) {
  static size_t cached[64] = {};
  static int cached_ctas[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && cached[dev]) {
    *fixed = cached[dev];
    *reg_ctas = cached_ctas[dev];
    return cudaSuccess;
  }
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, k_gemv_decode<MT, J, false>);
  int reserved = 0, regs_sm = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  *fixed = fa.sharedSizeBytes + (size_t)reserved;
  // registers are allocated per warp in units of 256
  const int per_warp = (fa.numRegs * 32 + 255) / 256 * 256;
  *reg_ctas = regs_sm / (per_warp * ((kThreads + 31) / 32));
  if (dev < 64) {
    cached[dev] = *fixed;
    cached_ctas[dev] = *reg_ctas;
  }
  return cudaSuccess;
}

cudaError_t sm_smem(size_t* cap) {
  int dev = 0, v = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  *cap = (size_t)v;
  return e;
}

cudaError_t variant_fixed_smem(int mt, int j, size_t* fixed, int* reg_ctas) {
  if (mt == 1 && j == 2) return fixed_smem<1, 2>(fixed, reg_ctas);
  if (mt == 1 && j == 4) return fixed_smem<1, 4>(fixed, reg_ctas);
  if (mt == 2 && j == 2) return fixed_smem<2, 2>(fixed, reg_ctas);
  if (mt == 4 && j == 1) return fixed_smem<4, 1>(fixed, reg_ctas);
  return cudaErrorNotSupported;
}

// Fills a Phase from the host description; rows split over `ctas` CTAs.
bool fill_phase(const DecodeTarget* targets, int count, const int8_t* xq, const float* x_scale,
                const uint16_t* x_bf16, int64_t K, const PhasePlan& pp, int ctas,
                int8_t* xq_out, float* x_scale_out, Phase* ph) {
  *ph = Phase{};
  int64_t rows = 0;
  for (int p = 0; p < count; ++p) {
    ph->t[p].Wq = targets[p].Wq;
    ph->t[p].w_scale = targets[p].w_scale;
    ph->t[p].y = targets[p].y;
    ph->t[p].acc_out = targets[p].acc_out;
    ph->t[p].row0 = (int)rows;
    ph->t[p].N = (int)targets[p].N;
    rows += targets[p].N;
  }
  if (rows < 1 || rows > (1 << 30)) return false;
  ph->count = count;
  ph->rows_total = (int)rows;
  ph->rows_per_cta = (int)((rows + ctas - 1) / ctas);
  ph->xb = x_bf16;
  ph->xq = xq;
  ph->x_scale = x_scale;
  ph->xq_out = xq_out;
  ph->xs_out = x_scale_out;
  ph->K = (int)K;
  ph->wk = pp.wk;
  ph->kpart = pp.kpart;
  ph->rows_per_stage = pp.rows_per_stage;
  ph->stage_bytes = pp.stage_bytes;
  return true;
}

constexpr int kChainCtas = 148;
constexpr size_t kChainHeader = 256;  // the barrier word, padded

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
  int64_t rows = 0;
  for (int p = 0; p < count; ++p) rows += targets[p].N;
  // One CTA per SM leaves room for the next decode kernel to start alongside
  // (programmatic dependent launch); large matrices take two per SM for more
  // warps and copies in flight, with the ring shortened (to no fewer than two
  // stages) until two CTAs fit in an SM's shared memory.
  bool two = rows * (K / 4) >= ((int64_t)16 << 20);
  if (two) {
    size_t cap = 0, fixed = 0;
    int reg_ctas = 0;
    cudaError_t e = sm_smem(&cap);
    if (e == cudaSuccess) e = variant_fixed_smem(pl.mt, pl.j, &fixed, &reg_ctas);
    if (e != cudaSuccess) return e;
    if (reg_ctas >= 2) {
      while (pl.stages > 2 && 2 * (pl.smem + fixed) > cap) {
        --pl.stages;
        pl.smem -= (size_t)pl.pp.stage_bytes;
      }
    }
    two = reg_ctas >= 2 && 2 * (pl.smem + fixed) <= cap;
  }
  const int64_t max_ctas = two ? 296 : 148;
  int64_t ctas = rows < max_ctas ? rows : max_ctas;
  const int64_t rpc = (rows + ctas - 1) / ctas;
  ctas = (rows + rpc - 1) / rpc;
  Args a = {};
  if (!fill_phase(targets, count, xq, x_scale, x_bf16, K, pl.pp, (int)ctas, xq_out, x_scale_out,
                  &a.ph0))
    return cudaErrorNotSupported;
  a.phases = nullptr;
  a.barrier = nullptr;
  a.nphases = 1;
  a.M = (int)M;
  a.stages = pl.stages;
  a.slot_bytes = pl.pp.stage_bytes;
  a.xs_bytes = (int)K;
  a.weights_early = weights_static ? 1 : 0;
  return dispatch(pl.mt, pl.j, false, a, (int)ctas, pl.smem, s);
}

size_t decode_chain_bytes(int nphases) {
  return kChainHeader + (size_t)(nphases > 0 ? nphases : 0) * sizeof(Phase);
}

cudaError_t build_decode_chain(const DecodePhaseDesc* phases, int nphases, int64_t M,
                               void* table, DecodeChainConfig* cfg) {
  if (nphases < 1 || M < 1 || M > kDecodeMaxM) return cudaErrorNotSupported;
  const int mt = tokens_per_pass(M);
  int j = 0;
  int64_t max_k = 0;
  for (int i = 0; i < nphases; ++i) {
    const int jj = min_j(mt, phases[i].K);
    if (!jj || phases[i].count < 1 || phases[i].count > kDecodeMaxTargets)
      return cudaErrorNotSupported;
    if (jj > j) j = jj;
    if (phases[i].K > max_k) max_k = phases[i].K;
  }
  Phase* host = new Phase[nphases];
  int slot = 0;
  for (int i = 0; i < nphases; ++i) {
    PhasePlan pp;
    if (!plan_phase(phases[i].K, j, &pp) ||
        !fill_phase(phases[i].targets, phases[i].count, nullptr, nullptr, phases[i].x,
                    phases[i].K, pp, kChainCtas, nullptr, nullptr, &host[i])) {
      delete[] host;
      return cudaErrorNotSupported;
    }
    if (pp.stage_bytes > slot) slot = pp.stage_bytes;
  }
  const int stages = ring_stages(slot);
  const size_t smem = (size_t)stages * slot + (size_t)mt * (size_t)max_k;
  if (smem > (size_t)kMaxSmem) {
    delete[] host;
    return cudaErrorNotSupported;
  }
  uint8_t* t = static_cast<uint8_t*>(table);
  cudaError_t e = cudaMemset(t, 0, kChainHeader);
  if (e == cudaSuccess)
    e = cudaMemcpy(t + kChainHeader, host, (size_t)nphases * sizeof(Phase), cudaMemcpyHostToDevice);
  delete[] host;
  if (e != cudaSuccess) return e;
  cfg->mt = mt;
  cfg->j = j;
  cfg->stages = stages;
  cfg->slot_bytes = slot;
  cfg->xs_bytes = (int)max_k;
  cfg->smem = (int)smem;
  return cudaSuccess;
}

cudaError_t launch_decode_chain(const void* table, int nphases, int64_t M,
                                const DecodeChainConfig& cfg, cudaStream_t s) {
  Args a = {};
  uint8_t* t = static_cast<uint8_t*>(const_cast<void*>(table));
  a.phases = reinterpret_cast<const Phase*>(t + kChainHeader);
  a.barrier = reinterpret_cast<unsigned long long*>(t);
  a.nphases = nphases;
  a.M = (int)M;
  a.stages = cfg.stages;
  a.slot_bytes = cfg.slot_bytes;
  a.xs_bytes = cfg.xs_bytes;
  a.weights_early = 0;
  return dispatch(cfg.mt, cfg.j, true, a, kChainCtas, (size_t)cfg.smem, s);
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
