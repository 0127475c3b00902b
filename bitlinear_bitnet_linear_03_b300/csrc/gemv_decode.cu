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
//  * The consumers store each row's K-part result in shared memory and
//    release the slot; the producer warp, when it takes the slot back for a
//    new copy, sums the parts and writes the stage's outputs (rows across its
//    lanes, coalesced).  The consumers' per-stage work is then only the dot
//    products.
//  * Before waiting on the previous kernel the CTA asks for its whole weight
//    range and its input to be prefetched into L2 and lets its successor
//    launch:
//    consecutive decode kernels overlap under programmatic dependent launch.
//    Weights are read after that wait, unless the caller declared them
//    static (not written by any work still in flight): then the producer
//    issues the first stages while the previous kernel finishes.  The rest
//    of the stages wait until the consumers have read the input x, whose
//    loads would otherwise queue behind the weight copies.
//  * Up to kDecodeMaxTargets matrices sharing the same input run in one
//    launch; their rows are concatenated, stages never straddle two matrices.
//  * The input is int8 with its scales, or bf16: then every CTA forms the
//    per-token absmax over all of K and quantises x with the rule of the
//    activation-quantisation kernel (bit-identical codes).
//  * Outputs: y (binary32) and/or y_bf16 (y rounded to the nearest bf16).
//  * Every mbarrier wait is bounded (about a second by default); on time-out
//    the kernel records an error code, stops issuing copies, waits (bounded)
//    for the copies it has in flight and returns.
#include "decode_common.cuh"

namespace bitnet {

__device__ int g_decode_error;

namespace {
using namespace dec;

constexpr int kMaxStages = 8;
constexpr int kRingBudget = 96 * 1024;
constexpr int kStageTarget = 24 * 1024;
// Stages the producer issues before the consumers have read the input x, so
// that the input's loads do not queue behind a full ring of weight copies
// (measured on B300: 3-4% faster for a 58 MB matrix).
constexpr int kEarlyStages = 1;
constexpr int kMaxSmem = 227 * 1024 - 10 * 1024;  // dynamic part; the static arrays fit in the rest
constexpr int kPrefetchMax = 1 << 16;
constexpr int kErrFullWait = 1;
constexpr int kErrEmptyWait = 2;
constexpr int kErrDrainWait = 3;

struct Target {
  const uint8_t* Wq;
  const float* w_scale;
  float* y;
  uint16_t* y_bf16;
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

struct Args {
  Phase ph;
  int M;
  int stages;
  int slot_bytes;
  int xs_bytes;       // per-token int8 staging (K)
  int weights_early;  // weights may be read before the previous kernel ends
  long long wait;     // bound of every wait but the final drain, in clocks
};

// The CTA's stage sequence: for each matrix overlapping the CTA's rows, the
// rows in pieces of at most rows_per_stage.  Calls f(p, first_row, nrows) in
// order; returns false if f stopped it.
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

// L2 prefetch hint for the CTA's weight rows.
__device__ __forceinline__ void prefetch_weights(const Phase& ph) {
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

// L2 prefetch hint for the input x (bf16 or int8, M rows).
__device__ __forceinline__ void prefetch_x(const Phase& ph, int M) {
  const void* p = ph.xb != nullptr ? (const void*)ph.xb : (const void*)ph.xq;
  const int64_t bytes = (int64_t)M * ph.K * (ph.xb != nullptr ? 2 : 1);
  for (int64_t off = 0; off < bytes; off += kPrefetchMax)
    prefetch_l2_bulk(static_cast<const uint8_t*>(p) + off,
                     (uint32_t)(bytes - off < kPrefetchMax ? bytes - off : kPrefetchMax));
}

// What the producer records when it fills a ring slot, read back when the
// consumers release the slot and it writes the stage's outputs.
struct StageRec {
  int p, row0, nrows;
};

// The consumers leave each row's K-part results in shared memory and release
// the slot; the producer warp writes the stage's outputs while the next
// stages are consumed.
template <int MT, int J>
__global__ void __launch_bounds__(kThreads, MT <= 2 ? 2 : 1)
k_gemv_decode(const __grid_constant__ Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ float s_max[kConsumerWarps][MT];
  __shared__ int s_abort;
  __shared__ int s_xgate;  // 1 once the consumers have read the input x
  // The phase descriptor in shared memory (read in the hot loop).
  __shared__ __align__(16) Phase s_ph;
  // Each K part's row result (part kw of stage row r at kw * R + r), the
  // stage records and the activation scales.
  __shared__ int s_part[kMaxStages][kConsumerWarps * kMaxRowsPerWarp][MT];
  __shared__ StageRec s_stage[kMaxStages];
  __shared__ float s_xscale[MT];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = smem_addr(smem);

  if (threadIdx.x < 32) {
    static_assert(sizeof(Phase) % 8 == 0, "phase descriptor is copied in 8-byte words");
    const unsigned long long* src = reinterpret_cast<const unsigned long long*>(&a.ph);
    unsigned long long* dst = reinterpret_cast<unsigned long long*>(&s_ph);
    for (int i = lane; i < (int)(sizeof(Phase) / 8); i += 32) dst[i] = src[i];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kConsumerWarps);
    }
    mbar_fence_init();
    s_abort = 0;
    s_xgate = 0;
    // L2 prefetch hints for the input and the weights (no data is read
    // before the dependency wait).
    prefetch_x(a.ph, a.M);
    prefetch_weights(a.ph);
  }
  griddep_launch_dependents();
  __syncthreads();

  // ------------------------------------------------------------ producer
  // Lane 0 fills the ring with bulk copies; the whole warp writes the
  // outputs of each stage the consumers have released (y = acc * (x_scale *
  // w_scale), rows across the lanes).
  if (warp == kConsumerWarps) {
    // Weights the caller declared static may stream in while the previous
    // kernel on the stream is still running (the first stages); otherwise
    // wait for it first.  Either way every bounded wait below starts after
    // the dependency wait.
    bool dep_done = !a.weights_early;
    if (dep_done) griddep_wait();
    const int S = a.stages;
    const Phase& ph = s_ph;
    const float ws_lane = lane < ph.count ? *ph.t[lane].w_scale : 0.0f;
    auto finish = [&](int slot) {
      const StageRec rec = s_stage[slot];
      const Target& T = ph.t[rec.p];
      const float wsc = __shfl_sync(0xffffffffu, ws_lane, rec.p);
      const int R = ph.rows_per_stage, wk = ph.wk;
      for (int m = 0; m < a.M; ++m) {
        const float c = __fmul_rn(s_xscale[m], wsc);
        for (int r = lane; r < rec.nrows; r += 32) {
          int tot = 0;
          for (int kw = 0; kw < wk; ++kw) tot += s_part[slot][kw * R + r][m];
          const int64_t o = (int64_t)m * T.N + rec.row0 + r;
          const float y = __fmul_rn(__int2float_rn(tot), c);
          if (T.y) T.y[o] = y;
          if (T.y_bf16) T.y_bf16[o] = f32_to_bf16_rn(y);
          if (T.acc_out) T.acc_out[o] = tot;
        }
      }
    };
    int i = 0, done = 0;
    const int64_t row_bytes = ph.K >> 2;
    bool ok = for_each_stage(ph, [&](int p, int row, int nrows) {
      const int slot = i % S, use = i / S;
      if (i == kEarlyStages) {
        // wait (bounded) until the consumers have read the input
        const long long t0 = clock64();
        while (*(volatile int*)&s_xgate == 0) {
          if (*(volatile int*)&s_abort) return false;
          if (clock64() - t0 > a.wait) {
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
        if (!mbar_wait(smem_addr(&empty_bar[slot]), (use - 1) & 1, a.wait) ||
            *(volatile int*)&s_abort) {
          if (lane == 0) atomicOr(&g_decode_error, 1 << kErrEmptyWait);
          *(volatile int*)&s_abort = 1;
          return false;
        }
        finish(slot);
        ++done;
      }
      if (lane == 0) {
        s_stage[slot] = StageRec{p, row, nrows};
        const uint32_t bytes = (uint32_t)(nrows * row_bytes);
        const uint32_t fb = smem_addr(&full_bar[slot]);
        mbar_arrive_expect_tx(fb, bytes);
        bulk_copy_g2s(ring + slot * a.slot_bytes, ph.t[p].Wq + (int64_t)row * row_bytes, bytes,
                      fb);
      }
      __syncwarp();
      ++i;
      return true;
    });
    if (!dep_done) griddep_wait();
    // The stages still in the ring.
    for (; ok && done < i; ++done) {
      const int slot = done % S;
      if (!mbar_wait(smem_addr(&empty_bar[slot]), (done / S) & 1, a.wait) ||
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
        if (!mbar_wait(smem_addr(&full_bar[j % S]), (j / S) & 1, kDrainCycles)) {
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
  const Phase& ph = s_ph;
  const int K = ph.K;
  const int64_t row_bytes = K >> 2;
  // This warp: K part kw (chunks k_lo .. k_hi-1) and row group wr of 8/wk.
  // Lane l holds the int8 activations of chunks k_lo + l + 32j (j < J) in
  // registers and the sum of those codes, which it subtracts from every
  // row's partial (sum q x = sum c x - sum x, taken part by part).
  const int kw = warp % ph.wk, wr = warp / ph.wk, nwr = kConsumerWarps / ph.wk;
  const int nch = K >> 6;
  const int k_lo = kw * ph.kpart, k_hi = min(nch, k_lo + ph.kpart);
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
          // eight loads in flight per thread, then their maxima (a value
          // past K reads as 0, which leaves the maximum unchanged)
          const int nv = K >> 3;
          for (int v0 = tid; v0 < nv; v0 += 8 * kConsumers) {
            uint4 q[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              q[u] = v0 + u * kConsumers < nv ? ld_nc_v4(xrow + v0 + u * kConsumers)
                                              : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint32_t w4[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                mx = fmaxf(mx, fabsf(bf16_bits_to_float(w4[t] & 0xffffu)));
                mx = fmaxf(mx, fabsf(bf16_bits_to_float(w4[t] >> 16)));
              }
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
      // two-pass inputs: the pieces of four steps are loaded before any is
      // quantised (the loads of pass two mostly hit in L1)
      uint4 pre[4][2];
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
          if ((j & 3) == 0) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int fu = f + u * kConsumers;
              pre[u][0] = fu < nitems ? ld_nc_v4(xrow + 2 * fu) : make_uint4(0, 0, 0, 0);
              pre[u][1] = fu < nitems ? ld_nc_v4(xrow + 2 * fu + 1) : make_uint4(0, 0, 0, 0);
            }
          }
          uint4 h0 = pre[0][0], h1 = pre[0][1];
#pragma unroll
          for (int u = 1; u < 4; ++u)
            if ((j & 3) == u) h0 = pre[u][0], h1 = pre[u][1];
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
    if (tid == 0) *(volatile int*)&s_xgate = 1;  // x is read: the weights may stream
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
    if (tid == 0) *(volatile int*)&s_xgate = 1;  // x is read: the weights may stream
  }
  if (tid == 0)
    for (int m = 0; m < MT; ++m) s_xscale[m] = xscale[m];

  // On a time-out a warp sets s_abort and from then on every warp only walks
  // the stage sequence (no waits, no work).
  const int full_rows = ph.rows_per_stage / nwr;  // rows of a full stage per warp
  int c_slot = 0;
  uint32_t c_parity = 0;
  for_each_stage(ph, [&](int p, int row0, int nrows) {
    (void)p;
    (void)row0;
    const int slot = c_slot;
    const uint32_t parity = c_parity;
    if (++c_slot == a.stages) {
      c_slot = 0;
      c_parity ^= 1u;
    }
    if (*(volatile int*)&s_abort) return true;
    if (!mbar_wait(smem_addr(&full_bar[slot]), parity, a.wait)) {
      if (lane == 0) atomicOr(&g_decode_error, 1 << kErrFullWait);
      *(volatile int*)&s_abort = 1;
      return true;
    }
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
    // Lane q*MT + m leaves row q's K-part sum for token m; the producer sums
    // the K parts and writes the row.
    {
      const int q = lane / MT, m = lane % MT;
      if (q < my_rows && q < kMaxRowsPerWarp)
        s_part[slot][kw * ph.rows_per_stage + wr + q * nwr][m] = tot;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[slot]));
    return true;
  });
}

// Work split for MT tokens per pass and J chunks per lane.
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

// Ring depth for a slot size.
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

template <int MT, int J>
cudaError_t launch_t(const Args& a, int ctas, size_t smem, cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(k_gemv_decode<MT, J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return launch_pdl(k_gemv_decode<MT, J>, dim3(ctas), dim3(kThreads), smem, s, a);
}

cudaError_t dispatch(int mt, int j, const Args& a, int ctas, size_t smem, cudaStream_t s) {
  if (mt == 1 && j == 2) return launch_t<1, 2>(a, ctas, smem, s);
  if (mt == 1 && j == 4) return launch_t<1, 4>(a, ctas, smem, s);
  if (mt == 2 && j == 2) return launch_t<2, 2>(a, ctas, smem, s);
  if (mt == 4 && j == 1) return launch_t<4, 1>(a, ctas, smem, s);
  return cudaErrorNotSupported;
}

// The fixed shared memory of one CTA (its static arrays plus the per-block
// reservation) and how many CTAs of the variant (mt, j) the registers allow
// per SM.
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
  e = cudaFuncGetAttributes(&fa, k_gemv_decode<MT, J>);
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

cudaError_t variant_fixed_smem(int mt, int j, size_t* fixed, int* reg_ctas) {
  if (mt == 1 && j == 2) return fixed_smem<1, 2>(fixed, reg_ctas);
  if (mt == 1 && j == 4) return fixed_smem<1, 4>(fixed, reg_ctas);
  if (mt == 2 && j == 2) return fixed_smem<2, 2>(fixed, reg_ctas);
  if (mt == 4 && j == 1) return fixed_smem<4, 1>(fixed, reg_ctas);
  return cudaErrorNotSupported;
}

cudaError_t device_info(int* sms, size_t* smem_per_sm) {
  static int cached_sms[64] = {};
  static size_t cached_smem[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cached_sms[dev]) {
    *sms = cached_sms[dev];
    *smem_per_sm = cached_smem[dev];
    return cudaSuccess;
  }
  int n = 0, v = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  *sms = n;
  *smem_per_sm = (size_t)v;
  if (dev >= 0 && dev < 64) {
    cached_sms[dev] = n;
    cached_smem[dev] = (size_t)v;
  }
  return cudaSuccess;
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
    ph->t[p].y_bf16 = targets[p].y_bf16;
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

}  // namespace

bool decode_supported(int64_t M, int64_t K) {
  Plan pl;
  return make_plan(M, K, &pl);
}

cudaError_t launch_decode(const DecodeTarget* targets, int count, const int8_t* xq,
                          const float* x_scale, const uint16_t* x_bf16, int64_t M, int64_t K,
                          int8_t* xq_out, float* x_scale_out, bool weights_static,
                          long long wait_cycles, cudaStream_t s) {
  Plan pl;
  if (count < 1 || count > kDecodeMaxTargets || !make_plan(M, K, &pl))
    return cudaErrorNotSupported;
  int64_t rows = 0;
  for (int p = 0; p < count; ++p) rows += targets[p].N;
  int sms = 0;
  size_t cap = 0;
  cudaError_t e = device_info(&sms, &cap);
  if (e != cudaSuccess) return e;
  // One CTA per SM leaves room for the next decode kernel to start alongside
  // (programmatic dependent launch); large matrices take two per SM for more
  // warps and copies in flight, with the ring shortened (to no fewer than two
  // stages) until two CTAs fit in an SM's shared memory.
  bool two = rows * (K / 4) >= ((int64_t)16 << 20);
  if (two) {
    size_t fixed = 0;
    int reg_ctas = 0;
    e = variant_fixed_smem(pl.mt, pl.j, &fixed, &reg_ctas);
    if (e != cudaSuccess) return e;
    if (reg_ctas >= 2) {
      while (pl.stages > 2 && 2 * (pl.smem + fixed) > cap) {
        --pl.stages;
        pl.smem -= (size_t)pl.pp.stage_bytes;
      }
    }
    two = reg_ctas >= 2 && 2 * (pl.smem + fixed) <= cap;
  }
  const int64_t max_ctas = two ? 2 * (int64_t)sms : (int64_t)sms;
  int64_t ctas = rows < max_ctas ? rows : max_ctas;
  const int64_t rpc = (rows + ctas - 1) / ctas;
  ctas = (rows + rpc - 1) / rpc;
  Args a = {};
  if (!fill_phase(targets, count, xq, x_scale, x_bf16, K, pl.pp, (int)ctas, xq_out, x_scale_out,
                  &a.ph))
    return cudaErrorNotSupported;
  a.M = (int)M;
  a.stages = pl.stages;
  a.slot_bytes = pl.pp.stage_bytes;
  a.xs_bytes = (int)K;
  a.weights_early = weights_static ? 1 : 0;
  a.wait = wait_cycles;
  return dispatch(pl.mt, pl.j, a, (int)ctas, pl.smem, s);
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
