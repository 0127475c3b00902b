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
//  * Lane l of a warp owns 64-weight chunks l, l+32, ... of its K-slice for
//    the whole kernel, so its int8 activations (and their byte sum) sit in
//    registers from the prologue on; each weight row is then read as 512
//    contiguous bytes per warp step and never touches shared memory.
//  * The 8 warps of a CTA split K into `ksplit` slices and the CTA's rows
//    into 8/ksplit row groups; a row group handles kB rows per step.  Partial
//    row sums are combined with a reduce-scatter over the lanes (kB*MT values
//    in log2 steps) and, across K-slices, through shared memory.
//  * Before waiting on the previous kernel, one thread asks the copy engine
//    to prefetch the CTA's whole weight range into L2 (weights never depend on
//    the previous kernel), and the kernel lets its successor launch; with
//    programmatic dependent launch consecutive decode kernels overlap.
//  * Up to kDecodeMaxTargets matrices sharing the same input run in one
//    launch: their rows are concatenated into one row space.
//  * The input is int8 with its scales, or bf16: then every CTA forms the
//    per-token absmax over all of K and quantises its own chunks with the
//    rule of the activation-quantisation kernel (bit-identical codes).
#include "common.cuh"

namespace bitnet {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kB = 4;           // rows per row-group step
constexpr int kPrefetchMax = 1 << 16;

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
  int M, K, ksplit, slice_chunks;
};

__device__ __forceinline__ uint32_t bf16_pair_lo(uint32_t w) { return w & 0xffffu; }
__device__ __forceinline__ uint32_t bf16_pair_hi(uint32_t w) { return w >> 16; }

// Reduce-scatter of V per-lane values over the warp: afterwards every lane
// holds the warp-wide total of value index(lane) (see value_index).
template <int V>
__device__ __forceinline__ int reduce_scatter(int (&v)[V], int lane) {
  int count = V;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (count > 1) {
      const int half = count >> 1;
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < V / 2; ++i) {
        if (i < half) {
          const int send = upper ? v[i] : v[i + half];
          const int keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      count = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
  return v[0];
}

// Index of the value a lane holds after reduce_scatter<V>: the stage with
// offset 16 keeps the upper half on lanes with bit 4 set, and so on.
template <int V>
__device__ __forceinline__ int value_index(int lane) {
  int idx = 0, half = V >> 1;
#pragma unroll
  for (int off = 16; off >= 1 && half >= 1; off >>= 1, half >>= 1)
    if (lane & off) idx += half;
  return idx;
}

// Lanes that write a value after reduce_scatter<V> (one per index).
template <int V>
__device__ __forceinline__ bool value_writer(int lane) {
  return (lane & (32 / V - 1)) == 0;
}

template <int MT, int J>
__global__ void __launch_bounds__(kThreads)
k_gemv_decode(const __grid_constant__ Args a) {
  __shared__ float s_max[kWarps][MT];
  __shared__ int s_part[kWarps][kB * MT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r_begin = blockIdx.x * a.rows_per_cta;
  const int r_end = min(r_begin + a.rows_per_cta, a.rows_total);
  const int64_t row_bytes = a.K >> 2;

  // 1. Prefetch this CTA's weight rows into L2 (independent of the
  //    previous kernel), then let the next kernel launch and wait for ours.
  if (threadIdx.x == 0) {
    for (int p = 0; p < a.count; ++p) {
      const int lo = max(r_begin, a.t[p].row0);
      const int hi = min(r_end, a.t[p].row0 + a.t[p].N);
      if (lo >= hi) continue;
      const uint8_t* base = a.t[p].Wq + (int64_t)(lo - a.t[p].row0) * row_bytes;
      int64_t bytes = (int64_t)(hi - lo) * row_bytes;
      for (int64_t off = 0; off < bytes; off += kPrefetchMax) {
        const int64_t n = bytes - off < kPrefetchMax ? bytes - off : kPrefetchMax;
        prefetch_l2_bulk(base + off, (uint32_t)n);
      }
    }
  }
  griddep_launch_dependents();
  griddep_wait();

  const int ks = warp % a.ksplit;
  const int rg = warp / a.ksplit;
  const int nrg = kWarps / a.ksplit;
  const int nch = a.K >> 6;
  const int c0 = ks * a.slice_chunks;
  const int c1 = min(c0 + a.slice_chunks, nch);

  // 2. This lane's activation chunks: xr[m][j][s] holds the int8 codes of
  //    weights 64c + 16s + 4i + {0..3} in word i, c = c0 + lane + 32j.
  uint4 xr[MT][J][4];
  int xsum[MT];
  float xscale[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    xsum[m] = 0;
    xscale[m] = 0.0f;
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int s = 0; s < 4; ++s) xr[m][j][s] = make_uint4(0, 0, 0, 0);
  }

  if (a.xb != nullptr) {
    // Per-token absmax over the whole of K, shared by the CTA.
    const int nv = a.K >> 3;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float mx = 0.0f;
      if (m < a.M) {
        const uint4* xrow = reinterpret_cast<const uint4*>(a.xb + (int64_t)m * a.K);
        for (int v = threadIdx.x; v < nv; v += kThreads) {
          const uint4 p = ld_nc_v4(xrow + v);
          const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            mx = fmaxf(mx, fabsf(bf16_bits_to_float(bf16_pair_lo(w4[q]))));
            mx = fmaxf(mx, fabsf(bf16_bits_to_float(bf16_pair_hi(w4[q]))));
          }
        }
      }
      mx = warp_max_f32(mx);
      if (lane == 0) s_max[warp][m] = mx;
    }
    __syncthreads();
    float inv[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float mx = s_max[0][m];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, s_max[w][m]);
      const ActScale sc = act_scale_from_absmax(mx);
      inv[m] = sc.inv;
      xscale[m] = sc.scale;
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = c0 + lane + 32 * j;
      if (c >= c1) continue;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= a.M) continue;
        const uint4* src = reinterpret_cast<const uint4*>(a.xb + (int64_t)m * a.K + c * 64);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          // elements 16s .. 16s+15 of the chunk: two 16-byte loads
          const uint4 p0 = ld_nc_v4(src + 2 * s), p1 = ld_nc_v4(src + 2 * s + 1);
          const uint32_t e[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          uint32_t words[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            int q[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int el = 4 * i + t;
              const uint32_t pair = e[el >> 1];
              const float f = bf16_bits_to_float((el & 1) ? bf16_pair_hi(pair) : bf16_pair_lo(pair));
              q[t] = round_clip(__fmul_rn(f, inv[m]), -128.f, 127.f);
            }
            words[i] = pack_i8x4(q[0], q[1], q[2], q[3]);
            xsum[m] = dp4a_ss(words[i], 0x01010101u, xsum[m]);
          }
          xr[m][j][s] = make_uint4(words[0], words[1], words[2], words[3]);
        }
      }
    }
    // One CTA also stores the quantised input when asked.
    if (blockIdx.x == 0 && a.xq_out != nullptr) {
      for (int m = 0; m < a.M && m < MT; ++m) {
        const uint4* xrow = reinterpret_cast<const uint4*>(a.xb + (int64_t)m * a.K);
        uint2* qrow = reinterpret_cast<uint2*>(a.xq_out + (int64_t)m * a.K);
        float im = inv[0];
#pragma unroll
        for (int mm = 1; mm < MT; ++mm)
          if (mm == m) im = inv[mm];
        for (int v = threadIdx.x; v < nv; v += kThreads) {
          const uint4 p = ld_nc_v4(xrow + v);
          const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
          int q[8];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            q[2 * t] = round_clip(__fmul_rn(bf16_bits_to_float(bf16_pair_lo(w4[t])), im), -128.f, 127.f);
            q[2 * t + 1] = round_clip(__fmul_rn(bf16_bits_to_float(bf16_pair_hi(w4[t])), im), -128.f, 127.f);
          }
          qrow[v] = make_uint2(pack_i8x4(q[0], q[1], q[2], q[3]), pack_i8x4(q[4], q[5], q[6], q[7]));
        }
        if (threadIdx.x == 0 && a.xs_out != nullptr) {
          float sc = xscale[0];
#pragma unroll
          for (int mm = 1; mm < MT; ++mm)
            if (mm == m) sc = xscale[mm];
          a.xs_out[m] = sc;
        }
      }
    }
  } else {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m >= a.M) continue;
      xscale[m] = a.x_scale[m];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int c = c0 + lane + 32 * j;
        if (c >= c1) continue;
        const uint4* src = reinterpret_cast<const uint4*>(a.xq + (int64_t)m * a.K + c * 64);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint4 v = ld_nc_v4(src + s);
          xr[m][j][s] = v;
          xsum[m] = dp4a_ss(v.x, 0x01010101u, xsum[m]);
          xsum[m] = dp4a_ss(v.y, 0x01010101u, xsum[m]);
          xsum[m] = dp4a_ss(v.z, 0x01010101u, xsum[m]);
          xsum[m] = dp4a_ss(v.w, 0x01010101u, xsum[m]);
        }
      }
    }
  }

  // 3. Stream the rows.
  const int per_step = nrg * kB;
  const int nsteps = (a.rows_per_cta + per_step - 1) / per_step;
  constexpr int V = kB * MT;
  const int my_idx = value_index<V>(lane);
  const bool writer = value_writer<V>(lane);

  for (int step = 0; step < nsteps; ++step) {
    const uint8_t* wrow[kB];
    int tgt[kB];
    int rloc[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int gr = r_begin + step * per_step + rg * kB + b;
      wrow[b] = nullptr;
      tgt[b] = -1;
      rloc[b] = 0;
      if (gr < r_end) {
#pragma unroll
        for (int p = 0; p < kDecodeMaxTargets; ++p) {
          if (p < a.count && gr >= a.t[p].row0 && gr < a.t[p].row0 + a.t[p].N) {
            tgt[b] = p;
            rloc[b] = gr - a.t[p].row0;
            wrow[b] = a.t[p].Wq + (int64_t)rloc[b] * row_bytes;
          }
        }
      }
    }
    uint4 w[kB][J];
#pragma unroll
    for (int b = 0; b < kB; ++b)
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int c = c0 + lane + 32 * j;
        w[b][j] = (wrow[b] != nullptr && c < c1) ? ld_stream_v4(wrow[b] + c * 16)
                                                  : make_uint4(0, 0, 0, 0);
      }
    int v[V];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const uint32_t ww[4] = {w[b][j].x, w[b][j].y, w[b][j].z, w[b][j].w};
          const uint32_t x0[4] = {xr[m][j][0].x, xr[m][j][0].y, xr[m][j][0].z, xr[m][j][0].w};
          const uint32_t x1[4] = {xr[m][j][1].x, xr[m][j][1].y, xr[m][j][1].z, xr[m][j][1].w};
          const uint32_t x2[4] = {xr[m][j][2].x, xr[m][j][2].y, xr[m][j][2].z, xr[m][j][2].w};
          const uint32_t x3[4] = {xr[m][j][3].x, xr[m][j][3].y, xr[m][j][3].z, xr[m][j][3].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a0 = dp4a_us(ww[i] & 0x03030303u, x0[i], a0);
            a1 = dp4a_us(ww[i] & 0x0c0c0c0cu, x1[i], a1);
            a2 = dp4a_us(ww[i] & 0x30303030u, x2[i], a2);
            a3 = dp4a_us(ww[i] & 0xc0c0c0c0u, x3[i], a3);
          }
        }
        v[b * MT + m] = a0 + (a1 >> 2) + (a2 >> 4) + (a3 >> 6) - xsum[m];
      }
    }
    int total = reduce_scatter<V>(v, lane);
    if (a.ksplit > 1) {
      if (writer) s_part[warp][my_idx] = total;
      __syncthreads();
      if (writer && ks == 0) {
        total = 0;
        for (int q = 0; q < a.ksplit; ++q) total += s_part[rg * a.ksplit + q][my_idx];
      }
      __syncthreads();
    }
    if (writer && ks == 0) {
      const int b = my_idx / MT, m = my_idx % MT;
      int p = -1, rl = 0;
#pragma unroll
      for (int bb = 0; bb < kB; ++bb)
        if (bb == b) {
          p = tgt[bb];
          rl = rloc[bb];
        }
      if (p >= 0 && m < a.M) {
        float sc = xscale[0];
#pragma unroll
        for (int mm = 1; mm < MT; ++mm)
          if (mm == m) sc = xscale[mm];
        const Target& T = a.t[p];
        T.y[(int64_t)m * T.N + rl] = __fmul_rn(__int2float_rn(total), __fmul_rn(sc, *T.w_scale));
        if (T.acc_out) T.acc_out[(int64_t)m * T.N + rl] = total;
      }
    }
  }
}

struct Shape {
  int mt, j, ksplit, slice_chunks;
};

// Picks the tokens-per-pass MT, chunks per lane J and the K-split so that a
// lane's activations stay within 16*MT*J <= 64 registers and ksplit <= 8.
bool pick_shape(int64_t M, int64_t K, Shape* out) {
  if (M < 1 || M > kDecodeMaxM || K % 64 != 0) return false;
  const int nch = (int)(K / 64);
  const int mt = M <= 1 ? 1 : M <= 2 ? 2 : 4;
  const int jopts[3] = {2, 4, 1};
  for (int jo = 0; jo < 3; ++jo) {
    const int j = jopts[jo];
    if (16 * mt * j > 64 && !(mt == 1 && j == 4)) continue;
    if (mt == 4 && j != 1) continue;
    if (mt == 2 && j != 2) continue;
    int ks = 1;
    while (ks <= 8 && (nch + ks - 1) / ks > 32 * j) ks *= 2;
    if (ks > 8) continue;
    out->mt = mt;
    out->j = j;
    out->ksplit = ks;
    out->slice_chunks = (nch + ks - 1) / ks;
    return true;
  }
  return false;
}

template <int MT, int J>
cudaError_t launch_t(const Args& a, int ctas, cudaStream_t s) {
  return launch_pdl(k_gemv_decode<MT, J>, dim3(ctas), dim3(kThreads), 0, s, a);
}

}  // namespace

bool decode_supported(int64_t M, int64_t K) {
  Shape sh;
  return pick_shape(M, K, &sh);
}

cudaError_t launch_decode(const DecodeTarget* targets, int count, const int8_t* xq,
                          const float* x_scale, const uint16_t* x_bf16, int64_t M, int64_t K,
                          int8_t* xq_out, float* x_scale_out, cudaStream_t s) {
  Shape sh;
  if (count < 1 || count > kDecodeMaxTargets || !pick_shape(M, K, &sh))
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
  a.ksplit = sh.ksplit;
  a.slice_chunks = sh.slice_chunks;
  // One CTA per SM while the weights are small enough for neighbouring
  // launches to overlap; two per SM for large matrices.
  const int64_t bytes = rows * (K / 4);
  const int per_step = (kWarps / sh.ksplit) * kB;
  int64_t ctas = bytes > (int64_t)24 << 20 ? 296 : 148;
  const int64_t max_ctas = (rows + per_step - 1) / per_step;
  if (ctas > max_ctas) ctas = max_ctas;
  a.rows_per_cta = (int)((rows + ctas - 1) / ctas);
  ctas = (rows + a.rows_per_cta - 1) / a.rows_per_cta;
  const int c = (int)ctas;
  if (sh.mt == 1 && sh.j == 2) return launch_t<1, 2>(a, c, s);
  if (sh.mt == 1 && sh.j == 4) return launch_t<1, 4>(a, c, s);
  if (sh.mt == 2) return launch_t<2, 2>(a, c, s);
  return launch_t<4, 1>(a, c, s);
}

}  // namespace bitnet
