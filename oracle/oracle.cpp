// BitLinear CPU oracle — TEST INFRASTRUCTURE (see oracle.h for the sources
// and the rules).  Plain loops, no intrinsics, no blocking beyond what the
// definitions state.  Build: g++ -O2 -ffp-contract=off -std=c++17 -fPIC.
#include "oracle.h"

#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

uint32_t float_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return u;
}

// ---------------------------------------------------------------------------
// Exact sum of |W| as an unsigned integer counted in units of 2^-149 (the
// smallest binary32 subnormal), little-endian 64-bit limbs.  Every finite
// binary32 magnitude is an integer multiple of 2^-149 below 2^277, so with
// six limbs (384 bits) the sum of up to 2^100 terms is exact.
constexpr int kLimbs = 6;
using Big = std::vector<uint64_t>;

void big_add_shifted(Big& a, uint64_t v, int shift) {
  int i = shift / 64, o = shift % 64;
  unsigned __int128 x = (unsigned __int128)v << o;
  uint64_t part[2] = {(uint64_t)x, (uint64_t)(x >> 64)};
  uint64_t carry = 0;
  for (int j = i; j < kLimbs; ++j) {
    uint64_t add = (j - i < 2) ? part[j - i] : 0;
    unsigned __int128 s = (unsigned __int128)a[j] + add + carry;
    a[j] = (uint64_t)s;
    carry = (uint64_t)(s >> 64);
  }
}

int big_bitlen(const Big& a) {
  for (int j = (int)a.size() - 1; j >= 0; --j)
    if (a[j]) return j * 64 + 64 - __builtin_clzll(a[j]);
  return 0;
}

int big_bit(const Big& a, int pos) {
  if (pos < 0 || pos >= (int)a.size() * 64) return 0;
  return (int)((a[pos / 64] >> (pos % 64)) & 1u);
}

Big big_shl(const Big& a, int t) {
  Big r(a.size() + (t + 63) / 64 + 1, 0);
  for (int pos = 0; pos < (int)a.size() * 64; ++pos)
    if (big_bit(a, pos)) r[(pos + t) / 64] |= (uint64_t)1 << ((pos + t) % 64);
  return r;
}

// Long division of a by d (d > 0): returns the quotient, *rem the remainder.
Big big_divmod(const Big& a, uint64_t d, uint64_t* rem) {
  Big q(a.size(), 0);
  unsigned __int128 r = 0;
  for (int j = (int)a.size() - 1; j >= 0; --j) {
    unsigned __int128 cur = (r << 64) | a[j];
    q[j] = (uint64_t)(cur / d);
    r = cur % d;
  }
  *rem = (uint64_t)r;
  return q;
}

// Nearest binary32 (ties to even) to S * 2^-149 / d, S an exact integer.
float round_quotient_to_f32(const Big& S, uint64_t d) {
  int bl = big_bitlen(S);
  if (bl == 0) return 0.0f;
  int dl = 64 - __builtin_clzll(d);
  // Scale the dividend by 2^t so the quotient carries >= 27 bits.
  int t = 28 + dl - bl;
  if (t < 0) t = 0;
  uint64_t rem = 0;
  Big Q = big_divmod(big_shl(S, t), d, &rem);
  int qb = big_bitlen(Q);
  // Bit j of Q weighs 2^(j - 149 - t).  Keep 24 bits, but never a bit below
  // 2^-149 (binary32 subnormals).
  int drop = qb - 24;
  if (drop < t) drop = t;
  uint64_t mant = 0;
  for (int j = 0; j < 25; ++j)
    mant |= (uint64_t)big_bit(Q, drop + j) << j;
  int round_bit = big_bit(Q, drop - 1);
  int sticky = rem != 0;
  for (int j = 0; j < drop - 1 && !sticky; ++j) sticky = big_bit(Q, j);
  if (round_bit && (sticky || (mant & 1u))) mant += 1;
  // mant <= 2^24 and mant * 2^(drop-149-t) is a binary32 value, so both
  // conversions below are exact.
  return (float)std::ldexp((double)mant, drop - 149 - t);
}

// round(v) with ties to even, clipped to [lo, hi]; NaN gives 0.
int round_clip(float v, int lo, int hi) {
  if (v != v) return 0;
  float r = std::nearbyint(v);  // default rounding mode: nearest-even
  if (r < (float)lo) return lo;
  if (r > (float)hi) return hi;
  return (int)r;
}

void quantize_row(const float* xf, int64_t K, int8_t* q, float* sx) {
  float a = 0.0f;
  for (int64_t k = 0; k < K; ++k) {
    float m = std::fabs(xf[k]);
    if (m > a) a = m;
  }
  float ap = a > 1e-5f ? a : 1e-5f;
  float inv = 127.0f / ap;
  for (int64_t k = 0; k < K; ++k) q[k] = (int8_t)round_clip(xf[k] * inv, -128, 127);
  *sx = ap / 127.0f;
}

}  // namespace

extern "C" {

float oracle_absmean(const float* W, int64_t n) {
  if (n <= 0) return 0.0f;
  Big S(kLimbs, 0);
  for (int64_t i = 0; i < n; ++i) {
    uint32_t u = float_bits(W[i]) & 0x7fffffffu;
    uint32_t e = u >> 23, m = u & 0x7fffffu;
    if (e == 255) return std::nanf("");
    if (e == 0)
      big_add_shifted(S, m, 0);  // subnormal: m * 2^-149
    else
      big_add_shifted(S, m | 0x800000u, (int)e - 1);  // (1.m) * 2^(e-127)
  }
  return round_quotient_to_f32(S, (uint64_t)n);
}

void oracle_ternarize(const float* W, int64_t N, int64_t K, float gamma,
                      int8_t* q, float* w_scale) {
  float g = gamma;
  if (g == g && g < 1e-5f) g = 1e-5f;
  *w_scale = g;
  for (int64_t i = 0; i < N * K; ++i) q[i] = (int8_t)round_clip(W[i] / g, -1, 1);
}

void oracle_pack(const int8_t* q, int64_t N, int64_t K, uint8_t* Wq) {
  std::memset(Wq, 0, (size_t)(N * K / 4));
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      int64_t b = k / 64, j = k % 64;
      uint8_t code = (uint8_t)(q[n * K + k] + 1);
      Wq[n * (K / 4) + b * 16 + (j % 16)] |= (uint8_t)(code << (2 * (j / 16)));
    }
}

int oracle_unpack(const uint8_t* Wq, int64_t N, int64_t K, int8_t* q) {
  int bad = 0;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      int64_t b = k / 64, j = k % 64;
      int code = (Wq[n * (K / 4) + b * 16 + (j % 16)] >> (2 * (j / 16))) & 3;
      if (code == 3) bad = 1;
      q[n * K + k] = (int8_t)(code - 1);
    }
  return bad ? -1 : 0;
}

void oracle_quantize_act_bf16(const uint16_t* x, int64_t M, int64_t K,
                              int8_t* q, float* sx) {
  std::vector<float> row((size_t)K);
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t k = 0; k < K; ++k) row[k] = bf16_to_float(x[m * K + k]);
    quantize_row(row.data(), K, q + m * K, sx + m);
  }
}

void oracle_quantize_act_f32(const float* x, int64_t M, int64_t K, int8_t* q,
                             float* sx) {
  for (int64_t m = 0; m < M; ++m) quantize_row(x + m * K, K, q + m * K, sx + m);
}

void oracle_linear_acc(const int8_t* qw, const int8_t* qx, int64_t M,
                       int64_t N, int64_t K, int32_t* acc, int threads) {
  auto rows = [&](int64_t n0, int64_t n1) {
    for (int64_t n = n0; n < n1; ++n)
      for (int64_t m = 0; m < M; ++m) {
        int64_t sum_pos = 0, sum_neg = 0;
        for (int64_t k = 0; k < K; ++k) {
          int8_t w = qw[n * K + k];
          if (w == 1) sum_pos += qx[m * K + k];
          else if (w == -1) sum_neg += qx[m * K + k];
        }
        acc[m * N + n] = (int32_t)(sum_pos - sum_neg);
      }
  };
  if (threads <= 1 || N < 2) {
    rows(0, N);
    return;
  }
  std::vector<std::thread> pool;
  int64_t per = (N + threads - 1) / threads;
  for (int64_t n0 = 0; n0 < N; n0 += per)
    pool.emplace_back(rows, n0, n0 + per < N ? n0 + per : N);
  for (auto& th : pool) th.join();
}

void oracle_rescale(const int32_t* acc, const float* sx, float w_scale,
                    int64_t M, int64_t N, float* y) {
  for (int64_t m = 0; m < M; ++m) {
    float c = sx[m] * w_scale;
    for (int64_t n = 0; n < N; ++n) y[m * N + n] = (float)acc[m * N + n] * c;
  }
}

int oracle_linear(const uint8_t* Wq, float w_scale, const int8_t* qx,
                  const float* sx, int64_t M, int64_t N, int64_t K, float* y,
                  int32_t* acc, int threads) {
  std::vector<int8_t> qw((size_t)(N * K));
  if (oracle_unpack(Wq, N, K, qw.data()) != 0) return -1;
  std::vector<int32_t> a((size_t)(M * N));
  oracle_linear_acc(qw.data(), qx, M, N, K, a.data(), threads);
  oracle_rescale(a.data(), sx, w_scale, M, N, y);
  if (acc) std::memcpy(acc, a.data(), a.size() * sizeof(int32_t));
  return 0;
}

void oracle_rmsnorm_bf16(const uint16_t* x, const float* g, float eps,
                         int64_t M, int64_t H, float* n, float* r_out) {
  for (int64_t m = 0; m < M; ++m) {
    // ss: the exact sum of the binary32 squares, rounded once.
    Big S(kLimbs, 0);
    bool any_nan = false, any_inf = false;
    for (int64_t k = 0; k < H; ++k) {
      float xf = bf16_to_float(x[m * H + k]);
      float t = xf * xf;  // one binary32 product
      uint32_t u = float_bits(t);
      uint32_t e = (u >> 23) & 0xffu, f = u & 0x7fffffu;
      if (e == 255) {
        if (f) any_nan = true;
        else any_inf = true;
      } else if (e == 0) {
        big_add_shifted(S, f, 0);
      } else {
        big_add_shifted(S, f | 0x800000u, (int)e - 1);
      }
    }
    float ss = any_nan ? std::nanf("") : any_inf ? INFINITY : round_quotient_to_f32(S, 1);
    float q = ss / (float)H;
    float t = q + eps;
    float s = std::sqrt(t);  // binary32 square root, correctly rounded
    float r = 1.0f / s;
    if (r_out) r_out[m] = r;
    for (int64_t k = 0; k < H; ++k) {
      float xf = bf16_to_float(x[m * H + k]);
      n[m * H + k] = (xf * r) * g[k];
    }
  }
}

void oracle_f32_to_bf16(const float* v, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) {
    uint32_t u = float_bits(v[i]);
    if ((u & 0x7fffffffu) > 0x7f800000u) {
      out[i] = (uint16_t)((u >> 16) | 0x40u);  // NaN stays NaN (quiet)
      continue;
    }
    // Keep the top 16 bits; round on the 16 dropped bits, ties to even.
    uint32_t lower = u & 0xffffu, upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;
    out[i] = (uint16_t)upper;
  }
}

void oracle_relu2_mul(const float* u, const float* v, int64_t count, float* h) {
  for (int64_t i = 0; i < count; ++i) {
    float t = v[i] > 0.0f ? v[i] : 0.0f;
    h[i] = (t * t) * u[i];
  }
}

int oracle_ffn(const uint16_t* x, const float* g, float eps,
               const uint8_t* Wup, float s_up, const uint8_t* Wgate,
               float s_gate, const uint8_t* Wdown, float s_down, int64_t M,
               int64_t H, int64_t F, float* y, int8_t* xq_out, float* sx_out,
               float* u_out, float* v_out, float* h_out, int8_t* hq_out,
               float* sh_out, int32_t* acc_down_out, int threads) {
  std::vector<float> nrm((size_t)(M * H)), u((size_t)(M * F)), v((size_t)(M * F)),
      h((size_t)(M * F)), sx((size_t)M), sh((size_t)M);
  std::vector<int8_t> xq((size_t)(M * H)), hq((size_t)(M * F));
  std::vector<int32_t> acc_d((size_t)(M * H));

  oracle_rmsnorm_bf16(x, g, eps, M, H, nrm.data(), nullptr);
  oracle_quantize_act_f32(nrm.data(), M, H, xq.data(), sx.data());
  if (oracle_linear(Wup, s_up, xq.data(), sx.data(), M, F, H, u.data(), nullptr, threads))
    return -1;
  if (oracle_linear(Wgate, s_gate, xq.data(), sx.data(), M, F, H, v.data(), nullptr, threads))
    return -1;
  oracle_relu2_mul(u.data(), v.data(), M * F, h.data());
  oracle_quantize_act_f32(h.data(), M, F, hq.data(), sh.data());
  if (oracle_linear(Wdown, s_down, hq.data(), sh.data(), M, H, F, y, acc_d.data(), threads))
    return -1;

  if (xq_out) std::memcpy(xq_out, xq.data(), xq.size());
  if (sx_out) std::memcpy(sx_out, sx.data(), sx.size() * sizeof(float));
  if (u_out) std::memcpy(u_out, u.data(), u.size() * sizeof(float));
  if (v_out) std::memcpy(v_out, v.data(), v.size() * sizeof(float));
  if (h_out) std::memcpy(h_out, h.data(), h.size() * sizeof(float));
  if (hq_out) std::memcpy(hq_out, hq.data(), hq.size());
  if (sh_out) std::memcpy(sh_out, sh.data(), sh.size() * sizeof(float));
  if (acc_down_out) std::memcpy(acc_down_out, acc_d.data(), acc_d.size() * sizeof(int32_t));
  return 0;
}

}  // extern "C"
