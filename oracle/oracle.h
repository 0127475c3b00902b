/*
 * BitLinear CPU oracle — TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously correct CPU statement of what the BitNet b1.58
 * BitLinear hot path computes.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library; the CUDA library
 * shares no code, header, table or helper with it.
 *
 * Sources (the web pages this method is described on):
 *  [P1] "Microsoft BitNet b1.58 ... 1-bit AI model" (communeify blog),
 *       section "Meet BitNet b1.58 2B4T": W1.58A8 (ternary weights, 8-bit
 *       integer activations), BitLinear layers, ReLU^2, subln, no bias terms.
 *  [P2] "How to run BitNet B1.58 (1-Bit LLM) locally" (onedollarvps), §2
 *       "Technical background", quantization process: divide the weights by
 *       their mean absolute value, then round and clip to {-1, 0, +1}.
 *  [P3] "BitNet.cpp deep dive" (dashen-tech), §2.3 "I2_S format" (2 bits per
 *       weight, 8 weights in 16 bits) and §3.1 "integer matrix multiplication"
 *       (Y = sum over +1 weights minus sum over -1 weights).
 *  [P4] "Microsoft BitNet: 100B models on CPU" (juejin), "CPU-friendly matrix
 *       multiplication": INT8 activations.
 *  [P5] "BitNet - 1-bit LLM inference framework" (news.hada.io), HN comment:
 *       the 2-bit storage can hold four values -1, 0, 1, 2.
 *
 * Every float operation below is one IEEE-754 binary32 (or binary64 where
 * marked) operation with round-to-nearest-even; the file is compiled with
 * -ffp-contract=off so no multiply-add is ever fused.
 *
 * Parity pins: every function here is pinned by tests/test_oracle.py against
 * worked examples, closed forms, exact rational arithmetic (Python
 * fractions), brute force on tiny inputs or library routines.  No function is
 * "parity unpinned".
 */
#ifndef BITLINEAR_ORACLE_H
#define BITLINEAR_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exact mean of |W| over n floats, rounded once to binary32 (nearest, ties to
 * even).  Returns NaN if any element is Inf or NaN, 0 for n == 0.
 * [P2] §2: the weights are divided by their "absolute mean". */
float oracle_absmean(const float* W, int64_t n);

/* q[n,k] = clamp(round_half_even(W[n,k] / g), -1, 1) with g = max(gamma,1e-5)
 * and an IEEE binary32 division.  [P2] §2 (divide, round, clip); [P1] the
 * ternary set {-1, 0, +1}.  Writes g to *w_scale. */
void oracle_ternarize(const float* W, int64_t N, int64_t K, float gamma,
                      int8_t* q, float* w_scale);

/* 2-bit packing, row-major [N, K/4] bytes.  code = q + 1 in {0,1,2}
 * ([P5] four representable values in 2 bits; [P3] §2.3 2 bits per weight).
 * Weight k of a row sits in 64-weight block b = k/64, position j = k%64:
 * byte b*16 + (j%16), bit shift 2*(j/16).  Requires K % 64 == 0. */
void oracle_pack(const int8_t* q, int64_t N, int64_t K, uint8_t* Wq);

/* Inverse of oracle_pack.  Returns 0, or -1 if a code 3 is found. */
int oracle_unpack(const uint8_t* Wq, int64_t N, int64_t K, int8_t* q);

/* Per-token absmax int8 quantisation of bf16 rows ([P1] "A8"; [P4] INT8
 * activations).  a = max|x|, a' = max(a, 1e-5), inv = 127/a',
 * q = clamp(round_half_even(x*inv), -128, 127), sx = a'/127.
 * x is given as raw bf16 bit patterns. */
void oracle_quantize_act_bf16(const uint16_t* x, int64_t M, int64_t K,
                              int8_t* q, float* sx);
/* Same rule on binary32 rows (used for the FFN hidden state). */
void oracle_quantize_act_f32(const float* x, int64_t M, int64_t K,
                             int8_t* q, float* sx);

/* acc[m,n] = sum_pos - sum_neg over k, with sum_pos the sum of qx[m,k] where
 * qw[n,k] = +1 and sum_neg where qw[n,k] = -1 ([P3] §3.1).  qw is [N,K]
 * ternary, qx is [M,K] int8.  Rows of the output are split over `threads`
 * std::threads (<= 1: the calling thread only); the result does not depend
 * on it. */
void oracle_linear_acc(const int8_t* qw, const int8_t* qx, int64_t M,
                       int64_t N, int64_t K, int32_t* acc, int threads);

/* y[m,n] = (float)acc[m,n] * (sx[m] * w_scale)  (two binary32 products). */
void oracle_rescale(const int32_t* acc, const float* sx, float w_scale,
                    int64_t M, int64_t N, float* y);

/* Full BitLinear from packed weights: unpack, sum_pos - sum_neg, rescale.
 * acc may be NULL.  Returns -1 on a bad code. */
int oracle_linear(const uint8_t* Wq, float w_scale, const int8_t* qx,
                  const float* sx, int64_t M, int64_t N, int64_t K, float* y,
                  int32_t* acc, int threads);

/* subln RMSNorm of bf16 rows ([P1] "subln"; the pages give no formula, so
 * this is the build's reading, order-free like the absmean):
 *   t_k = x_k * x_k            one binary32 product per element;
 *   ss  = sum_k t_k            the exact sum, rounded once to binary32
 *                              (NaN if a t_k is NaN, else +Inf if one is Inf);
 *   r   = 1 / sqrt(ss / H + eps)   four binary32 operations (division,
 *                              addition, correctly rounded square root,
 *                              division), in that order;
 *   n_k = (x_k * r) * g_k      binary32.
 * r_out (may be NULL) receives r per row. */
void oracle_rmsnorm_bf16(const uint16_t* x, const float* g, float eps,
                         int64_t M, int64_t H, float* n, float* r_out);

/* Nearest bf16 (ties to even) to each binary32 value: the bf16 output form of
 * a BitLinear result (the rescale "to fp32/bf16"; the pages fix no rounding,
 * the reading is round-to-nearest-even).  A value above the largest bf16
 * rounds to Inf; NaN stays NaN. */
void oracle_f32_to_bf16(const float* v, int64_t count, uint16_t* out);

/* h = (t * t) * u with t = max(v, 0): ReLU^2 of the gate times the up
 * projection ([P1] ReLU^2). */
void oracle_relu2_mul(const float* u, const float* v, int64_t count, float* h);

/* Fused BitNet FFN block ([P1]: subln, BitLinear, ReLU^2, no bias):
 *   RMSNorm(x) -> int8 quant -> up, gate BitLinear (H -> F) ->
 *   h = relu(gate)^2 * up -> int8 quant over F -> down BitLinear (F -> H).
 * Every debug pointer may be NULL: xq [M,H], sx [M], u, v, h [M,F],
 * hq [M,F], sh [M], acc_down [M,H].  Returns -1 on a bad code. */
int oracle_ffn(const uint16_t* x, const float* g, float eps,
               const uint8_t* Wup, float s_up, const uint8_t* Wgate,
               float s_gate, const uint8_t* Wdown, float s_down, int64_t M,
               int64_t H, int64_t F, float* y, int8_t* xq, float* sx,
               float* u, float* v, float* h, int8_t* hq, float* sh,
               int32_t* acc_down, int threads);

#ifdef __cplusplus
}
#endif
#endif
