/*
 * bitnet_b300.h — BitNet b1.58 BitLinear hot path for NVIDIA B300 (sm_103a).
 *
 * Ternary weights {-1, 0, +1} times int8 activations, int32 accumulation,
 * binary32 rescale, and the fused BitNet feed-forward block built on it.
 *
 * Sources (web pages describing the method):
 *  [P1] "Microsoft BitNet b1.58 ... 1-bit AI model" (communeify blog),
 *       "Meet BitNet b1.58 2B4T": W1.58A8, BitLinear, ReLU^2, subln, no bias.
 *  [P2] "How to run BitNet B1.58 (1-Bit LLM) locally" (onedollarvps), §2
 *       "Technical background": weights divided by their mean absolute value,
 *       rounded and clipped to {-1, 0, +1}.
 *  [P3] "BitNet.cpp deep dive" (dashen-tech), §2.3 "I2_S format" (2 bits per
 *       weight, 8 weights in 16 bits), §3.1 "integer matrix multiplication"
 *       (Y = sum_pos - sum_neg, no multiplications).
 *  [P4] "Microsoft BitNet: 100B models on CPU" (juejin), "CPU-friendly
 *       matrix multiplication": INT8 activations.
 *  [P5] "BitNet - 1-bit LLM inference framework" (news.hada.io), HN comment:
 *       2-bit storage holds four values.
 *
 * Conventions for every call:
 *  - Every array argument is a DEVICE pointer owned by the caller; the
 *    library never allocates or frees device memory and keeps no state
 *    across calls other than a per-device error word (bitnet_device_error).
 *  - Arrays are row-major.  W is [N = out features, K = in features].
 *  - bf16 arrays are passed as uint16_t bit patterns.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous on it, never synchronise, and may be captured in a CUDA
 *    graph.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns a status and launches nothing:
 *      BITNET_ERR_NULL       a required pointer is NULL;
 *      BITNET_ERR_SHAPE      a size is <= 0, K (or H, F) is not a multiple of
 *                            64, or a size exceeds the stated maximum;
 *      BITNET_ERR_ALIGN      a pointer is not 16-byte aligned;
 *      BITNET_ERR_WORKSPACE  ws_bytes is below the *_workspace() figure;
 *      BITNET_ERR_UNSUPPORTED the current device is not compute capability
 *                            10.3 (sm_103);
 *      BITNET_ERR_CUDA       a CUDA call or launch failed (code in
 *                            bitnet_last_cuda_error());
 *      BITNET_ERR_ALIAS      arrays of a decode chain overlap in a way the
 *                            chain does not allow (bitnet_decode_chain_build).
 *  - Inputs must be finite; see each call for what non-finite input gives.
 *  - No C++ exception crosses this interface.
 */
#ifndef BITNET_B300_H
#define BITNET_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bitnet_status {
  BITNET_OK = 0,
  BITNET_ERR_NULL = 1,
  BITNET_ERR_SHAPE = 2,
  BITNET_ERR_ALIGN = 3,
  BITNET_ERR_WORKSPACE = 4,
  BITNET_ERR_UNSUPPORTED = 5,
  BITNET_ERR_CUDA = 6,
  BITNET_ERR_ALIAS = 7
} bitnet_status;

/* Largest K, H or F accepted (int32 partial sums stay exact below it). */
#define BITNET_MAX_K 65536

/* Static text for a status code; never NULL. */
const char* bitnet_status_string(int status);

/* The cudaError_t of the last BITNET_ERR_CUDA returned on this host thread. */
int bitnet_last_cuda_error(void);

/* Interface version (bumped on any incompatible change). */
int bitnet_abi_version(void);

/* Reads and clears the current device's error word: 0, or a code set by a
 * kernel whose internal wait ran past its time limit (the kernel then
 * returns without finishing its output).  Synchronises `stream`.  Bits 0-7:
 * tensor-core kernel; bits 8-15: single decode launches; bits 16-23: decode
 * chains (bit 16: a chain input was not produced in time; 17, 18: the weight
 * ring; 19: the final wait for copies in flight). */
bitnet_status bitnet_device_error(int* code_out, void* stream);

/* For tests of the time-out path: the bound, in SM clock cycles, of every
 * wait inside the library's kernels other than the final wait for their own
 * copies in flight (which keeps its bound of about one second, so that no
 * kernel ever returns with a copy outstanding).  0 restores the default
 * (2e9 cycles, about one second).  Applies to launches made after the call,
 * on every device; not thread-safe against concurrent launches. */
void bitnet_set_wait_limit(long long cycles);

/* ------------------------------------------------------------------------
 * Weight quantisation ([P2] §2; [P3] §2.3; [P5]).
 *   gamma   = mean of |W| over all N*K entries, computed exactly and rounded
 *             once to binary32 (nearest, ties to even);
 *   w_scale = max(gamma, 1e-5);
 *   q       = clamp(round_half_even(W / w_scale), -1, 1), IEEE binary32
 *             division;
 *   Wq      = codes q + 1 in {0, 1, 2}, 2 bits each, [N, K/4] bytes: weight
 *             k of row n is in byte n*K/4 + (k/64)*16 + (k%16) at bit shift
 *             2*((k%64)/16).
 * W: [N, K] binary32.  Wq: [N*K/4] bytes.  w_scale: one float (device).
 * ws: scratch of bitnet_quantize_weights_workspace() bytes, no initial
 * contents required.  If any W entry is Inf or NaN, w_scale becomes NaN
 * and every code is 1 (q = 0).  Requires K % 64 == 0, N*K < 2^40. */
size_t bitnet_quantize_weights_workspace(int64_t N, int64_t K);
bitnet_status bitnet_quantize_weights(const float* W, int64_t N, int64_t K,
                                      uint8_t* Wq, float* w_scale, void* ws,
                                      size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * bitnet_quantize_weights without a workspace argument.  The pages have no
 * counterpart to this call: it exists for callers that cannot allocate
 * device memory, e.g. a plugin inside a framework that owns the whole device
 * memory pool, or a latency-critical path where cudaMalloc (which may
 * synchronise the device) is not allowed.  Results are identical to
 * bitnet_quantize_weights.
 * The scratch is a fixed array of 1,212,416 bytes inside the library, held by
 * every device that loads the library until the process exits; it covers
 * every N*K the call accepts (N*K < 2^40, K % 64 == 0; anything else gives
 * BITNET_ERR_SHAPE).  Nothing is allocated or freed.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The address is kept for the life of the process: after a
 * cudaDeviceReset (which unloads the library's device code, so the array
 * may move) do not call this entry again in that process.  Every call uses the same array: calls whose work overlaps on the
 * GPU (other streams, other host threads) race and must be serialised by the
 * caller.  Each call writes all the scratch it reads, so no state carries
 * over between calls. */
bitnet_status bitnet_quantize_weights_noalloc(const float* W, int64_t N, int64_t K,
                                              uint8_t* Wq, float* w_scale, void* stream);

/* ------------------------------------------------------------------------
 * Per-token absmax int8 activation quantisation ([P1] "A8"; [P4]).
 * For each row m of x [M, K] (bf16):
 *   a = max_k |x|, a' = max(a, 1e-5), inv = 127 / a' (binary32 division),
 *   xq = clamp(round_half_even(x * inv), -128, 127), x_scale[m] = a' / 127.
 * xq: [M, K] int8.  x_scale: [M] float.  K % 64 == 0, K <= BITNET_MAX_K. */
bitnet_status bitnet_quantize_act(const uint16_t* x, int64_t M, int64_t K,
                                  int8_t* xq, float* x_scale, void* stream);

/* ------------------------------------------------------------------------
 * BitLinear ([P3] §3.1; rescale: [P1] no bias).
 *   acc[m,n] = sum over k of q[n,k] * xq[m,k]  (= sum_pos - sum_neg, exact
 *              int32), q unpacked from Wq;
 *   y[m,n]   = (float)acc[m,n] * (x_scale[m] * w_scale[0]);
 *   y_bf16   = y rounded to the nearest bf16 (ties to even).
 * Wq [N, K/4] bytes, w_scale [1], xq [M, K], x_scale [M].  Outputs, each
 * optional but at least one of y / y_bf16 required: y [M, N] float,
 * y_bf16 [M, N] bf16 (the rescale "to fp32/bf16"; with y NULL the binary32
 * result is never stored), acc_out [M, N] int32 copy of acc.
 * ws: scratch of bitnet_linear_workspace(M, N, K) bytes (0 when none is
 * needed), no initial contents required.  M <= 4096*64 rows per call;
 * K % 64 == 0.  Paths, all giving the same bits: M <= 4 streams the packed
 * weights through the decode kernel (no workspace); 5 <= M < 12 runs a
 * CUDA-core kernel when the matrix has fewer than 16 Mi weights; larger M
 * or matrices run the tensor cores (M <= 256: the packed
 * weights are expanded on chip, and K is split over CTAs when the output
 * has few 128 x 256 tiles; M > 256: an expanded copy of the weights is made
 * in the workspace first).  sm_103a has no integer tensor-core product, so
 * the tensor cores multiply exact stand-ins: for K >= 128 and M <= 64 or
 * M > 256, e4m3 copies of the ternary weights and of the two digits of each
 * activation (x = 16 (x >> 4) + (x & 15)); otherwise bf16 copies.  Every
 * partial sum is an integer below 2^24, so the binary32 accumulators hold
 * acc exactly. */
size_t bitnet_linear_workspace(int64_t M, int64_t N, int64_t K);
bitnet_status bitnet_linear(const uint8_t* Wq, const float* w_scale,
                            const int8_t* xq, const float* x_scale, int64_t M,
                            int64_t N, int64_t K, float* y, uint16_t* y_bf16,
                            int32_t* acc_out, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * One-token BitLinear with a lookup-table inner product: the ablation of the
 * dp4a kernels against the table-lookup kernel family ([P3] §3.2: I2_S vs
 * TL1/TL2; [P4] T-MAC section: lookups instead of multiplications).  Same
 * result as bitnet_linear at M = 1, bit for bit:
 *   acc[n] = sum_k q[n,k] * xq[k],  y[n] = (float)acc[n] * (x_scale[0] * w_scale[0]).
 * variant 0: for each pair of activations that shares a nibble of the packed
 *   weights (two 2-bit codes), a 16-entry table of c0*x0 + c1*x1 is built in
 *   shared memory; each byte of weights costs two table reads.
 * variant 1: the masked-field dp4a inner product on the same kernel skeleton
 *   (the control of the ablation).
 * Wq [N, K/4] packed, w_scale [1], xq [K] int8, x_scale [1]; y [N] float
 * (required), acc_out [N] int32 (optional).  K % 64 == 0, 64 <= K <=
 * BITNET_LUT_MAX_K; 1 <= N < 2^31; variant 0 or 1 (else BITNET_ERR_SHAPE).
 * No workspace. */
#define BITNET_LUT_MAX_K 12288
bitnet_status bitnet_linear_lut(const uint8_t* Wq, const float* w_scale, const int8_t* xq,
                                const float* x_scale, int64_t N, int64_t K, float* y,
                                int32_t* acc_out, int variant, void* stream);

/* ------------------------------------------------------------------------
 * Decode BitLinear from bf16 activations ([P1] W1.58A8; [P3] §3.1).
 * For up to BITNET_MAX_TARGETS weight matrices that share the same input
 * (e.g. the Q, K, V, up and gate projections of one token), in one launch:
 *   xq, sx  = per-token int8 quantisation of x (the rule of
 *             bitnet_quantize_act, bit for bit);
 *   y_i     = BitLinear(Wq_i, w_scale_i; xq, sx)  (the rule of bitnet_linear).
 * x: [M, K] bf16, 1 <= M <= BITNET_DECODE_MAX_M.  targets[i]: Wq [N_i, K/4]
 * packed, w_scale [1]; outputs y [M, N_i] float and y_bf16 [M, N_i] bf16
 * (at least one of the two), acc_out optional [M, N_i] int32.
 * xq_out [M, K] and x_scale_out [M] are optional copies of xq and sx.
 * K % 64 == 0; K <= 65536 for M = 1, 32768 for M = 2, 16384 for M <= 4
 * (BITNET_ERR_SHAPE beyond); sum of N_i <= 2^30.  Needs no workspace.  The
 * kernel may start while the previous kernel on `stream` is finishing
 * (programmatic dependent launch) and waits for it before reading x or
 * writing any output.
 * flags: 0, or BITNET_WEIGHTS_STATIC to promise that no work still in flight
 * on `stream` writes any Wq_i or w_scale_i (true for model weights quantised
 * ahead of time); the kernel then starts streaming the weights before the
 * previous kernel has finished.  Any other bit gives BITNET_ERR_SHAPE. */
#define BITNET_DECODE_MAX_M 4
#define BITNET_MAX_TARGETS 8
#define BITNET_WEIGHTS_STATIC 1u
typedef struct bitnet_linear_target {
  const uint8_t* Wq;
  const float* w_scale;
  int64_t N;
  float* y;
  int32_t* acc_out;
  uint16_t* y_bf16;
} bitnet_linear_target;

bitnet_status bitnet_linear_bf16(const uint16_t* x, int64_t M, int64_t K,
                                 const bitnet_linear_target* targets, int count,
                                 int8_t* xq_out, float* x_scale_out, unsigned flags,
                                 void* stream);

/* ------------------------------------------------------------------------
 * A decode chain: the BitLinear phases of a decoder step (e.g. QKV, O,
 * up+gate, down of every layer) run by one persistent kernel, one CTA per SM
 * ([P1] BitLinear, subln, ReLU^2; [P5] HN comment: memory bandwidth is the
 * bottleneck, so the weights of later phases stream in while earlier phases
 * compute).  Phase p:
 *   input   = x [M, K] bf16, or x_f32 [M, K] binary32 (exactly one given);
 *   norm    = optional subln RMSNorm of a bf16 input with gain norm_gain [K]
 *             and norm_eps (the rule of bitnet_ffn's normalisation);
 *   xq, sx  = per-token int8 quantisation of the (normalised) input (the
 *             rule of bitnet_quantize_act; for a binary32 input the same rule
 *             on its values);
 *   targets as in bitnet_linear_bf16 (outputs y, y_bf16, acc_out);
 *   flags & BITNET_PHASE_GATED: exactly two targets of equal N, up and gate;
 *             h = (t * t) * u with t = max(v, 0), u and v the two BitLinear
 *             results (the rule of bitnet_ffn), written to h [M, N]; the
 *             targets' own outputs are then optional.
 *   xq_out [M, K], x_scale_out [M]: optional copies of xq and sx.
 * Links: a phase input that IS an output of an earlier phase (x equal to a
 * target's y_bf16, or x_f32 equal to a target's y or a gated phase's h, with
 * N == K) is read as that phase produces it: each value travels with a tag of
 * the run and phase through the chain's table, and a CTA waits only for the
 * values it reads.  There is no other ordering between phases: every other
 * array the chain reads (x, x_f32, norm_gain, Wq, w_scale) must not overlap
 * any array the chain writes, and the arrays it writes must not overlap one
 * another (BITNET_ERR_ALIAS otherwise).  A CTA that owns no rows of a phase
 * skips it.  The weights stream in ahead, across phases.
 * table: device memory of bitnet_decode_chain_bytes(phases, nphases, M)
 * bytes (computed for the current device's SM count), 256-byte aligned,
 * owned by the caller; _build fills it
 * (synchronously: call it outside stream capture; it returns after the
 * copy) and clears it.  `chain` (host) receives what _run needs.  Runs of one
 * table must not overlap on the GPU.  All CTAs must be resident at once
 * (cooperative launch); _run returns BITNET_ERR_CUDA if the launch is
 * refused.  After a run that reported a device error (bitnet_device_error),
 * build the chain again before the next run.  At most 16384 phases. */
#define BITNET_PHASE_GATED 1u
typedef struct bitnet_decode_phase {
  const uint16_t* x;
  int64_t K;
  const bitnet_linear_target* targets;
  int count;
  unsigned flags;
  const float* x_f32;
  const float* norm_gain;
  float norm_eps;
  float* h;
  int8_t* xq_out;
  float* x_scale_out;
} bitnet_decode_phase;

typedef struct bitnet_decode_chain {
  void* table;
  int64_t M;
  int nphases;
  int cfg[12]; /* launch configuration, filled by bitnet_decode_chain_build */
} bitnet_decode_chain;

/* 0 if the description is invalid (the same checks as _build). */
size_t bitnet_decode_chain_bytes(const bitnet_decode_phase* phases, int nphases, int64_t M);
bitnet_status bitnet_decode_chain_build(const bitnet_decode_phase* phases, int nphases,
                                        int64_t M, void* table, size_t table_bytes,
                                        bitnet_decode_chain* chain);
bitnet_status bitnet_decode_chain_run(const bitnet_decode_chain* chain, void* stream);

/* ------------------------------------------------------------------------
 * Fused BitNet feed-forward block ([P1] subln, ReLU^2, no bias):
 *   ss  = sum over k of x_k * x_k: each square one binary32 product, the
 *         sum exact (order-free) and rounded once to binary32;
 *   r   = 1 / sqrt(ss / H + eps), four binary32 operations in that order
 *         (division, addition, correctly rounded square root, division);
 *   nrm = (x * r) * g;                          binary32, per element
 *   xq, sx = per-token int8 quantisation of nrm (rule of bitnet_quantize_act)
 *   u   = BitLinear(Wup, s_up; xq, sx)          [M, F]
 *   v   = BitLinear(Wgate, s_gate; xq, sx)      [M, F]
 *   h   = (t * t) * u, t = max(v, 0)            binary32
 *   hq, sh = per-token int8 quantisation of h over F
 *   y   = BitLinear(Wdown, s_down; hq, sh)      [M, H]
 * x [M, H] bf16, g [H] float, Wup / Wgate [F, H/4], Wdown [H, F/4] packed,
 * s_* one float each, y [M, H] float.  H % 64 == 0, F % 64 == 0.
 * dbg: NULL, or a struct whose non-NULL members receive the named
 * intermediate (xq [M,H], sx [M], u, v, h [M,F], hq [M,F], sh [M],
 * acc_down [M,H]).  ws: bitnet_ffn_workspace(M, H, F) bytes, no initial
 * contents required. */
typedef struct bitnet_ffn_debug {
  int8_t* xq;
  float* sx;
  float* u;
  float* v;
  float* h;
  int8_t* hq;
  float* sh;
  int32_t* acc_down;
} bitnet_ffn_debug;

size_t bitnet_ffn_workspace(int64_t M, int64_t H, int64_t F);
bitnet_status bitnet_ffn(const uint16_t* x, const float* g, float eps,
                         const uint8_t* Wup, const float* s_up,
                         const uint8_t* Wgate, const float* s_gate,
                         const uint8_t* Wdown, const float* s_down, int64_t M,
                         int64_t H, int64_t F, float* y,
                         const bitnet_ffn_debug* dbg, void* ws,
                         size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif
