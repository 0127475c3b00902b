"""GPU parity: every C-ABI call against the CPU oracle on the same seeded
inputs.  Integer outputs (packed bytes, int8 codes, int32 accumulators) and
the scales must match bit for bit; fp32 outputs must be within a relative
1e-5 (they are expected to match bit for bit as well).  Sizes span several
tiles and ragged tails; the full workload sizes are checked on sampled rows
that the oracle computes one by one."""
import json
import os
import time

import numpy as np
import pytest
import torch

import oracle
import bitlinear_bitnet_linear_03_b300 as bn
from bitlinear_bitnet_linear_03_b300 import synth
from gpu_util import assert_bits_equal, assert_f32_close, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


# ---------------------------------------------------------------- weights
def gpu_quantize_weights(W: np.ndarray):
    Wq, ws = bn.bitnet_quantize_weights(dev(W))
    return host(Wq), host(ws)[0]


def check_weights(W: np.ndarray, what: str):
    Wq_g, s_g = gpu_quantize_weights(W)
    Wq_o, s_o, _ = oracle.quantize_weights(W)
    assert_bits_equal(np.array([s_g], np.float32), np.array([s_o], np.float32), what + " w_scale")
    assert_bits_equal(Wq_g, Wq_o, what + " Wq")


@pytest.mark.parametrize("N,K", [(1, 64), (3, 192), (17, 640), (33, 128), (640, 2560),
                                 (2560, 2560), (6912, 2560), (2560, 6912)])
def test_quantize_weights_seeded(N, K):
    check_weights(synth.weights_f32(N, K, seed=N + K), f"W[{N}x{K}]")


def test_quantize_weights_worked_examples():
    # The 2x4 tie example, laid into the first columns of a 2x64 matrix whose
    # other entries are chosen so that the mean stays 2: |W| sums to 256.
    W = np.zeros((2, 64), np.float32)
    W[:, :4] = np.array(GOLD["weights_ties"]["W"], np.float32)
    W[:, 4:] = np.float32(2.0)          # sum|W| = 16 + 120*2 = 256 = 2 * 128
    Wq_g, s_g = gpu_quantize_weights(W)
    assert s_g == np.float32(2.0)
    # the worked example's codes, the rest +1, packed by the oracle
    q_want = np.ones((2, 64), np.int8)
    q_want[:, :4] = np.array(GOLD["weights_ties"]["q"], np.int8)
    assert_bits_equal(Wq_g, oracle.pack(q_want), "tie codes")
    check_weights(W, "ties")


def test_quantize_weights_special_cases():
    check_weights(np.zeros((3, 64), np.float32), "zeros")
    rng = np.random.default_rng(0)
    s = rng.choice([-1.0, 1.0], size=(32, 128)).astype(np.float32)
    check_weights(s * np.float32(0.25), "sign pattern")
    # mixed magnitudes: subnormals to 1e38, so any float sum order would round
    W = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-140, 120, (64, 256)))).astype(
        np.float32)
    check_weights(W, "mixed exponents")
    W = np.full((7, 64), 1e-44, np.float32)
    check_weights(W, "subnormal only")
    # exact half-ties of the scale in every position
    W = np.ones((16, 64), np.float32)
    W[::2, ::3] = 0.5
    W[1::2, ::5] = -1.5
    check_weights(W, "half ties")


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_quantize_weights_nonfinite(bad):
    W = synth.weights_f32(5, 128, seed=3)
    W[2, 77] = bad
    Wq_g, s_g = gpu_quantize_weights(W)
    assert np.isnan(s_g)
    assert (Wq_g == 0x55).all()


def test_quantize_weights_full_100b_shape_sampled():
    N, K = 28672, 8192
    W = synth.weights_f32(N, K, seed=0)
    Wq_g, s_g = gpu_quantize_weights(W)
    gamma = oracle.absmean(W)
    rows = np.random.default_rng(0).choice(N, 64, replace=False)
    rows[:2] = [0, N - 1]
    q, s_o = oracle.ternarize(W[rows], gamma)
    assert_bits_equal(np.array([s_g], np.float32), np.array([s_o], np.float32), "w_scale")
    assert_bits_equal(Wq_g[rows], oracle.pack(q), "sampled Wq rows")


# ---------------------------------------------------------------- activations
def check_act(x_bits: np.ndarray, what: str):
    xq, sx = bn.bitnet_quantize_act(dev_bf16(x_bits))
    q_o, s_o = oracle.quantize_act_bf16(x_bits)
    assert_bits_equal(host(sx), s_o, what + " x_scale")
    assert_bits_equal(host(xq), q_o, what + " xq")


@pytest.mark.parametrize("M,K,frac", [(1, 64, 0), (3, 2560, 0), (1, 2560, 0.01), (64, 6912, 0.01),
                                      (5, 28672, 0.01), (4096, 2560, 0), (4096, 6912, 0),
                                      (2, 65536, 0.01)])
def test_quantize_act_seeded(M, K, frac):
    check_act(synth.tokens_bf16(M, K, seed=M + K, outlier_frac=frac), f"x[{M}x{K}]")


def test_quantize_act_worked_example_and_special_rows():
    x = np.zeros((4, 64), np.float32)
    x[0, :4] = GOLD["act_ties"]["x"]
    x[2, :] = 1.0
    x[3, 5] = -3.0
    bits = synth.f32_to_bf16_bits(x)
    xq, sx = bn.bitnet_quantize_act(dev_bf16(bits))
    q = host(xq)
    assert q[0, :4].tolist() == GOLD["act_ties"]["q"] and host(sx)[0] == np.float32(1.0)
    assert (q[1] == 0).all()                          # all-zero token
    assert (q[2] == 127).all() and (q[3, 5] == -127)
    check_act(bits, "special rows")


def test_quantize_act_nonfinite():
    bits = synth.tokens_bf16(3, 128, seed=5)
    bits[0, 3] = 0x7f80  # +inf
    bits[1, 9] = 0x7fc0  # nan
    check_act(bits, "non-finite")


# ---------------------------------------------------------------- linear
def linear_inputs(M, N, K, seed, frac=0.0):
    W = synth.weights_f32(N, K, seed=seed)
    x = synth.tokens_bf16(M, K, seed=seed + 1000, outlier_frac=frac)
    Wq, ws, _ = oracle.quantize_weights(W)
    qx, sx = oracle.quantize_act_bf16(x)
    return Wq, ws, qx, sx


def gpu_linear(Wq, ws, qx, sx, K):
    M, N = qx.shape[0], Wq.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = bn.bitnet_linear(dev(Wq), dev(np.array([ws], np.float32)), dev(qx), dev(sx), K=K,
                         acc_out=acc)
    return host(y), host(acc)


LINEAR_SHAPES = [(1, 1, 64), (1, 7, 64), (2, 65, 192), (3, 640, 2560), (1, 2560, 2560),
                 (5, 2560, 2560), (8, 6912, 2560), (1, 2560, 6912), (17, 2560, 6912),
                 # 5 <= M < 12: CUDA cores below 16 Mi weights, tensor cores above
                 (7, 1000, 1088), (11, 640, 2560), (5, 8192, 2048), (9, 4100, 4096),
                 (12, 100, 640),
                 (4, 100, 8192), (63, 96, 2560), (64, 33, 128), (65, 130, 640), (129, 64, 320),
                 (1, 31, 65536),
                 # tensor-core path with K split over several CTAs (few output tiles)
                 (20, 300, 4096), (64, 33, 8192), (200, 777, 2048), (16, 2560, 4096),
                 # e4m3 digit form (M <= 64, K >= 128): K a half stage past a
                 # multiple of 128, ragged N, split K, and K = 64 (bf16 form)
                 (24, 257, 320), (33, 2048, 192), (40, 1000, 1088), (48, 600, 6912),
                 (16, 8, 64), (64, 4000, 2560),
                 # prefill digit form (M > 256): ragged K and N, BN = 128, K = 64
                 # (bf16 form)
                 (300, 333, 192), (260, 1000, 1088), (257, 100, 640), (300, 64, 64)]


@pytest.mark.parametrize("M,N,K", LINEAR_SHAPES)
def test_linear_seeded(M, N, K):
    Wq, ws, qx, sx = linear_inputs(M, N, K, seed=M * 7 + N, frac=0.01)
    y_g, acc_g = gpu_linear(Wq, ws, qx, sx, K)
    y_o, acc_o = oracle.linear(Wq, ws, qx, sx, K)
    assert_bits_equal(acc_g, acc_o, "acc")
    assert_f32_close(y_g, y_o, "y")
    assert_bits_equal(y_g, y_o, "y bits")


def test_linear_worked_example():
    g = GOLD["linear"]
    q = np.zeros((2, 64), np.int8)
    q[:, :4] = np.array(g["qw"], np.int8)
    qx = np.zeros((1, 64), np.int8)
    qx[0, :4] = g["qx"]
    y, acc = gpu_linear(oracle.pack(q), np.float32(g["w_scale"]), qx,
                        np.array([g["sx"]], np.float32), 64)
    assert acc.ravel().tolist() == g["acc"]
    assert y.ravel().tolist() == g["y"]


def test_linear_extreme_accumulators():
    K = 65536
    q = np.ones((2, K), np.int8)
    q[1] = -1
    qx = np.full((1, K), -128, np.int8)
    y, acc = gpu_linear(oracle.pack(q), np.float32(1.0), qx, np.array([1.0], np.float32), K)
    assert acc.ravel().tolist() == [-128 * K, 128 * K]


@pytest.mark.parametrize("M", [16, 257])
def test_linear_digit_form_extremes(M):
    """Tokens at the ends of the int8 range (digits hi = -8, lo = 0 and hi = 7,
    lo = 15) against all +1 / all -1 / alternating weights at K = 65536, and a
    row whose sum first grows to 2^22 and then moves by single units: every
    sum must stay exact in the binary32 accumulators of the e4m3 MMAs (M = 16:
    the small-M digit form; M = 257: the prefill digit form, whose hi digits
    are scaled by 16, so that its sums reach 2^23)."""
    K = 65536
    q = np.ones((3, K), np.int8)
    q[1] = -1
    q[2, 1::2] = -1
    qx = np.random.default_rng(3).integers(-128, 128, (M, K)).astype(np.int8)
    qx[0] = -128
    qx[1] = 127
    qx[2, : K // 2] = 127
    qx[2, K // 2:] = 1
    qx[3, : K // 2] = -128
    qx[3, K // 2:] = np.where(np.arange(K // 2) % 3 == 0, 1, 0)
    sx = np.ones(M, np.float32)
    y, acc = gpu_linear(oracle.pack(q), np.float32(1.0), qx, sx, K)
    y_o, acc_o = oracle.linear(oracle.pack(q), np.float32(1.0), qx, sx, K)
    assert acc[0].tolist() == [-128 * K, 128 * K, 0]
    assert acc[1].tolist() == [127 * K, -127 * K, 0]
    assert_bits_equal(acc, acc_o, "acc")
    assert_bits_equal(y, y_o, "y bits")


@pytest.mark.parametrize("M", [1, 4, 16, 64])
@pytest.mark.parametrize("N,K", [(28672, 8192), (8192, 28672)])
def test_linear_100b_shapes_sampled(M, N, K):
    W = synth.weights_f32(N, K, seed=11)
    x = synth.tokens_bf16(M, K, seed=12, outlier_frac=0.01)
    Wq_d, ws_d = bn.bitnet_quantize_weights(dev(W))
    xq_d, sx_d = bn.bitnet_quantize_act(dev_bf16(x))
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = host(bn.bitnet_linear(Wq_d, ws_d, xq_d, sx_d, acc_out=acc))
    acc = host(acc)
    gamma = oracle.absmean(W)
    rows = np.random.default_rng(M).choice(N, 48, replace=False)
    rows[:2] = [0, N - 1]
    q, ws = oracle.ternarize(W[rows], gamma)
    qx, sx = oracle.quantize_act_bf16(x)
    y_o, acc_o = oracle.linear(oracle.pack(q), ws, qx, sx, K)
    assert_bits_equal(acc[:, rows], acc_o, "acc sampled")
    assert_f32_close(y[:, rows], y_o, "y sampled")
    assert_bits_equal(y[:, rows], y_o, "y sampled bits")


@pytest.mark.parametrize("N,K", [(6912, 2560), (2560, 6912), (14336, 4096), (4096, 14336)])
def test_linear_prefill_shapes_sampled(N, K):
    """Prefill at seq 4096 on the 2B-class FFN shapes (hidden 2560, FFN 6912)
    and the 8B-class ones (hidden 4096, FFN 14336)."""
    M = 4096
    W = synth.weights_f32(N, K, seed=21)
    x = synth.tokens_bf16(M, K, seed=22)
    Wq, ws, _ = oracle.quantize_weights(W)
    qx, sx = oracle.quantize_act_bf16(x)
    y_g, acc_g = gpu_linear(Wq, ws, qx, sx, K)
    rows = np.random.default_rng(1).choice(N, 24, replace=False)
    rows[:2] = [0, N - 1]
    y_o, acc_o = oracle.linear(Wq[rows], ws, qx, sx, K, threads=oracle.default_threads())
    assert_bits_equal(acc_g[:, rows], acc_o, "acc sampled")
    assert_bits_equal(y_g[:, rows], y_o, "y sampled bits")
    # every output row: the properties that hold at any size
    assert np.isfinite(y_g).all()
    assert (np.abs(acc_g) <= 127 * K).all()


def test_quantize_then_linear_chain():
    M, N, K = 3, 2560, 2560
    W = synth.weights_f32(N, K, seed=31)
    x = synth.tokens_bf16(M, K, seed=32, outlier_frac=0.01)
    Wq_d, ws_d = bn.bitnet_quantize_weights(dev(W))
    xq_d, sx_d = bn.bitnet_quantize_act(dev_bf16(x))
    y = host(bn.bitnet_linear(Wq_d, ws_d, xq_d, sx_d))
    Wq, ws, _ = oracle.quantize_weights(W)
    qx, sx = oracle.quantize_act_bf16(x)
    y_o, _ = oracle.linear(Wq, ws, qx, sx, K)
    assert_bits_equal(y, y_o, "chain y")


# ---------------------------------------------------------------- grouped decode from bf16
def check_linear_bf16(M, K, Ns, seed, frac=0.01, weights_static=False):
    x = synth.tokens_bf16(M, K, seed=seed, outlier_frac=frac)
    packs = [oracle.quantize_weights(synth.weights_f32(N, K, seed=seed + 1 + i))
             for i, N in enumerate(Ns)]
    targets = []
    for (Wq, ws, _), N in zip(packs, Ns):
        targets.append((dev(Wq), dev(np.array([ws], np.float32)),
                        torch.empty((M, N), dtype=torch.float32, device="cuda"),
                        torch.empty((M, N), dtype=torch.int32, device="cuda")))
    xq_out = torch.empty((M, K), dtype=torch.int8, device="cuda")
    xs_out = torch.empty(M, dtype=torch.float32, device="cuda")
    bn.bitnet_linear_bf16(dev_bf16(x), targets, xq_out, xs_out, weights_static=weights_static)
    qx, sx = oracle.quantize_act_bf16(x)
    assert_bits_equal(host(xq_out), qx, "xq_out")
    assert_bits_equal(host(xs_out), sx, "x_scale_out")
    for i, ((Wq, ws, _), t) in enumerate(zip(packs, targets)):
        y_o, acc_o = oracle.linear(Wq, ws, qx, sx, K)
        assert_bits_equal(host(t[3]), acc_o, f"acc target {i}")
        assert_bits_equal(host(t[2]), y_o, f"y target {i}")


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_linear_bf16_decode_layer_group(M):
    # Q, K, V, up, gate of a 2B-class layer share one input
    check_linear_bf16(M, 2560, [2560, 640, 640, 6912, 6912], seed=40 + M,
                      weights_static=(M % 2 == 1))


@pytest.mark.parametrize("M,K,Ns", [(1, 64, [1]), (1, 6912, [2560]), (2, 6912, [33, 2560]),
                                    (1, 28672, [8192]), (2, 28672, [100]), (4, 16384, [77]),
                                    (2, 32768, [9]), (3, 16384, [70]),
                                    (3, 192, [5, 6, 7, 8, 9, 10, 11, 12]), (1, 65536, [40]),
                                    (1, 4096, [4096, 1024, 1024]), (1, 4096, [14336, 14336]),
                                    (1, 14336, [4096])])
def test_linear_bf16_shapes(M, K, Ns):
    check_linear_bf16(M, K, Ns, seed=M * 3 + K, weights_static=True)


def test_linear_bf16_rejects_unsupported():
    x = torch.zeros((4, 65536), dtype=torch.bfloat16, device="cuda")
    Wq = torch.zeros((1, 16384), dtype=torch.uint8, device="cuda")
    t = [(Wq, torch.ones(1, device="cuda"), torch.empty((4, 1), device="cuda"))]
    with pytest.raises(bn.BitnetError) as e:
        bn.bitnet_linear_bf16(x, t)
    assert e.value.status == 2


# ---------------------------------------------------------------- decode chain
def test_decode_chain_matches_separate_calls():
    """A chain of phases with different K and target counts, run twice; every
    output equals the oracle's BitLinear of the phase's own input."""
    M = 1
    spec = [(2560, [2560, 640, 640]), (2560, [2560]), (2560, [6912, 6912]), (6912, [2560]),
            (192, [5, 70]), (28672, [300])]
    phases, refs = [], []
    for i, (K, Ns) in enumerate(spec):
        x = synth.tokens_bf16(M, K, seed=900 + i, outlier_frac=0.01)
        qx, sx = oracle.quantize_act_bf16(x)
        targets, want = [], []
        for j, N in enumerate(Ns):
            Wq, ws, _ = oracle.quantize_weights(synth.weights_f32(N, K, seed=1000 + 10 * i + j))
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
            targets.append((dev(Wq), dev(np.array([ws], np.float32)), y, acc))
            want.append(oracle.linear(Wq, ws, qx, sx, K))
        phases.append((dev_bf16(x), targets))
        refs.append(want)
    chain = bn.bitnet_decode_chain_build(phases)
    for run in range(2):
        for t in (t for _, tg in phases for t in tg):
            t[2].fill_(float("nan"))
        bn.bitnet_decode_chain_run(chain)
        torch.cuda.synchronize()
        assert bn.bitnet_device_error() == 0
        for i, ((_, tg), want) in enumerate(zip(phases, refs)):
            for j, (t, (y_o, acc_o)) in enumerate(zip(tg, want)):
                assert_bits_equal(host(t[3]), acc_o, f"run {run} phase {i} target {j} acc")
                assert_bits_equal(host(t[2]), y_o, f"run {run} phase {i} target {j} y")


def test_decode_chain_phases_without_rows():
    """Phases so small that most CTAs own no row in them, first, last and
    several in a row: every output still matches the oracle (the grid barrier
    counts the CTAs that have nothing to do)."""
    M = 1
    spec = [(192, [5]), (192, [7]), (2560, [2560]), (64, [3]), (64, [2]), (128, [1]),
            (2560, [640]), (64, [4])]
    phases, refs = [], []
    for i, (K, Ns) in enumerate(spec):
        x = synth.tokens_bf16(M, K, seed=1200 + i)
        qx, sx = oracle.quantize_act_bf16(x)
        targets, want = [], []
        for j, N in enumerate(Ns):
            Wq, ws, _ = oracle.quantize_weights(synth.weights_f32(N, K, seed=1300 + 10 * i + j))
            targets.append((dev(Wq), dev(np.array([ws], np.float32)),
                            torch.empty((M, N), dtype=torch.float32, device="cuda")))
            want.append(oracle.linear(Wq, ws, qx, sx, K)[0])
        phases.append((dev_bf16(x), targets))
        refs.append(want)
    chain = bn.bitnet_decode_chain_build(phases)
    for run in range(3):
        bn.bitnet_decode_chain_run(chain)
    torch.cuda.synchronize()
    assert bn.bitnet_device_error() == 0
    for i, ((_, tg), want) in enumerate(zip(phases, refs)):
        for t, y_o in zip(tg, want):
            assert_bits_equal(host(t[2]), y_o, f"phase {i} y")


@pytest.mark.parametrize("M", [2, 3])
def test_decode_chain_multi_token(M):
    spec = [(2560, [2560, 640]), (6912, [2560]), (2560, [6912])]
    phases, refs = [], []
    for i, (K, Ns) in enumerate(spec):
        x = synth.tokens_bf16(M, K, seed=950 + i)
        qx, sx = oracle.quantize_act_bf16(x)
        targets, want = [], []
        for j, N in enumerate(Ns):
            Wq, ws, _ = oracle.quantize_weights(synth.weights_f32(N, K, seed=1100 + 10 * i + j))
            targets.append((dev(Wq), dev(np.array([ws], np.float32)),
                            torch.empty((M, N), dtype=torch.float32, device="cuda")))
            want.append(oracle.linear(Wq, ws, qx, sx, K)[0])
        phases.append((dev_bf16(x), targets))
        refs.append(want)
    chain = bn.bitnet_decode_chain_build(phases)
    bn.bitnet_decode_chain_run(chain)
    torch.cuda.synchronize()
    for (_, tg), want in zip(phases, refs):
        for t, y_o in zip(tg, want):
            assert_bits_equal(host(t[2]), y_o, "chain y")


# ---------------------------------------------------------------- bf16 outputs
def _bf16(t):
    return host(t.view(torch.int16)).view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(1, 2560, 2560), (3, 100, 192), (8, 2560, 6912),
                                   (64, 6912, 2560), (300, 264, 640), (4096, 2560, 2560)])
def test_linear_bf16_output_every_path(M, N, K):
    """The bf16 form of the rescaled output (nearest, ties to even) on every
    path of bitnet_linear: decode (M <= 4), CUDA cores (5..15), fused tensor
    cores (16..256, split K included), pre-expanded tensor cores (> 256)."""
    Wq, ws, qx, sx = linear_inputs(M, N, K, seed=M + N, frac=0.01)
    y_o, acc_o = oracle.linear(Wq, ws, qx, sx, K, threads=oracle.default_threads())
    yb = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    args = (dev(Wq), dev(np.array([ws], np.float32)), dev(qx), dev(sx))
    bn.bitnet_linear(*args, K=K, y=None, y_bf16=yb)            # bf16 only
    assert_bits_equal(_bf16(yb), oracle.f32_to_bf16(y_o), "y_bf16 alone")
    yb.view(torch.int16).fill_(0x7fc1)
    bn.bitnet_linear(*args, K=K, y=y, y_bf16=yb)               # both forms
    assert_bits_equal(host(y), y_o, "y")
    assert_bits_equal(_bf16(yb), oracle.f32_to_bf16(y_o), "y_bf16 with y")


# ---------------------------------------------------------------- dependent launches
@pytest.mark.parametrize("weights_static", [False, True])
def test_back_to_back_decode_launches_carry_the_data(weights_static):
    """Programmatic dependent launch: launch 2 reads, as its bf16 input, the
    bytes launch 1 writes; launch 3 reads launch 2's output.  With static
    weights the weight stream starts before the previous launch ends; the
    input must still be read after it.  Repeated with the outputs poisoned."""
    H = 2560
    x = synth.tokens_bf16(1, H, seed=61, outlier_frac=0.01)
    W = [oracle.quantize_weights(synth.weights_f32(H, H, seed=610 + i))[:2] for i in range(3)]
    Wd = [(dev(Wq), dev(np.array([ws], np.float32))) for Wq, ws in W]
    ys = [torch.empty((1, H), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    xd = dev_bf16(x)
    want, cur = [], x
    for Wq, ws in W:
        qx, sx = oracle.quantize_act_bf16(cur)
        cur = oracle.f32_to_bf16(oracle.linear(Wq, ws, qx, sx, H)[0])
        want.append(cur)
    for rep in range(5):
        for t in ys:
            t.view(torch.int16).fill_(0x7fc1)
        for i in range(3):
            bn.bitnet_linear_bf16(xd if i == 0 else ys[i - 1],
                                  [(*Wd[i], None, None, ys[i])], weights_static=weights_static)
        for i in range(3):
            assert_bits_equal(_bf16(ys[i]), want[i], f"rep {rep} launch {i}")


# ---------------------------------------------------------------- bounded waits
def test_a_wait_that_runs_out_reports_and_leaves_the_context_usable():
    """A link word that nothing will write: the chain's run counter is set so
    that one CTA takes another run number than the rest, so the tags it waits
    for are never written (and the others wait for its outputs under their
    own tag).  With a short wait bound (about a millisecond) every such wait
    runs out: the kernel records the link-wait bit, its producer waits for
    its copies in flight, and it returns; nothing hangs or faults.
    bitnet_device_error reports the bit; the chain rebuilt with the default
    bound is exact again."""
    H = 2560
    x = synth.tokens_bf16(1, H, seed=65)
    packs = [oracle.quantize_weights(synth.weights_f32(H, H, seed=650 + i))[:2] for i in range(2)]
    Wd = [(dev(Wq), dev(np.array([ws], np.float32))) for Wq, ws in packs]
    y0 = torch.empty((1, H), dtype=torch.bfloat16, device="cuda")
    y1 = torch.empty((1, H), dtype=torch.float32, device="cuda")
    phases = [{"x": dev_bf16(x), "targets": [(*Wd[0], None, None, y0)]},
              {"x": y0, "targets": [(*Wd[1], y1)]}]
    chain = bn.bitnet_decode_chain_build(phases)
    assert bn.bitnet_device_error() == 0
    ctas = chain.chain.cfg[6]
    base = chain.chain.table - chain.table.data_ptr()   # the table's first word: the run counter
    chain.table[base:base + 8].view(torch.int64).fill_(ctas - 1)
    try:
        bn.bitnet_set_wait_limit(2_000_000)             # ~1 ms
        t0 = time.perf_counter()
        bn.bitnet_decode_chain_run(chain)
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 30
        code = bn.bitnet_device_error()
        assert code & (1 << 16), hex(code)              # a chain input never came
        assert bn.bitnet_device_error() == 0            # read and cleared
    finally:
        bn.bitnet_set_wait_limit(0)
    chain = bn.bitnet_decode_chain_build(phases)        # rebuilt after the error
    for _ in range(2):
        bn.bitnet_decode_chain_run(chain)
    torch.cuda.synchronize()
    assert bn.bitnet_device_error() == 0
    qx, sx = oracle.quantize_act_bf16(x)
    y0_o = oracle.f32_to_bf16(oracle.linear(*packs[0], qx, sx, H)[0])
    assert_bits_equal(_bf16(y0), y0_o, "y0 after the time-out")
    qx, sx = oracle.quantize_act_bf16(y0_o)
    assert_bits_equal(host(y1), oracle.linear(*packs[1], qx, sx, H)[0], "y1 after the time-out")
