"""GPU parity of the fused BitNet feed-forward block against the oracle,
stage by stage (normalised-and-quantised input, up, gate, h, its quantisation,
the down accumulator) and end to end."""
import numpy as np
import pytest
import torch

import oracle
import bitlinear_bitnet_linear_03_b300 as bn
from bitlinear_bitnet_linear_03_b300 import synth
from gpu_util import assert_bits_equal, assert_f32_close, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

H, F = 2560, 6912


def ffn_inputs(M, seed, H=H, F=F, random_gain=False):
    Wup = synth.weights_f32(F, H, seed=seed * 10 + 1)
    Wgate = synth.weights_f32(F, H, seed=seed * 10 + 2)
    Wdown = synth.weights_f32(H, F, seed=seed * 10 + 3)
    x = synth.tokens_bf16(M, H, seed=seed * 10 + 4)
    g = synth.gain_random(H, seed) if random_gain else synth.gain_ones(H)
    return x, g, [oracle.quantize_weights(W) for W in (Wup, Wgate, Wdown)]


def run_gpu(x, g, eps, ws, M, H, F):
    dbg = dict(xq=torch.empty((M, H), dtype=torch.int8, device="cuda"),
               sx=torch.empty(M, dtype=torch.float32, device="cuda"),
               u=torch.empty((M, F), dtype=torch.float32, device="cuda"),
               v=torch.empty((M, F), dtype=torch.float32, device="cuda"),
               h=torch.empty((M, F), dtype=torch.float32, device="cuda"),
               hq=torch.empty((M, F), dtype=torch.int8, device="cuda"),
               sh=torch.empty(M, dtype=torch.float32, device="cuda"),
               acc_down=torch.empty((M, H), dtype=torch.int32, device="cuda"))
    (Wu, su, _), (Wg, sg, _), (Wd, sd, _) = ws
    f32 = lambda v: dev(np.array([v], np.float32))
    y = bn.bitnet_ffn(dev_bf16(x), dev(g), eps, dev(Wu), f32(su), dev(Wg), f32(sg), dev(Wd),
                      f32(sd), debug=dbg)
    out = {k: host(v) for k, v in dbg.items()}
    out["y"] = host(y)
    return out


def check_ffn(M, seed, H=H, F=F, random_gain=False, eps=1e-5):
    x, g, ws = ffn_inputs(M, seed, H, F, random_gain)
    got = run_gpu(x, g, eps, ws, M, H, F)
    (Wu, su, _), (Wg, sg, _), (Wd, sd, _) = ws
    want = oracle.ffn(x, g, eps, Wu, su, Wg, sg, Wd, sd, threads=oracle.default_threads())
    # every intermediate stage against the oracle's own (the oracle computes
    # each stage from its previous one; no GPU value enters it)
    for k in ("sx", "xq", "u", "v", "h", "sh", "hq", "acc_down"):
        assert_bits_equal(got[k], want[k], k)
    # end to end
    assert_f32_close(got["y"], want["y"], "y")
    assert_bits_equal(got["y"], want["y"], "y bits")


@pytest.mark.parametrize("seed", range(4))
def test_ffn_seq1(seed):
    check_ffn(1, seed)


@pytest.mark.parametrize("M", [3, 8, 64])
def test_ffn_small_batches(M):
    check_ffn(M, 0, random_gain=True)


def test_ffn_ragged_dims():
    check_ffn(5, 1, H=192, F=320, random_gain=True)


def test_ffn_without_debug_matches():
    M = 2
    x, g, ws = ffn_inputs(M, 3)
    (Wu, su, _), (Wg, sg, _), (Wd, sd, _) = ws
    f32 = lambda v: dev(np.array([v], np.float32))
    y = host(bn.bitnet_ffn(dev_bf16(x), dev(g), 1e-5, dev(Wu), f32(su), dev(Wg), f32(sg),
                           dev(Wd), f32(sd)))
    want = oracle.ffn(x, g, 1e-5, Wu, su, Wg, sg, Wd, sd)
    assert_bits_equal(y, want["y"], "y")


@pytest.mark.parametrize("M,seed", [(1, 0), (1, 1), (3, 2), (4, 3)])
def test_ffn_partial_debug_outputs(M, seed):
    """Only some intermediate outputs requested (no fp32 h): the codes, scale
    and accumulators reported, and y, equal the oracle's."""
    x, g, ws = ffn_inputs(M, seed, random_gain=(seed % 2 == 1))
    (Wu, su, _), (Wg, sg, _), (Wd, sd, _) = ws
    dbg = dict(u=torch.empty((M, F), dtype=torch.float32, device="cuda"),
               v=torch.empty((M, F), dtype=torch.float32, device="cuda"),
               hq=torch.empty((M, F), dtype=torch.int8, device="cuda"),
               sh=torch.empty(M, dtype=torch.float32, device="cuda"),
               acc_down=torch.empty((M, H), dtype=torch.int32, device="cuda"))
    f32 = lambda v: dev(np.array([v], np.float32))
    y = host(bn.bitnet_ffn(dev_bf16(x), dev(g), 1e-5, dev(Wu), f32(su), dev(Wg), f32(sg),
                           dev(Wd), f32(sd), debug=dbg))
    got = {k: host(v) for k, v in dbg.items()}
    want = oracle.ffn(x, g, 1e-5, Wu, su, Wg, sg, Wd, sd)
    for k in ("u", "v", "sh", "hq", "acc_down"):
        assert_bits_equal(got[k], want[k], k)
    assert_bits_equal(y, want["y"], "y end to end")


@pytest.mark.parametrize("H", [256, 2560])
def test_ffn_norm_special_rows(H):
    """Rows that exercise the exact sum of squares: the row whose exact sum
    rounds differently from a binary64 or running binary32 sum, an all-zero
    row, subnormal and tiny values (a row whose squares span more than the
    128-bit window), values whose squares overflow binary32 (ss = inf,
    r = 0), and an ordinary row."""
    M, F = 6, 320
    rows = np.zeros((M, H), np.float32)
    rows[0, 3], rows[0, 20], rows[0, 41], rows[0, 63] = 1490944.0, 256.0, 256.0, 2.0 ** -20
    rows[2, ::3] = 2.0 ** -130                      # subnormal bf16 values: squares underflow
    rows[3, ::5] = 3.0e-20
    rows[3, 1] = 7.0
    rows[4, 7] = 3.0e20                             # square above the binary32 range
    rows[5] = synth.bf16_bits_to_f32(synth.tokens_bf16(1, H, seed=5))[0]
    x = synth.f32_to_bf16_bits(rows)
    g = synth.gain_random(H, 3)
    ws = [oracle.quantize_weights(synth.weights_f32(n, k, seed=80 + i))
          for i, (n, k) in enumerate([(F, H), (F, H), (H, F)])]
    got = run_gpu(x, g, 1e-5, ws, M, H, F)
    n, _ = oracle.rmsnorm_bf16(x, g, np.float32(1e-5))
    q, s = oracle.quantize_act_f32(n)
    assert_bits_equal(got["xq"], q, "xq")
    assert_bits_equal(got["sx"], s, "sx")
    assert (got["xq"][1] == 0).all() and (got["xq"][4] == 0).all()


@pytest.mark.parametrize("seed", range(4))
def test_ffn_seq4096_sampled_tokens(seed):
    """The prefill-sized FFN (seq 4096, hidden 2560, FFN 6912): the GPU runs
    every token; the oracle recomputes 24 sampled tokens (the block is
    independent per token), first and last included, and every intermediate
    at those tokens must match bit for bit."""
    M = 4096
    x, g, ws = ffn_inputs(M, seed, random_gain=(seed % 2 == 1))
    got = run_gpu(x, g, 1e-5, ws, M, H, F)
    rows = np.random.default_rng(seed).choice(M, 24, replace=False)
    rows[:2] = [0, M - 1]
    (Wu, su, _), (Wg, sg, _), (Wd, sd, _) = ws
    want = oracle.ffn(x[rows], g, 1e-5, Wu, su, Wg, sg, Wd, sd, threads=oracle.default_threads())
    for k in ("sx", "xq", "u", "v", "h", "sh", "hq", "acc_down", "y"):
        assert_bits_equal(got[k][rows], want[k], f"seed {seed} {k}")
    # every token: the properties that hold at any size
    assert np.isfinite(got["y"]).all()
    assert (np.abs(got["xq"]).max(axis=1) == 127).all()


@pytest.mark.parametrize("H_,F_", [(64, 192), (128, 64)])
def test_ffn_prefill_small_dims(H_, F_):
    """Above 256 tokens with K below 128 on one side: (64, 192) runs the gated
    up/gate GEMM on bf16 operands and the down GEMM in the e4m3 digit form
    (K = 192, one and a half 128-deep stages); (128, 64) the reverse.  Every
    stage, all 300 tokens."""
    check_ffn(300, 7, H=H_, F=F_, random_gain=True)


@pytest.mark.parametrize("M,seed", [(300, 5), (512, 6)])
def test_ffn_prefill_gated_gemm_without_intermediates(M, seed):
    """Above 256 tokens the up and gate products run as one GEMM whose
    epilogue forms h; with no intermediate outputs requested h lives in the
    workspace.  Sampled tokens (first and last included) must match the
    oracle bit for bit: the codes and scale of h, the down accumulators, y."""
    x, g, ws = ffn_inputs(M, seed, random_gain=True)
    (Wu, su, _), (Wg, sg, _), (Wd, sd, _) = ws
    dbg = dict(hq=torch.empty((M, F), dtype=torch.int8, device="cuda"),
               sh=torch.empty(M, dtype=torch.float32, device="cuda"),
               acc_down=torch.empty((M, H), dtype=torch.int32, device="cuda"))
    f32 = lambda v: dev(np.array([v], np.float32))
    y = host(bn.bitnet_ffn(dev_bf16(x), dev(g), 1e-5, dev(Wu), f32(su), dev(Wg), f32(sg),
                           dev(Wd), f32(sd), debug=dbg))
    got = {k: host(v) for k, v in dbg.items()}
    rows = np.random.default_rng(seed).choice(M, 16, replace=False)
    rows[:2] = [0, M - 1]
    want = oracle.ffn(x[rows], g, 1e-5, Wu, su, Wg, sg, Wd, sd, threads=oracle.default_threads())
    for k in ("sh", "hq", "acc_down"):
        assert_bits_equal(got[k][rows], want[k], k)
    assert_bits_equal(y[rows], want["y"], "y")
