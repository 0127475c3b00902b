"""Pins for the CPU oracle: worked examples, exact rational arithmetic, closed
forms, invariants and brute force.  CPU only (no GPU marker).

Each test names the definition it pins; a plausible mistake in the oracle (a
dropped term, a wrong sign or index, a transposed operand, ties rounded away
from zero, a reciprocal instead of a division, a wrong bit layout) fails at
least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bitlinear_bitnet_linear_03_b300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


# ---------------------------------------------------------------- helpers
def exact(v) -> Fraction:
    return Fraction(*float(v).as_integer_ratio())


def rn32(fr: Fraction) -> np.float32:
    """Nearest binary32 to an exact rational, ties to even (test-side)."""
    if fr == 0:
        return np.float32(0.0)
    neg = fr < 0
    a = -fr if neg else fr
    c = np.float32(float(a))
    cands = [np.nextafter(c, np.float32(0), dtype=np.float32), c,
             np.nextafter(c, np.float32(np.inf), dtype=np.float32)]
    best = None
    for cand in cands:
        d = abs(exact(cand) - a)
        key = (d, int(np.array(cand, np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    r = best[1]
    return np.float32(-r) if neg else np.float32(r)


def exact_mean_abs(W) -> Fraction:
    s = sum((exact(abs(float(w))) for w in np.asarray(W, np.float32).ravel()), Fraction(0))
    return s / W.size


# ---------------------------------------------------------------- absmean
def test_absmean_worked_examples():
    g = GOLD["weights_ties"]
    assert oracle.absmean(np.array(g["W"], np.float32)) == np.float32(g["gamma"])
    g = GOLD["weights_plain"]
    assert oracle.absmean(np.array(g["W"], np.float32)) == np.float32(g["gamma"])


@pytest.mark.parametrize("seed", range(6))
def test_absmean_is_exact_mean_rounded_once(seed):
    rng = np.random.default_rng(seed)
    shape = [(3, 5), (17, 64), (64, 128), (1, 1), (200, 33), (7, 1000)][seed]
    # Mixed magnitudes so that a float sum in any fixed order would round.
    W = (rng.standard_normal(shape) * np.exp2(rng.integers(-30, 30, shape))).astype(np.float32)
    assert oracle.absmean(W) == rn32(exact_mean_abs(W))


def test_absmean_subnormals_and_huge():
    tiny = np.array([1e-45, 3e-45, 1e-40, 0.0], np.float32)
    assert oracle.absmean(tiny) == rn32(exact_mean_abs(tiny))
    big = np.array([3.0e38, 3.0e38, 1.0, 2.0e38], np.float32)
    assert oracle.absmean(big) == rn32(exact_mean_abs(big))


def test_absmean_ties_to_even():
    one = np.float32(1.0)
    u = np.float32(2.0 ** -23)
    # mean = 1 + 2^-24: exactly halfway between 1 and 1+2^-23 -> 1 (even)
    assert oracle.absmean(np.array([one, one + u], np.float32)) == one
    # mean = 1 + 3*2^-24: halfway between 1+2^-23 (odd) and 1+2^-22 (even)
    assert oracle.absmean(np.array([one + u, one + 2 * u], np.float32)) == one + 2 * u


def test_absmean_closed_forms():
    c = np.float32(0.0137)
    W = np.full((64, 64), c, np.float32)
    W[::2] *= -1
    assert oracle.absmean(W) == c                     # |c| * n / n
    assert oracle.absmean(np.zeros((4, 64), np.float32)) == 0.0
    # 2^24 + 1 ones cannot be summed in binary32; exact mean is 1
    assert oracle.absmean(np.ones(2 ** 24 + 1, np.float32)) == 1.0


def test_absmean_nonfinite_is_nan():
    W = np.ones(64, np.float32)
    W[5] = np.inf
    assert np.isnan(oracle.absmean(W))
    W[5] = np.nan
    assert np.isnan(oracle.absmean(W))


def test_absmean_large_random_matches_fraction():
    W = synth.weights_f32(96, 640, seed=7)
    assert oracle.absmean(W) == rn32(exact_mean_abs(W))


# ---------------------------------------------------------------- ternarize
def test_ternarize_worked_examples():
    g = GOLD["weights_ties"]
    q, ws = oracle.ternarize(np.array(g["W"], np.float32), np.float32(g["gamma"]))
    assert ws == np.float32(g["gamma"])
    assert q.tolist() == g["q"]
    g = GOLD["weights_plain"]
    W = np.array(g["W"], np.float32).reshape(1, -1)
    q, ws = oracle.ternarize(W, oracle.absmean(W))
    assert q.ravel().tolist() == g["q"]


def test_ternarize_zero_matrix_uses_floor_scale():
    W = np.zeros((3, 64), np.float32)
    Wq, ws, q = oracle.quantize_weights(W)
    assert ws == np.float32(1e-5)
    assert (q == 0).all() and (Wq == 0x55).all()


def test_ternarize_sign_pattern():
    rng = np.random.default_rng(1)
    s = rng.choice([-1.0, 1.0], size=(32, 128)).astype(np.float32)
    c = np.float32(0.25)
    Wq, ws, q = oracle.quantize_weights(s * c)
    assert ws == c
    assert (q == s).all()


def test_ternarize_uses_true_division():
    # W/g rounded once, not W*(1/g): search weights next to g/2 until the two
    # forms land on different sides of the 0.5 tie, then check the oracle.
    rng = np.random.default_rng(11)
    found = 0
    for _ in range(20000):
        g = np.float32(rng.uniform(0.005, 0.05))
        rec = np.float32(np.float32(1.0) / g)
        w = np.float32(g / np.float32(2.0))
        for _ in range(3):
            a = np.rint(np.float32(w / g))
            b = np.rint(np.float32(w * rec))
            if a != b:
                q, _ = oracle.ternarize(np.array([[w, -w]], np.float32), g)
                assert q.ravel().tolist() == [int(a), -int(a)]
                found += 1
            w = np.nextafter(w, np.float32(1), dtype=np.float32)
        if found >= 5:
            break
    assert found >= 1
    # exact tie g/2 -> 0 (half to even)
    g = np.float32(0.3)
    q, _ = oracle.ternarize(np.array([[g / np.float32(2.0)]], np.float32), g)
    assert q[0, 0] == 0


def test_zero_fraction_statistic():
    # For N(0, s) weights: P(|w| < gamma/2), gamma = s*sqrt(2/pi) -> erf(0.5/sqrt(pi))
    W = synth.weights_f32(2560, 2560, seed=0)
    _, _, q = oracle.quantize_weights(W)
    frac = float((q == 0).mean())
    assert abs(frac - math.erf(0.5 / math.sqrt(math.pi))) < 0.002
    assert set(np.unique(q).tolist()) == {-1, 0, 1}
    # symmetric distribution -> +1 and -1 about equally often
    assert abs(float((q == 1).mean()) - float((q == -1).mean())) < 0.002


# ---------------------------------------------------------------- pack
def test_pack_single_weight_layout():
    g = GOLD["pack_single"]
    q = np.zeros((1, g["K"]), np.int8)
    q[0, g["nonzero_k"]] = g["nonzero_q"]
    assert oracle.pack(q).ravel().tolist() == g["bytes"]


def test_pack_roundtrip_and_size():
    rng = np.random.default_rng(3)
    for N, K in [(1, 64), (5, 192), (33, 2560)]:
        q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
        Wq = oracle.pack(q)
        assert Wq.nbytes == N * K // 4              # 2 bits per weight
        assert (oracle.unpack(Wq, K) == q).all()


def test_pack_word_fields_are_consecutive_weights():
    # In a 16-byte block, 32-bit word i shifted right by 2s and masked with
    # 0x03030303 gives the codes of weights 64b + 16s + 4i + {0,1,2,3}.
    rng = np.random.default_rng(4)
    K = 256
    q = rng.integers(-1, 2, size=(2, K)).astype(np.int8)
    words = oracle.pack(q).view("<u4")
    for n in range(2):
        for b in range(K // 64):
            for i in range(4):
                w = int(words[n, b * 4 + i])
                for s in range(4):
                    v = (w >> (2 * s)) & 0x03030303
                    codes = [(v >> (8 * t)) & 0xFF for t in range(4)]
                    k0 = 64 * b + 16 * s + 4 * i
                    assert codes == (q[n, k0:k0 + 4] + 1).tolist()


def test_unpack_rejects_code_3():
    Wq = np.full((1, 16), 0x55, np.uint8)
    Wq[0, 3] = 0x57
    with pytest.raises(ValueError):
        oracle.unpack(Wq, 64)


def test_100b_footprint_scales_as_two_bits():
    # 8192 x 28672 ternary weights occupy N*K/4 bytes (2 bits each)
    N, K = 8192, 28672
    assert N * K // 4 == 58_720_256


# ---------------------------------------------------------------- act quant
def test_act_quant_worked_example():
    g = GOLD["act_ties"]
    x = synth.f32_to_bf16_bits(np.array([g["x"]], np.float32))
    assert (synth.bf16_bits_to_f32(x) == np.array(g["x"], np.float32)).all()
    q, sx = oracle.quantize_act_bf16(x)
    assert q.ravel().tolist() == g["q"]
    assert sx[0] == np.float32(g["sx"])
    q2, sx2 = oracle.quantize_act_f32(np.array([g["x"]], np.float32))
    assert q2.ravel().tolist() == g["q"] and sx2[0] == sx[0]


def test_act_quant_zero_token():
    q, sx = oracle.quantize_act_f32(np.zeros((2, 64), np.float32))
    assert (q == 0).all()
    assert sx[0] == np.float32(np.float32(1e-5) / np.float32(127.0))


def test_act_quant_invariants():
    x = synth.tokens_bf16(16, 2560, seed=1, outlier_frac=0.01)
    q, sx = oracle.quantize_act_bf16(x)
    xf = synth.bf16_bits_to_f32(x)
    assert (np.abs(q).max(axis=1) == 127).all()          # absmax maps to 127
    assert (q >= -127).all()                               # -128 unreachable
    err = np.abs(q.astype(np.float64) * sx[:, None] - xf)
    assert (err <= sx[:, None] * (0.5 + 1e-5)).all()       # half a step
    amax = np.abs(xf).max(axis=1)
    assert (sx == (amax / np.float32(127.0)).astype(np.float32)).all()


def test_act_quant_scale_uses_product_with_inverse():
    # q = rint(x * (127/a)).  Search x next to half-integer quotients until
    # x*(127/a) and (127*x)/a round to different integers, then check the
    # oracle follows the first form.
    rng = np.random.default_rng(5)
    found = 0
    for _ in range(4000):
        a = np.float32(rng.uniform(1, 10))
        inv = np.float32(127.0) / a
        t = np.float32(rng.integers(0, 126) + 0.5)
        x = np.float32(t * a / np.float32(127.0))
        for _ in range(4):
            p = np.float32(x * inv)
            d = np.float32(np.float32(x * np.float32(127.0)) / a)
            if np.rint(p) != np.rint(d):
                q, _ = oracle.quantize_act_f32(np.array([[a, x]], np.float32))
                assert q[0, 1] == np.rint(p)
                found += 1
            x = np.nextafter(x, np.float32(100), dtype=np.float32)
        if found >= 5:
            break
    assert found >= 1


# ---------------------------------------------------------------- linear
def test_linear_worked_example():
    g = GOLD["linear"]
    qw = np.array(g["qw"], np.int8)
    qx = np.array([g["qx"]], np.int8)
    acc = oracle.linear_acc(qw, qx)
    assert acc.ravel().tolist() == g["acc"]
    y = oracle.rescale(acc, np.array([g["sx"]], np.float32), np.float32(g["w_scale"]))
    assert y.ravel().tolist() == g["y"]


@pytest.mark.parametrize("M,N,K", [(1, 7, 64), (3, 65, 192), (5, 128, 2560)])
def test_linear_acc_brute_force_matmul(M, N, K):
    rng = np.random.default_rng(M * 1000 + N)
    qw = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    qx = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    acc = oracle.linear_acc(qw, qx)
    assert (acc == qx.astype(np.int64) @ qw.astype(np.int64).T).all()
    # offset form used with 2-bit codes: sum(code*x) - sum(x)
    codes = (qw + 1).astype(np.int64)
    off = qx.astype(np.int64) @ codes.T - qx.astype(np.int64).sum(axis=1, keepdims=True)
    assert (acc == off).all()
    assert (oracle.linear_acc(qw, qx, threads=4) == acc).all()


def test_linear_extreme_values_exact():
    K = 65536 - 64
    qw = np.ones((2, K), np.int8)
    qw[1] = -1
    qx = np.full((1, K), -128, np.int8)
    acc = oracle.linear_acc(qw, qx)
    assert acc.ravel().tolist() == [-128 * K, 128 * K]


def test_linear_one_hot_token():
    W = synth.weights_f32(64, 128, seed=2)
    Wq, ws, q = oracle.quantize_weights(W)
    x = np.zeros((1, 128), np.float32)
    x[0, 37] = 3.0
    qx, sx = oracle.quantize_act_f32(x)
    y, acc = oracle.linear(Wq, ws, qx, sx, 128)
    assert (acc[0] == 127 * q[:, 37]).all()
    assert np.allclose(y[0], q[:, 37] * ws * 3.0, rtol=1e-6)


def test_linear_matches_fp64_dequantized_matmul():
    W = synth.weights_f32(96, 256, seed=3)
    x = synth.tokens_bf16(4, 256, seed=4)
    Wq, ws, q = oracle.quantize_weights(W)
    qx, sx = oracle.quantize_act_bf16(x)
    y, _ = oracle.linear(Wq, ws, qx, sx, 256)
    ref = (qx.astype(np.float64) * sx[:, None].astype(np.float64)) @ (
        q.astype(np.float64) * np.float64(ws)).T
    assert np.allclose(y, ref, rtol=1e-6, atol=1e-6 * np.abs(ref).max())


def test_rescale_operation_order():
    # y = (float)acc * (sx * w): find operands where the other order differs
    rng = np.random.default_rng(6)
    found = 0
    for _ in range(2000):
        acc = np.int32(rng.integers(-100000, 100000))
        sx = np.float32(rng.uniform(0.01, 0.1))
        w = np.float32(rng.uniform(0.01, 0.03))
        want = np.float32(np.float32(acc) * np.float32(sx * w))
        other = np.float32(np.float32(np.float32(acc) * sx) * w)
        if want != other:
            found += 1
            y = oracle.rescale(np.array([[acc]], np.int32), np.array([sx], np.float32), w)
            assert y[0, 0] == want
        if found > 5:
            break
    assert found > 0


# ---------------------------------------------------------------- rmsnorm / FFN pieces
def test_rmsnorm_constant_row():
    g = GOLD["rmsnorm_constant"]
    H = g["H"]
    x = synth.f32_to_bf16_bits(np.full((1, H), g["c"], np.float32))
    n, r = oracle.rmsnorm_bf16(x, synth.gain_ones(H), g["eps"])
    assert (n == np.float32(g["n_all"])).all()
    q, _ = oracle.quantize_act_f32(n)
    assert (q == g["q_all"]).all()


def _rmsnorm_r_by_fractions(xf32_row, H, eps):
    """Test-side statement of the reading: exact sum of the binary32 squares
    (Fractions), one rounding to binary32, then binary32 steps (numpy)."""
    sq = [np.float32(v) * np.float32(v) for v in xf32_row]
    ss = rn32(sum((exact(t) for t in sq), Fraction(0)))
    q = np.float32(ss) / np.float32(H)
    t = np.float32(q + np.float32(eps))
    return np.float32(np.float32(1.0) / np.sqrt(t))


def test_rmsnorm_exact_sum_and_binary32_steps():
    x = synth.tokens_bf16(8, 2560, seed=9, outlier_frac=0.01)
    gain = synth.gain_random(2560, seed=1)
    eps = np.float32(1e-5)
    n, r = oracle.rmsnorm_bf16(x, gain, eps)
    xf = synth.bf16_bits_to_f32(x)
    ref = xf.astype(np.float64) / np.sqrt((xf.astype(np.float64) ** 2).mean(axis=1, keepdims=True)
                                          + float(eps)) * gain
    assert np.allclose(n, ref, rtol=3e-7 * 4, atol=0)
    for m in range(8):
        assert r[m] == _rmsnorm_r_by_fractions(xf[m], 2560, eps), m
        # n is two binary32 products per element, in this order
        assert (n[m] == (xf[m] * r[m]) * gain).all()


def test_rmsnorm_sum_is_exact_not_sequential():
    """x = 1490944 (= 182 * 2^13), 256, 256 and 2^-20: the squares 182^2 * 2^26,
    2^16, 2^16 and 2^-40 sum to just above the tie between two binary32
    neighbours (2^16 + 2^16 is exactly half an ulp of the first square), so
    the exact sum rounds up.  A binary64 sum drops 2^-40, lands on the tie
    and rounds to even (down); a binary32 running sum drops both 2^16 terms.
    With H = 64 and eps = 0 the two candidate sums give different r."""
    H = 64
    row = np.zeros(H, np.float32)
    row[3], row[20], row[41], row[63] = 1490944.0, 256.0, 256.0, 2.0 ** -20
    x = synth.f32_to_bf16_bits(row[None, :])
    assert (synth.bf16_bits_to_f32(x)[0] == row).all()
    _, r = oracle.rmsnorm_bf16(x, synth.gain_ones(H), np.float32(0.0))
    sq = [exact(np.float32(v) * np.float32(v)) for v in row]
    ss_exact = rn32(sum(sq, Fraction(0)))
    ss_f64 = np.float32(sum(float(t) for t in sq))
    assert ss_exact != ss_f64
    r_of = lambda ss: np.float32(np.float32(1.0) / np.sqrt(np.float32(ss / np.float32(H))))
    assert r[0] == r_of(ss_exact)
    assert r_of(ss_f64) != r[0]
    assert r[0] == _rmsnorm_r_by_fractions(row, H, np.float32(0.0))


def test_rmsnorm_nonfinite_rows():
    H = 64
    x = synth.tokens_bf16(3, H, seed=4)
    x[0, 7] = 0x7f80          # +inf: ss = inf, r = 0
    x[1, 9] = 0x7fc0          # nan
    x[2, :] = 0               # zero row: r = 1/sqrt(eps)
    n, r = oracle.rmsnorm_bf16(x, synth.gain_ones(H), np.float32(1e-5))
    assert r[0] == 0.0 and np.isnan(r[1])
    assert r[2] == np.float32(np.float32(1.0) / np.sqrt(np.float32(1e-5)))
    assert (n[2] == 0).all()


def test_relu2_worked_example():
    g = GOLD["relu2"]
    h = oracle.relu2_mul(np.array(g["up"], np.float32), np.array(g["gate"], np.float32))
    assert h.tolist() == g["h"]


def _ffn_inputs(M, H, F, seed):
    Wup = synth.weights_f32(F, H, seed=seed * 10 + 1)
    Wgate = synth.weights_f32(F, H, seed=seed * 10 + 2)
    Wdown = synth.weights_f32(H, F, seed=seed * 10 + 3)
    x = synth.tokens_bf16(M, H, seed=seed * 10 + 4)
    up = oracle.quantize_weights(Wup)
    gate = oracle.quantize_weights(Wgate)
    down = oracle.quantize_weights(Wdown)
    return x, up, gate, down


def test_ffn_is_the_composition_and_close_to_fp64():
    M, H, F = 3, 128, 192
    x, up, gate, down = _ffn_inputs(M, H, F, seed=0)
    g = synth.gain_random(H, seed=2)
    eps = 1e-5
    out = oracle.ffn(x, g, eps, up[0], up[1], gate[0], gate[1], down[0], down[1])
    # composition of the separately pinned pieces
    n, _ = oracle.rmsnorm_bf16(x, g, eps)
    xq, sx = oracle.quantize_act_f32(n)
    u, _ = oracle.linear(up[0], up[1], xq, sx, H)
    v, _ = oracle.linear(gate[0], gate[1], xq, sx, H)
    h = oracle.relu2_mul(u, v)
    hq, sh = oracle.quantize_act_f32(h)
    y, accd = oracle.linear(down[0], down[1], hq, sh, F)
    for k, ref in dict(xq=xq, sx=sx, u=u, v=v, h=h, hq=hq, sh=sh, y=y, acc_down=accd).items():
        assert (out[k] == ref).all(), k
    # fp64 model on the same integer codes: u, v and y agree to rounding
    u64 = (xq.astype(np.float64) @ up[2].T.astype(np.float64)) * sx[:, None] * float(up[1])
    assert np.allclose(out["u"], u64, rtol=1e-6, atol=1e-6 * np.abs(u64).max())
    y64 = (hq.astype(np.float64) @ down[2].T.astype(np.float64)) * sh[:, None] * float(down[1])
    assert np.allclose(out["y"], y64, rtol=1e-6, atol=1e-6 * np.abs(y64).max())
    # h is relu(v)^2 * u
    assert np.allclose(out["h"], np.maximum(v, 0).astype(np.float64) ** 2 * u, rtol=1e-6)


# ---------------------------------------------------------------- bf16 output rounding
def test_f32_to_bf16_worked_ties():
    one = 1.0
    cases = [
        (one, 0x3F80),
        (one + 2.0 ** -8, 0x3F80),                 # tie between 1 and 1 + 2^-7: even (down)
        (one + 3 * 2.0 ** -8, 0x3F82),             # tie between 1 + 2^-7 and 1 + 2^-6: even (up)
        (one + 2.0 ** -8 + 2.0 ** -20, 0x3F81),    # just above the tie: up
        (-(one + 2.0 ** -8), 0xBF80),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (float(np.finfo(np.float32).max), 0x7F80),  # above the largest bf16: Inf
    ]
    v = np.array([c[0] for c in cases], np.float32)
    got = oracle.f32_to_bf16(v)
    assert got.tolist() == [c[1] for c in cases]


def test_f32_to_bf16_is_nearest_even_by_fractions():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(4000) * np.exp2(rng.integers(-130, 120, 4000))).astype(np.float32)
    got = oracle.f32_to_bf16(v)
    for x, b in zip(v, got):
        cand = [int(b) - 1, int(b), int(b) + 1]
        vals = [exact(synth.bf16_bits_to_f32(np.array([c & 0xFFFF], np.uint16))[0]) for c in cand]
        d = [abs(val - exact(x)) for val in vals]
        assert d[1] <= d[0] and d[1] <= d[2]
        if d[1] in (d[0], d[2]):
            assert b % 2 == 0  # a tie goes to the even pattern
    nan = oracle.f32_to_bf16(np.array([np.nan], np.float32))
    assert np.isnan(synth.bf16_bits_to_f32(nan)[0])
