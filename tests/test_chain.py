"""GPU parity of the decode chain (bitnet_decode_chain_*) with real data flow
between phases: a phase reads, as its input, bytes that an earlier phase of
the same run writes (bf16 and binary32 links), the subln norm and the gated
ReLU^2 pair inside the chain, several tokens, phases most CTAs own no rows
of, and the 30-layer decode step exactly as the benchmark builds it.  Every
output is compared bit for bit with the oracle run on the same host inputs,
phase after phase (the oracle feeds each phase the oracle's own output of the
phase before; no GPU value enters it)."""
import numpy as np
import pytest
import torch

import oracle
import bitlinear_bitnet_linear_03_b300 as bn
from bitlinear_bitnet_linear_03_b300 import synth
from gpu_util import assert_bits_equal, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

EPS = np.float32(1e-5)


def bf16_host(t):
    return host(t.view(torch.int16)).view(np.uint16)


def packed(N, K, seed):
    """Host weights of a test matrix: absmean-quantised N(0, 0.02) weights."""
    Wq, ws, _ = oracle.quantize_weights(synth.weights_f32(N, K, seed=seed))
    return Wq, np.float32(ws)


def on_dev(Wq, ws):
    return dev(Wq), dev(np.array([ws], np.float32))


def poison(tensors):
    for t in tensors:
        if t.dtype == torch.bfloat16:
            t.view(torch.int16).fill_(0x7fc1)
        elif t.dtype == torch.float32:
            t.fill_(float("nan"))
        else:
            t.fill_(-7)


def run_twice(chain, outs, check):
    """Two runs of the chain (the second reuses the table: new run tags), each
    after poisoning every output, each checked against the oracle."""
    for run in range(2):
        poison(outs)
        bn.bitnet_decode_chain_run(chain)
        torch.cuda.synchronize()
        assert bn.bitnet_device_error() == 0
        check(run)


# ---------------------------------------------------------------- links
@pytest.mark.parametrize("M", [1, 2, 4])
def test_chain_bf16_link_carries_the_previous_output(M):
    """Phase 0 writes y0 as bf16; phase 1 reads exactly those bytes as its
    input; phase 2 reads phase 1's bf16 output."""
    H = 2560
    x = synth.tokens_bf16(M, H, seed=70 + M, outlier_frac=0.01)
    W = [packed(H, H, seed=700 + i) for i in range(3)]
    ys = [torch.empty((M, H), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    accs = [torch.empty((M, H), dtype=torch.int32, device="cuda") for _ in range(3)]
    xd = dev_bf16(x)
    phases = []
    for i in range(3):
        Wq, ws = on_dev(*W[i])
        phases.append({"x": xd if i == 0 else ys[i - 1],
                       "targets": [(Wq, ws, None, accs[i], ys[i])]})
    chain = bn.bitnet_decode_chain_build(phases)

    def check(run):
        cur = x
        for i in range(3):
            qx, sx = oracle.quantize_act_bf16(cur)
            y_o, acc_o = oracle.linear(W[i][0], W[i][1], qx, sx, H)
            yb = oracle.f32_to_bf16(y_o)
            assert_bits_equal(host(accs[i]), acc_o, f"run {run} phase {i} acc")
            assert_bits_equal(bf16_host(ys[i]), yb, f"run {run} phase {i} y_bf16")
            cur = yb
    run_twice(chain, ys + accs, check)


def test_chain_f32_link_and_mixed_outputs():
    """A binary32 output read as the next phase's binary32 input; the first
    phase also writes its other target in both forms."""
    M, K0, N0 = 1, 2560, 6912
    x = synth.tokens_bf16(M, K0, seed=81)
    Wa, Wb, Wc = packed(N0, K0, 801), packed(640, K0, 802), packed(K0, N0, 803)
    ya = torch.empty((M, N0), dtype=torch.float32, device="cuda")
    yb32 = torch.empty((M, 640), dtype=torch.float32, device="cuda")
    yb16 = torch.empty((M, 640), dtype=torch.bfloat16, device="cuda")
    yc = torch.empty((M, K0), dtype=torch.float32, device="cuda")
    xq1 = torch.empty((M, N0), dtype=torch.int8, device="cuda")
    xs1 = torch.empty(M, dtype=torch.float32, device="cuda")
    phases = [{"x": dev_bf16(x), "targets": [(*on_dev(*Wa), ya), (*on_dev(*Wb), yb32, None, yb16)]},
              {"x_f32": ya, "targets": [(*on_dev(*Wc), yc)], "xq_out": xq1, "x_scale_out": xs1}]
    chain = bn.bitnet_decode_chain_build(phases)

    def check(run):
        qx, sx = oracle.quantize_act_bf16(x)
        ya_o, _ = oracle.linear(Wa[0], Wa[1], qx, sx, K0)
        yb_o, _ = oracle.linear(Wb[0], Wb[1], qx, sx, K0)
        assert_bits_equal(host(ya), ya_o, "ya")
        assert_bits_equal(host(yb32), yb_o, "yb")
        assert_bits_equal(bf16_host(yb16), oracle.f32_to_bf16(yb_o), "yb bf16")
        q1, s1 = oracle.quantize_act_f32(ya_o)
        assert_bits_equal(host(xq1), q1, "phase 1 codes")
        assert_bits_equal(host(xs1), s1, "phase 1 scale")
        yc_o, _ = oracle.linear(Wc[0], Wc[1], q1, s1, N0)
        assert_bits_equal(host(yc), yc_o, "yc")
    run_twice(chain, [ya, yb32, yb16, yc, xq1, xs1], check)


@pytest.mark.parametrize("M,K", [(1, 192), (3, 192), (1, 6912)])
def test_chain_stages_that_cross_target_boundaries(M, K):
    """Eight targets of very different sizes in one phase: with a few rows per
    CTA, many CTAs' stages hold rows of two targets (one stage per CTA where
    its share crosses one boundary, split where it would cross two); every
    output form of every target equals the oracle's."""
    Ns = [3, 1, 7, 2, 40, 5, 1, 300]
    x = synth.tokens_bf16(M, K, seed=90 + M, outlier_frac=0.01)
    W = [packed(N, K, seed=900 + i) for i, N in enumerate(Ns)]
    ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for N in Ns]
    accs = [torch.empty((M, N), dtype=torch.int32, device="cuda") for N in Ns]
    yb = torch.empty((M, 300), dtype=torch.bfloat16, device="cuda")
    targets = [(*on_dev(*W[i]), ys[i], accs[i]) + ((yb,) if i == 7 else ())
               for i in range(len(Ns))]
    phases = [{"x": dev_bf16(x), "targets": targets}]
    chain = bn.bitnet_decode_chain_build(phases)

    def check(run):
        qx, sx = oracle.quantize_act_bf16(x)
        for i in range(len(Ns)):
            y_o, acc_o = oracle.linear(W[i][0], W[i][1], qx, sx, K)
            assert_bits_equal(host(accs[i]), acc_o, f"run {run} target {i} acc")
            assert_bits_equal(host(ys[i]), y_o, f"run {run} target {i} y")
            if i == 7:
                assert_bits_equal(bf16_host(yb), oracle.f32_to_bf16(y_o), f"run {run} bf16")
    run_twice(chain, ys + accs + [yb], check)


# ---------------------------------------------------------------- norm + gated pair
@pytest.mark.parametrize("M,seed", [(1, 0), (1, 1), (2, 2), (4, 3)])
def test_chain_ffn_block_matches_oracle_ffn(M, seed):
    """subln norm + quantisation + gated up/gate pair (h = relu(gate)^2 * up)
    + binary32 link + down, as two chain phases: every intermediate equals the
    oracle's fused FFN."""
    H, F = 2560, 6912
    x = synth.tokens_bf16(M, H, seed=seed * 10 + 4)
    g = synth.gain_random(H, seed)
    up, gate, down = packed(F, H, seed * 10 + 1), packed(F, H, seed * 10 + 2), packed(H, F, seed * 10 + 3)
    t = lambda shape, dt: torch.empty(shape, dtype=dt, device="cuda")
    u, v, h = t((M, F), torch.float32), t((M, F), torch.float32), t((M, F), torch.float32)
    xq, sx = t((M, H), torch.int8), t(M, torch.float32)
    hq, sh = t((M, F), torch.int8), t(M, torch.float32)
    acc_d, y = t((M, H), torch.int32), t((M, H), torch.float32)
    phases = [{"x": dev_bf16(x), "norm_gain": dev(g), "norm_eps": float(EPS), "gated": True,
               "h": h, "targets": [(*on_dev(*up), u), (*on_dev(*gate), v)],
               "xq_out": xq, "x_scale_out": sx},
              {"x_f32": h, "targets": [(*on_dev(*down), y, acc_d)], "xq_out": hq,
               "x_scale_out": sh}]
    chain = bn.bitnet_decode_chain_build(phases)
    want = oracle.ffn(x, g, EPS, up[0], up[1], gate[0], gate[1], down[0], down[1])

    def check(run):
        got = dict(xq=xq, sx=sx, u=u, v=v, h=h, hq=hq, sh=sh, acc_down=acc_d, y=y)
        for k, tns in got.items():
            assert_bits_equal(host(tns), want[k], f"run {run} {k}")
    run_twice(chain, [u, v, h, xq, sx, hq, sh, acc_d, y], check)


def test_chain_norm_on_a_linked_input_and_special_rows():
    """subln on a bf16 link (the attention-side norm before O), with a row of
    equal values, an all-zero row and a row whose squares need the exact sum."""
    M, H = 3, 2560
    x = synth.tokens_bf16(M, H, seed=91)
    W0, W1 = packed(H, H, 901), packed(H, H, 902)
    g = synth.gain_random(H, 7)
    # the first phase's weights are chosen so its output rows stay generic;
    # the special rows go straight into a phase with a norm on an external input
    xs = x.copy()
    xs[1, :] = 0
    row = np.zeros(H, np.float32)
    row[3], row[20], row[41], row[63] = 1490944.0, 256.0, 256.0, 2.0 ** -20
    xs[2] = synth.f32_to_bf16_bits(row[None, :])[0]
    y0 = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    y1 = torch.empty((M, H), dtype=torch.float32, device="cuda")
    y2 = torch.empty((M, H), dtype=torch.float32, device="cuda")
    phases = [{"x": dev_bf16(x), "targets": [(*on_dev(*W0), None, None, y0)]},
              {"x": y0, "norm_gain": dev(g), "norm_eps": float(EPS),
               "targets": [(*on_dev(*W1), y1)]},
              {"x": dev_bf16(xs), "norm_gain": dev(g), "norm_eps": float(EPS),
               "targets": [(*on_dev(*W1), y2)]}]
    chain = bn.bitnet_decode_chain_build(phases)

    def check(run):
        qx, sx = oracle.quantize_act_bf16(x)
        y0_o = oracle.f32_to_bf16(oracle.linear(W0[0], W0[1], qx, sx, H)[0])
        assert_bits_equal(bf16_host(y0), y0_o, "y0")
        for src, out, what in ((y0_o, y1, "y1"), (xs, y2, "y2")):
            n, _ = oracle.rmsnorm_bf16(src, g, EPS)
            q, s = oracle.quantize_act_f32(n)
            assert_bits_equal(host(out), oracle.linear(W1[0], W1[1], q, s, H)[0], what)
    run_twice(chain, [y0, y1, y2], check)


def special_norm_rows(H):
    """Rows for the chain's exact sum of squares: a NaN, an infinity, a value
    whose square overflows binary32, subnormal bf16 values, and warps of very
    different magnitudes (each warp anchors its own partial sum)."""
    rows = synth.bf16_bits_to_f32(synth.tokens_bf16(6, H, seed=95)).copy()
    rows[0, 17] = np.nan
    rows[1, 900] = np.inf
    rows[2, 5] = 3.0e20
    rows[3, :] = 0.0
    rows[3, ::7] = 2.0 ** -130
    rows[4, : H // 2] *= 2.0 ** 20          # first half large, second half small
    rows[4, H // 2:] *= 2.0 ** -12
    rows[5, ::2] = 0.0
    return synth.f32_to_bf16_bits(rows)


@pytest.mark.parametrize("row", range(6))
def test_chain_norm_special_rows_one_token(row):
    H = 2560
    x = special_norm_rows(H)[row:row + 1]
    g = synth.gain_random(H, 11)
    W = packed(320, H, 950)
    y = torch.empty((1, 320), dtype=torch.float32, device="cuda")
    xq = torch.empty((1, H), dtype=torch.int8, device="cuda")
    sx = torch.empty(1, dtype=torch.float32, device="cuda")
    chain = bn.bitnet_decode_chain_build(
        [{"x": dev_bf16(x), "norm_gain": dev(g), "norm_eps": float(EPS),
          "targets": [(*on_dev(*W), y)], "xq_out": xq, "x_scale_out": sx}])

    def check(run):
        n, _ = oracle.rmsnorm_bf16(x, g, EPS)
        q, s = oracle.quantize_act_f32(n)
        assert_bits_equal(host(sx), s, f"run {run} scale")
        assert_bits_equal(host(xq), q, f"run {run} codes")
        assert_bits_equal(host(y), oracle.linear(W[0], W[1], q, s, H)[0], f"run {run} y")
    run_twice(chain, [y, xq, sx], check)


def test_chain_norm_special_rows_four_tokens():
    H = 2560
    x = special_norm_rows(H)[[0, 2, 3, 4]]
    g = synth.gain_random(H, 12)
    W = packed(320, H, 951)
    y = torch.empty((4, 320), dtype=torch.float32, device="cuda")
    xq = torch.empty((4, H), dtype=torch.int8, device="cuda")
    sx = torch.empty(4, dtype=torch.float32, device="cuda")
    chain = bn.bitnet_decode_chain_build(
        [{"x": dev_bf16(x), "norm_gain": dev(g), "norm_eps": float(EPS),
          "targets": [(*on_dev(*W), y)], "xq_out": xq, "x_scale_out": sx}])

    def check(run):
        n, _ = oracle.rmsnorm_bf16(x, g, EPS)
        q, s = oracle.quantize_act_f32(n)
        assert_bits_equal(host(sx), s, f"run {run} scale")
        assert_bits_equal(host(xq), q, f"run {run} codes")
        assert_bits_equal(host(y), oracle.linear(W[0], W[1], q, s, H)[0], f"run {run} y")
    run_twice(chain, [y, xq, sx], check)


def test_chain_links_through_phases_most_ctas_skip():
    """Small phases (64 rows: most CTAs own none and skip the phase without
    reading its input) linked to each other and to large ones."""
    M = 1
    spec = [(2560, 64), (64, 64), (64, 2560), (2560, 128), (128, 64)]
    x = synth.tokens_bf16(M, 2560, seed=93)
    W = [packed(N, K, 930 + i) for i, (K, N) in enumerate(spec)]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _, N in spec]
    phases = [{"x": dev_bf16(x) if i == 0 else ys[i - 1],
               "targets": [(*on_dev(*W[i]), None, None, ys[i])]} for i in range(len(spec))]
    chain = bn.bitnet_decode_chain_build(phases)

    def check(run):
        cur = x
        for i, (K, N) in enumerate(spec):
            qx, sx = oracle.quantize_act_bf16(cur)
            cur = oracle.f32_to_bf16(oracle.linear(W[i][0], W[i][1], qx, sx, K)[0])
            assert_bits_equal(bf16_host(ys[i]), cur, f"run {run} phase {i}")
    run_twice(chain, ys, check)


def test_chain_alias_is_rejected_before_launch():
    M, H = 1, 2560
    W = on_dev(*packed(H, H, 950))
    y = torch.empty((M, H), dtype=torch.float32, device="cuda")
    yb = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    x = dev_bf16(synth.tokens_bf16(M, H, seed=95))
    with pytest.raises(bn.BitnetError) as e:   # output over an earlier phase's output
        bn.bitnet_decode_chain_build([{"x": x, "targets": [(*W, y)]},
                                      {"x": x, "targets": [(*W, y)]}])
    assert e.value.status == 7
    with pytest.raises(bn.BitnetError) as e:   # input written later in the chain
        bn.bitnet_decode_chain_build([{"x": yb, "targets": [(*W, y)]},
                                      {"x": x, "targets": [(*W, None, None, yb)]}])
    assert e.value.status == 7


# ---------------------------------------------------------------- the decode step
def oracle_decode_step(host_w, x0, g_attn, g_ffn, layers):
    """The decode step's data flow in the oracle: per layer QKV of the layer
    input; O of the subln-normalised Q output (bf16); up/gate of the
    subln-normalised O output (bf16), gated; down of h; its bf16 output is the
    next layer's input."""
    out = []
    x = x0
    H = x0.shape[1]
    for li in range(layers):
        W = host_w[li]
        q, s = oracle.quantize_act_bf16(x)
        Q = oracle.f32_to_bf16(oracle.linear(*W["q"], q, s, H)[0])
        Kc = oracle.linear(*W["k"], q, s, H)[0]
        Vc = oracle.linear(*W["v"], q, s, H)[0]
        n, _ = oracle.rmsnorm_bf16(Q, g_attn[li], EPS)
        q, s = oracle.quantize_act_f32(n)
        O = oracle.f32_to_bf16(oracle.linear(*W["o"], q, s, H)[0])
        n, _ = oracle.rmsnorm_bf16(O, g_ffn[li], EPS)
        q, s = oracle.quantize_act_f32(n)
        u = oracle.linear(*W["up"], q, s, H, threads=oracle.default_threads())[0]
        v = oracle.linear(*W["gate"], q, s, H, threads=oracle.default_threads())[0]
        h = oracle.relu2_mul(u, v)
        q, s = oracle.quantize_act_f32(h)
        F = h.shape[1]
        Y = oracle.f32_to_bf16(oracle.linear(*W["down"], q, s, F,
                                             threads=oracle.default_threads())[0])
        out.append(dict(q=Q, k=Kc, v=Vc, o=O, h=h, y=Y))
        x = Y
    return out


def check_decode_step(layers, dims, seed):
    """The benchmark's decode-step chain (same builder, shapes, links, norms
    and gated pairs) for `layers` layers of the model dims (hidden, FFN, K/V),
    with host-made ternary weights: every output of every phase equals the
    oracle's, over two runs."""
    import bench
    H = dims[0]
    host_w, dev_w = [], []
    for li in range(layers):
        Lh, Ld = {}, {}
        for j, (name, N, K, _) in enumerate(bench.layer_shapes(dims)):
            q = synth.ternary_codes(N, K, seed=seed + li * 16 + j)
            Wq, ws = oracle.pack(q), synth.weight_scale(seed + li * 16 + j)
            Lh[name] = (Wq, ws)
            Ld[name] = on_dev(Wq, ws)
            del q
        host_w.append(Lh)
        dev_w.append(Ld)
    x0 = synth.tokens_bf16(1, H, seed=seed + 77)
    g_attn = [synth.gain_random(H, seed + 300 + li) for li in range(layers)]
    g_ffn = [synth.gain_random(H, seed + 600 + li) for li in range(layers)]
    step = bench.DecodeStep(layers, weights=dev_w, x0=dev_bf16(x0),
                            gains=([dev(g) for g in g_attn], [dev(g) for g in g_ffn]), dims=dims)
    step.build_chain()
    want = oracle_decode_step(host_w, x0, g_attn, g_ffn, layers)
    for run in range(2):
        poison(step.output_tensors())
        step.step()
        torch.cuda.synchronize()
        assert bn.bitnet_device_error() == 0
        for li in range(layers):
            got = step.layer_outputs(li)
            for k, w in want[li].items():
                g = got[k]
                g = bf16_host(g) if g.dtype == torch.bfloat16 else host(g)
                assert_bits_equal(g, w, f"run {run} layer {li} {k}")


def test_decode_step_30_layers_as_benchmarked_matches_oracle():
    """The benchmarked 2B-class step: 30 layers, 120 phases."""
    import bench
    check_decode_step(30, bench.DIMS_2B, 5000)


def test_decode_step_8b_class_layers_match_oracle():
    """Two layers (8 phases) of the 8B-class step: hidden 4096, FFN 14336,
    K/V 1024; the down phase reads K = 14336 inputs, more than a CTA's
    registers hold at one token."""
    import bench
    check_decode_step(2, bench.DIMS_8B, 9000)


@pytest.mark.parametrize("K", [2560, 16384])
def test_chain_norm_rows_beyond_the_128_bit_window(K):
    """Rows whose squares span more than 2^88 (values 2^50 and 2^-30) take the
    five-limb exact sum; K = 16384 also exercises the inputs beyond those a
    thread keeps in registers.  Every row must equal the oracle's subln."""
    M = 2
    x = synth.tokens_bf16(M, K, seed=97)
    row = synth.bf16_bits_to_f32(x[1:2]).copy()
    row[0, 11], row[0, K - 3] = 2.0 ** 50, 2.0 ** -30
    x[1] = synth.f32_to_bf16_bits(row)[0]
    g = synth.gain_random(K, 9)
    W = packed(320, K, 970)
    y = torch.empty((M, 320), dtype=torch.float32, device="cuda")
    xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    phases = [{"x": dev_bf16(x), "norm_gain": dev(g), "norm_eps": float(EPS),
               "targets": [(*on_dev(*W), y)], "xq_out": xq, "x_scale_out": sx}]
    chain = bn.bitnet_decode_chain_build(phases)

    def check(run):
        n, _ = oracle.rmsnorm_bf16(x, g, EPS)
        q, s = oracle.quantize_act_f32(n)
        assert_bits_equal(host(sx), s, f"run {run} scale")
        assert_bits_equal(host(xq), q, f"run {run} codes")
        assert_bits_equal(host(y), oracle.linear(W[0], W[1], q, s, K)[0], f"run {run} y")
    run_twice(chain, [y, xq, sx], check)
