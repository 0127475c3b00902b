"""GPU parity of the lookup-table BitLinear ablation (bitnet_linear_lut) and
its dp4a control against the oracle: both variants must give the oracle's
accumulators and outputs bit for bit, including the extreme accumulators and
the largest K the tables fit."""
import numpy as np
import pytest
import torch

import oracle
import bitlinear_bitnet_linear_03_b300 as bn
from bitlinear_bitnet_linear_03_b300 import synth
from gpu_util import assert_bits_equal, dev, host

pytestmark = pytest.mark.gpu


def run_lut(Wq, ws, qx, sx, variant):
    N = Wq.shape[0]
    acc = torch.empty((1, N), dtype=torch.int32, device="cuda")
    y = bn.bitnet_linear_lut(dev(Wq), dev(np.array([ws], np.float32)), dev(qx),
                             dev(np.asarray(sx, np.float32).reshape(1)), variant=variant,
                             acc_out=acc)
    torch.cuda.synchronize()
    return host(y), host(acc)


@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("N,K", [(1, 64), (3, 192), (33, 640), (2560, 2560), (6912, 2560),
                                 (2560, 6912), (100, 12288), (28672, 8192)])
def test_lut_matches_oracle(variant, N, K):
    W = synth.weights_f32(N, K, seed=N + K)
    Wq, ws, _ = oracle.quantize_weights(W)
    qx, sx = oracle.quantize_act_bf16(synth.tokens_bf16(1, K, seed=K, outlier_frac=0.01))
    y, acc = run_lut(Wq, ws, qx, sx, variant)
    y_o, acc_o = oracle.linear(Wq, ws, qx, sx, K, threads=oracle.default_threads())
    assert_bits_equal(acc, acc_o, f"variant {variant} acc")
    assert_bits_equal(y, y_o, f"variant {variant} y")


@pytest.mark.parametrize("variant", [0, 1])
def test_lut_extreme_accumulators(variant):
    """x = -128 everywhere against rows of all -1 and all +1 codes: the table
    entries reach their extremes and acc = +-128 K."""
    K = 4096
    q = np.stack([np.full(K, -1, np.int8), np.full(K, 1, np.int8), np.zeros(K, np.int8)])
    Wq = oracle.pack(q)
    qx = np.full((1, K), -128, np.int8)
    y, acc = run_lut(Wq, np.float32(1.0), qx, np.array([1.0], np.float32), variant)
    assert acc.ravel().tolist() == [128 * K, -128 * K, 0]
    assert y.ravel().tolist() == [128.0 * K, -128.0 * K, 0.0]
