"""bitnet_quantize_weights_noalloc: the allocation-free weight quantisation.

It serves callers that cannot allocate device memory (a plugin inside a
framework that owns the device memory pool, a latency-critical path where
cudaMalloc is not allowed).  Its scratch is a fixed array inside the library,
shared by every call.  This test calls it through the C ABI twice in a row, on
two different matrices, and requires each result to equal that of
bitnet_quantize_weights (bit for bit: packed bytes and the scale).  The file
is named to be collected last, so a run that stops at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import bitlinear_bitnet_linear_03_b300 as bn
from bitlinear_bitnet_linear_03_b300 import synth

pytestmark = pytest.mark.gpu


def _noalloc_via_abi(W):
    N, K = W.shape
    Wq = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
    ws = torch.empty(1, dtype=torch.float32, device="cuda")
    st = bn.lib().bitnet_quantize_weights_noalloc(
        ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_void_p(Wq.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, bn.lib().bitnet_status_string(st)
    torch.cuda.synchronize()
    return Wq.cpu().numpy(), ws.cpu().numpy()


def _with_workspace(W):
    Wq, ws = bn.bitnet_quantize_weights(W)
    torch.cuda.synchronize()
    return Wq.cpu().numpy(), ws.cpu().numpy()


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    # A large matrix (all 592 scratch rows in use), then a small one that uses
    # only part of the scratch the first call left behind.
    first = torch.from_numpy(synth.weights_f32(6912, 2560, seed=101)).cuda()
    second = torch.from_numpy(synth.weights_f32(3, 192, seed=102)).cuda()
    got1 = _noalloc_via_abi(first)
    got2 = _noalloc_via_abi(second)
    want1 = _with_workspace(first)
    want2 = _with_workspace(second)
    for got, want in ((got1, want1), (got2, want2)):
        assert (got[0] == want[0]).all()
        assert got[1].view(np.uint32)[0] == want[1].view(np.uint32)[0]


def test_noalloc_rejects_unsupported_sizes():
    W = torch.zeros((2, 96), dtype=torch.float32, device="cuda")
    Wq = torch.empty((2, 24), dtype=torch.uint8, device="cuda")
    ws = torch.empty(1, dtype=torch.float32, device="cuda")
    st = bn.lib().bitnet_quantize_weights_noalloc(
        ctypes.c_void_p(W.data_ptr()), 2, 96, ctypes.c_void_p(Wq.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), None)
    assert st == 2  # K not a multiple of 64
