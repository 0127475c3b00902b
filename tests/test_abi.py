"""The C-ABI library: it loads, exports every symbol the header declares, and
rejects bad arguments on the host before touching a GPU.  CPU only."""
import ctypes
import os
import re
import subprocess

import pytest

import bitlinear_bitnet_linear_03_b300 as bn
from bitlinear_bitnet_linear_03_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(bitnet_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("bitnet_quantize_weights", "bitnet_quantize_act", "bitnet_linear", "bitnet_ffn"):
        assert fn in names


def test_library_exports_every_declared_symbol():
    L = bn.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", bn.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert declared_functions() <= exported


def test_binding_covers_every_symbol():
    assert declared_functions() == set(_lib.SIGNATURES)


def test_status_strings_and_version():
    L = bn.lib()
    assert L.bitnet_abi_version() == 1
    for s in range(7):
        assert L.bitnet_status_string(s)
    assert L.bitnet_status_string(99) == b"unknown status"


def test_workspace_queries():
    L = bn.lib()
    assert L.bitnet_quantize_weights_workspace(2560, 2560) > 0
    assert L.bitnet_quantize_weights_workspace(0, 64) == 0
    assert L.bitnet_linear_workspace(0, 1, 64) == 0
    # ffn workspace holds at least xq, u, v and hq
    M, H, F = 4, 2560, 6912
    assert L.bitnet_ffn_workspace(M, H, F) >= M * H + 2 * 4 * M * F + M * F


def test_linear_workspace_follows_the_dispatch():
    """Workspace per path: none for decode (M <= 4), the bf16 activations for
    the fused tensor-core path (16 <= M <= 256) plus the split-K sums when the
    output has few tiles, the bf16 weights and activations for prefill."""
    L = bn.lib()
    assert L.bitnet_linear_workspace(1, 28672, 8192) == 0
    assert L.bitnet_linear_workspace(4, 2560, 6912) == 0
    M, N, K = 64, 28672, 8192          # 112 tiles: no split
    w = L.bitnet_linear_workspace(M, N, K)
    assert M * K * 2 <= w < M * K * 2 + M * N * 4
    M, N, K = 64, 8192, 28672          # 32 tiles: K split, fp32 sums + tile counters
    assert L.bitnet_linear_workspace(M, N, K) >= M * K * 2 + M * N * 4 + 32 * 4
    M, N, K = 4096, 6912, 2560         # prefill: expanded weights and activations
    assert L.bitnet_linear_workspace(M, N, K) >= N * K * 2 + M * K * 2


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first
MIS = 0x10004   # 4-byte aligned only


def p(v):
    return ctypes.c_void_p(v)


def test_argument_errors_are_reported_before_launch():
    L = bn.lib()
    # NULL pointers
    assert L.bitnet_linear(None, p(FAKE), p(FAKE), p(FAKE), 1, 64, 64, p(FAKE), None, None, 0,
                           None) == 1
    assert L.bitnet_quantize_act(None, 1, 64, p(FAKE), p(FAKE), None) == 1
    assert L.bitnet_quantize_weights(p(FAKE), 1, 64, None, p(FAKE), p(FAKE), 1 << 20, None) == 1
    # shapes: K not a multiple of 64, non-positive sizes, K too large
    assert L.bitnet_linear(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1, 64, 100, p(FAKE), None, None,
                           0, None) == 2
    assert L.bitnet_linear(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 0, 64, 64, p(FAKE), None, None, 0,
                           None) == 2
    assert L.bitnet_quantize_act(p(FAKE), 1, 65536 + 64, p(FAKE), p(FAKE), None) == 2
    assert L.bitnet_quantize_weights(p(FAKE), 3, 96, p(FAKE), p(FAKE), p(FAKE), 1 << 20,
                                     None) == 2
    # misaligned pointers
    assert L.bitnet_linear(p(MIS), p(FAKE), p(FAKE), p(FAKE), 1, 64, 64, p(FAKE), None, None, 0,
                           None) == 3
    assert L.bitnet_quantize_act(p(FAKE), 1, 64, p(MIS), p(FAKE), None) == 3
    # workspace too small
    need = L.bitnet_quantize_weights_workspace(64, 64)
    assert L.bitnet_quantize_weights(p(FAKE), 64, 64, p(FAKE), p(FAKE), p(FAKE), need - 1,
                                     None) == 4
    ffn_need = L.bitnet_ffn_workspace(1, 64, 64)
    args = [p(FAKE)] * 9
    assert L.bitnet_ffn(p(FAKE), p(FAKE), ctypes.c_float(1e-5), *args[:6], 1, 64, 64, p(FAKE),
                        None, p(FAKE), ffn_need - 1, None) == 4
    assert L.bitnet_ffn(p(FAKE), p(FAKE), ctypes.c_float(1e-5), *args[:6], 1, 64, 100, p(FAKE),
                        None, p(FAKE), ffn_need, None) == 2
    assert L.bitnet_device_error(None, None) == 1


def test_decode_chain_arguments_are_checked_on_the_host():
    L = bn.lib()
    TABLE = 0x100000  # 256-byte aligned, never dereferenced
    need = L.bitnet_decode_chain_bytes(2)
    assert L.bitnet_decode_chain_bytes(3) - need == need - L.bitnet_decode_chain_bytes(1) > 0

    def phase(x=FAKE, K=2560, count=1, N=64, y=FAKE):
        tg = (_lib.LinearTarget * max(count, 1))(
            *[_lib.LinearTarget(FAKE, FAKE, N, y, None) for _ in range(max(count, 1))])
        return _lib.DecodePhase(x, K, ctypes.cast(tg, ctypes.c_void_p), count), tg

    def build(phases, M=1, table=TABLE, nbytes=None):
        arr = (_lib.DecodePhase * len(phases))(*[ph for ph, _ in phases])
        chain = _lib.DecodeChain()
        n = len(phases)
        return L.bitnet_decode_chain_build(arr, n, M, p(table),
                                           L.bitnet_decode_chain_bytes(n) if nbytes is None
                                           else nbytes, ctypes.byref(chain))

    ok = [phase(), phase(K=6912, count=2)]
    assert L.bitnet_decode_chain_build(None, 1, 1, p(TABLE), need, None) == 1    # NULL
    assert build(ok, M=5) == 2                                                   # M > 4
    assert build(ok, M=0) == 2
    assert build(ok, table=TABLE + 128) == 3                                     # table alignment
    assert build(ok, nbytes=need - 1) == 4                                       # table too small
    assert build([phase(count=9)]) == 2                                          # > 8 targets
    assert build([phase(count=0)]) == 2
    assert build([phase(K=100)]) == 2                                            # K % 64 != 0
    assert build([phase(K=65536 * 2)]) == 2                                      # K too large
    assert build([phase(N=0)]) == 2                                              # empty matrix
    assert build([phase(x=MIS)]) == 3                                            # x alignment
    assert build([phase(y=MIS)]) == 3                                            # y alignment
    assert build([phase(x=0)]) == 1
    assert L.bitnet_decode_chain_run(None, None) == 1


def test_no_device_reports_unsupported_or_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = bn.lib()
    st = L.bitnet_quantize_act(p(FAKE), 1, 64, p(FAKE), p(FAKE), None)
    assert st in (5, 6)
