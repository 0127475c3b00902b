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
    assert L.bitnet_abi_version() == 2
    for s in range(8):
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
    """Workspace per path: none for decode (M <= 4); 2 bytes per activation
    (bf16, or two e4m3 digits) for the fused tensor-core path (M <= 256)
    plus the split-K sums when the output has few tiles; for prefill the e4m3
    weights (1 byte each) and the activations' two e4m3 digits."""
    L = bn.lib()
    assert L.bitnet_linear_workspace(1, 28672, 8192) == 0
    assert L.bitnet_linear_workspace(4, 2560, 6912) == 0
    M, N, K = 64, 28672, 8192          # 112 tiles: no split
    w = L.bitnet_linear_workspace(M, N, K)
    assert M * K * 2 <= w < M * K * 2 + M * N * 4
    M, N, K = 64, 8192, 28672          # 32 tiles: K split, fp32 sums + tile counters
    assert L.bitnet_linear_workspace(M, N, K) >= M * K * 2 + M * N * 4 + 32 * 4
    M, N, K = 4096, 6912, 2560         # prefill: expanded weights and activation digits
    assert L.bitnet_linear_workspace(M, N, K) >= N * K + M * K * 2


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first
MIS = 0x10004   # 4-byte aligned only


def p(v):
    return ctypes.c_void_p(v)


def test_argument_errors_are_reported_before_launch():
    L = bn.lib()
    # NULL pointers
    assert L.bitnet_linear(None, p(FAKE), p(FAKE), p(FAKE), 1, 64, 64, p(FAKE), None, None, None,
                           0, None) == 1
    # neither output form requested
    assert L.bitnet_linear(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1, 64, 64, None, None, None, None,
                           0, None) == 1
    assert L.bitnet_quantize_act(None, 1, 64, p(FAKE), p(FAKE), None) == 1
    assert L.bitnet_quantize_weights(p(FAKE), 1, 64, None, p(FAKE), p(FAKE), 1 << 20, None) == 1
    # shapes: K not a multiple of 64, non-positive sizes, K too large
    assert L.bitnet_linear(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1, 64, 100, p(FAKE), None, None,
                           None, 0, None) == 2
    assert L.bitnet_linear(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 0, 64, 64, p(FAKE), None, None,
                           None, 0, None) == 2
    assert L.bitnet_quantize_act(p(FAKE), 1, 65536 + 64, p(FAKE), p(FAKE), None) == 2
    assert L.bitnet_quantize_weights(p(FAKE), 3, 96, p(FAKE), p(FAKE), p(FAKE), 1 << 20,
                                     None) == 2
    # misaligned pointers
    assert L.bitnet_linear(p(MIS), p(FAKE), p(FAKE), p(FAKE), 1, 64, 64, p(FAKE), None, None,
                           None, 0, None) == 3
    assert L.bitnet_linear(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1, 64, 64, None, p(MIS), None,
                           None, 0, None) == 3
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


def test_lut_entry_checks_its_arguments():
    L = bn.lib()
    args = [p(FAKE)] * 4
    assert L.bitnet_linear_lut(*args, 64, 64, None, None, 0, None) == 1          # y
    assert L.bitnet_linear_lut(*args, 64, 12288 + 64, p(FAKE), None, 0, None) == 2  # K too large
    assert L.bitnet_linear_lut(*args, 64, 100, p(FAKE), None, 0, None) == 2        # K % 64
    assert L.bitnet_linear_lut(*args, 0, 64, p(FAKE), None, 1, None) == 2          # N
    assert L.bitnet_linear_lut(*args, 64, 64, p(FAKE), None, 2, None) == 2         # variant
    assert L.bitnet_linear_lut(p(MIS), *args[1:], 64, 64, p(FAKE), None, 0, None) == 3


class FakeMem:
    """Distinct fake device addresses (never dereferenced: every check below
    fails, or passes, on the host before anything touches a device)."""

    def __init__(self):
        self.next = 0x1000000

    def __call__(self, nbytes):
        a = self.next
        self.next += (nbytes + 4095) // 4096 * 4096 + 4096
        return a


def _chain_phase(mem, K=2560, Ns=(64,), M=1, x=None, x_f32=None, gated=False, h=None, ys=None,
                 ybs=None, norm=False, bf16_out=False):
    count = len(Ns)
    ys = ys or [None] * count
    ybs = ybs or [None] * count
    tg = (_lib.LinearTarget * count)()
    for i, N in enumerate(Ns):
        y = ys[i] if ys[i] is not None else (None if bf16_out else mem(4 * M * N))
        yb = ybs[i] if ybs[i] is not None else (mem(2 * M * N) if bf16_out else None)
        tg[i] = _lib.LinearTarget(mem(N * K // 4), mem(16), N, y, None, yb)
    if x is None and x_f32 is None:
        x = mem(2 * M * K)
    ph = _lib.DecodePhase(x, K, ctypes.cast(tg, ctypes.c_void_p), count, 1 if gated else 0, x_f32,
                          mem(4 * K) if norm else None, 1e-5, h, None, None)
    return ph, tg


def _chain_status(L, phases, M=1, table=0x100000, nbytes=None):
    arr = (_lib.DecodePhase * len(phases))(*[ph for ph, _ in phases])
    chain = _lib.DecodeChain()
    n = len(phases)
    need = L.bitnet_decode_chain_bytes(arr, n, M)
    return L.bitnet_decode_chain_build(arr, n, M, p(table) if table else None,
                                       need if nbytes is None else nbytes,
                                       ctypes.byref(chain)), need


def test_decode_chain_arguments_are_checked_on_the_host():
    L = bn.lib()
    mem = FakeMem()
    ok = [_chain_phase(mem), _chain_phase(mem, K=6912, Ns=(64, 128))]
    # a valid description passes the host checks and then stops at the missing
    # table (no device is touched)
    st, need = _chain_status(L, ok, table=0)
    assert need > 0 and st == 1
    assert L.bitnet_decode_chain_build(None, 1, 1, p(0x100000), need, None) == 1
    assert _chain_status(L, ok, M=5)[0] == 2                      # M > 4
    assert _chain_status(L, ok, M=0)[0] == 2
    assert _chain_status(L, ok, table=0x100080)[0] == 3          # table alignment
    assert _chain_status(L, ok, nbytes=need - 1)[0] == 4         # table too small
    assert _chain_status(L, [_chain_phase(mem, Ns=(64,) * 9)])[0] == 2   # > 8 targets
    assert _chain_status(L, [_chain_phase(mem, K=100)])[0] == 2          # K % 64 != 0
    assert _chain_status(L, [_chain_phase(mem, K=65536 * 2)])[0] == 2    # K too large
    assert _chain_status(L, [_chain_phase(mem, Ns=(0,))])[0] == 2        # empty matrix
    assert _chain_status(L, [_chain_phase(mem, x=MIS)])[0] == 3          # x alignment
    assert _chain_status(L, [_chain_phase(mem, ys=[MIS])])[0] == 3       # y alignment
    both = _chain_phase(mem, x_f32=mem(4 * 2560))                        # x and x_f32 both
    both[0].x = mem(2 * 2560)
    assert _chain_status(L, [both])[0] == 2
    none = _chain_phase(mem)
    none[0].x = None
    assert _chain_status(L, [none])[0] == 1                              # no input
    assert _chain_status(L, [_chain_phase(mem, gated=True, Ns=(64, 64))])[0] == 1  # gated: no h
    h = mem(4 * 64)
    assert _chain_status(L, [_chain_phase(mem, gated=True, Ns=(64, 128), h=h)])[0] == 2
    assert _chain_status(L, [_chain_phase(mem, gated=True, Ns=(64,), h=h)])[0] == 2
    assert _chain_status(L, [_chain_phase(mem, x_f32=mem(4 * 2560), norm=True)])[0] == 2
    assert L.bitnet_decode_chain_run(None, None) == 1


def test_decode_chain_links_and_overlaps_are_checked_on_the_host():
    """A phase input that is exactly an earlier output is a link; any other
    overlap between an array the chain writes and any array it touches is
    BITNET_ERR_ALIAS."""
    L = bn.lib()
    mem = FakeMem()
    M, H = 1, 2560
    yb = mem(2 * M * H)
    p0 = _chain_phase(mem, Ns=(H,), ybs=[yb], bf16_out=True)
    p1 = _chain_phase(mem, x=yb, Ns=(H,), norm=True)                 # bf16 link, with norm
    st, need = _chain_status(L, [p0, p1], table=0)                   # valid: stops at the table
    assert need > 0 and st == 1
    # the link buffer lives in the table: a linked chain needs more table
    p1b = _chain_phase(mem, Ns=(H,))
    assert _chain_status(L, [p0, p1b], table=0)[1] < need
    # a gated phase's h read as a binary32 link
    h = mem(4 * M * 6912)
    pg = _chain_phase(mem, Ns=(6912, 6912), gated=True, h=h)
    pd = _chain_phase(mem, K=6912, x_f32=h, Ns=(H,))
    assert _chain_status(L, [pg, pd], table=0)[0] == 1
    # overlaps that are not links
    assert _chain_status(L, [p1, p0])[0] == 7                        # reads a LATER output
    part = _chain_phase(mem, x=yb + 16, K=2496, Ns=(H,))             # inside an output, not equal
    assert _chain_status(L, [p0, part])[0] == 7
    y0 = mem(4 * M * H)
    q0 = _chain_phase(mem, Ns=(H,), ys=[y0])
    q1 = _chain_phase(mem, Ns=(H,), ys=[y0 + 64])                    # two outputs overlap
    assert _chain_status(L, [q0, q1])[0] == 7
    q2 = _chain_phase(mem, x=y0, Ns=(H,))                            # bf16 x over a binary32 y
    assert _chain_status(L, [q0, q2])[0] == 7
    r0 = _chain_phase(mem, Ns=(H,))
    r0[1][0].y = r0[1][0].Wq                                         # output over the weights
    assert _chain_status(L, [r0])[0] == 7
    self_link = _chain_phase(mem, Ns=(H,), ybs=[yb], bf16_out=True)
    self_link[0].x = yb                                              # reads its own output
    assert _chain_status(L, [self_link])[0] == 7


def test_no_device_reports_unsupported_or_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = bn.lib()
    st = L.bitnet_quantize_act(p(FAKE), 1, 64, p(FAKE), p(FAKE), None)
    assert st in (5, 6)
