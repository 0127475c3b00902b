"""BitLinear CPU oracle — TEST INFRASTRUCTURE, not part of the product.

Thin numpy wrappers over liboracle.so (oracle.cpp).  Only tests/, the smoke
check in __graft_entry__ and the CPU-baseline leg of bench.py may import this
package; the CUDA library never does, and this package never imports the
CUDA library.  See oracle.h for the page passages each function follows.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = os.environ.get("BITNET_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        F = ctypes.c_float
        INT = ctypes.c_int
        sig = {
            "oracle_absmean": (F, [P, I64]),
            "oracle_ternarize": (None, [P, I64, I64, F, P, P]),
            "oracle_pack": (None, [P, I64, I64, P]),
            "oracle_unpack": (INT, [P, I64, I64, P]),
            "oracle_quantize_act_bf16": (None, [P, I64, I64, P, P]),
            "oracle_quantize_act_f32": (None, [P, I64, I64, P, P]),
            "oracle_linear_acc": (None, [P, P, I64, I64, I64, P, INT]),
            "oracle_rescale": (None, [P, P, F, I64, I64, P]),
            "oracle_linear": (INT, [P, F, P, P, I64, I64, I64, P, P, INT]),
            "oracle_rmsnorm_bf16": (None, [P, P, F, I64, I64, P, P]),
            "oracle_relu2_mul": (None, [P, P, I64, P]),
            "oracle_f32_to_bf16": (None, [P, I64, P]),
            "oracle_ffn": (INT, [P, P, F, P, F, P, F, P, F, I64, I64, I64, P,
                                 P, P, P, P, P, P, P, P, INT]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def default_threads() -> int:
    return os.cpu_count() or 1


def absmean(W) -> np.float32:
    W = _c(W, np.float32)
    return np.float32(lib().oracle_absmean(_p(W), W.size))


def ternarize(W, gamma):
    W = _c(W, np.float32)
    N, K = W.shape
    q = np.empty((N, K), np.int8)
    ws = np.zeros(1, np.float32)
    lib().oracle_ternarize(_p(W), N, K, float(gamma), _p(q), _p(ws))
    return q, np.float32(ws[0])


def pack(q):
    q = _c(q, np.int8)
    N, K = q.shape
    assert K % 64 == 0
    Wq = np.empty((N, K // 4), np.uint8)
    lib().oracle_pack(_p(q), N, K, _p(Wq))
    return Wq


def unpack(Wq, K):
    Wq = _c(Wq, np.uint8)
    N = Wq.shape[0]
    q = np.empty((N, K), np.int8)
    if lib().oracle_unpack(_p(Wq), N, K, _p(q)) != 0:
        raise ValueError("packed weights hold the unused 2-bit code 3")
    return q


def quantize_weights(W):
    """absmean -> ternarize -> pack.  Returns (Wq [N,K/4] u8, w_scale, q)."""
    gamma = absmean(W)
    q, ws = ternarize(W, gamma)
    return pack(q), ws, q


def quantize_act_bf16(x_bits):
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    q = np.empty((M, K), np.int8)
    sx = np.empty(M, np.float32)
    lib().oracle_quantize_act_bf16(_p(x_bits), M, K, _p(q), _p(sx))
    return q, sx


def quantize_act_f32(x):
    x = _c(x, np.float32)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    sx = np.empty(M, np.float32)
    lib().oracle_quantize_act_f32(_p(x), M, K, _p(q), _p(sx))
    return q, sx


def linear_acc(qw, qx, threads=1):
    qw = _c(qw, np.int8)
    qx = _c(qx, np.int8)
    N, K = qw.shape
    M, K2 = qx.shape
    assert K == K2
    acc = np.empty((M, N), np.int32)
    lib().oracle_linear_acc(_p(qw), _p(qx), M, N, K, _p(acc), int(threads))
    return acc


def rescale(acc, sx, w_scale):
    acc = _c(acc, np.int32)
    sx = _c(sx, np.float32)
    M, N = acc.shape
    y = np.empty((M, N), np.float32)
    lib().oracle_rescale(_p(acc), _p(sx), float(w_scale), M, N, _p(y))
    return y


def linear(Wq, w_scale, qx, sx, K, threads=1):
    """Packed ternary W [N,K/4] x int8 qx [M,K] -> (y f32 [M,N], acc i32)."""
    Wq = _c(Wq, np.uint8)
    qx = _c(qx, np.int8)
    sx = _c(sx, np.float32)
    N = Wq.shape[0]
    M = qx.shape[0]
    y = np.empty((M, N), np.float32)
    acc = np.empty((M, N), np.int32)
    rc = lib().oracle_linear(_p(Wq), float(w_scale), _p(qx), _p(sx), M, N, K,
                             _p(y), _p(acc), int(threads))
    if rc != 0:
        raise ValueError("packed weights hold the unused 2-bit code 3")
    return y, acc


def rmsnorm_bf16(x_bits, g, eps):
    x_bits = _c(x_bits, np.uint16)
    g = _c(g, np.float32)
    M, H = x_bits.shape
    n = np.empty((M, H), np.float32)
    r = np.empty(M, np.float32)
    lib().oracle_rmsnorm_bf16(_p(x_bits), _p(g), float(eps), M, H, _p(n), _p(r))
    return n, r


def relu2_mul(u, v):
    u = _c(u, np.float32)
    v = _c(v, np.float32)
    h = np.empty_like(u)
    lib().oracle_relu2_mul(_p(u), _p(v), u.size, _p(h))
    return h


def f32_to_bf16(v):
    """binary32 -> bf16 bit patterns (uint16), nearest, ties to even."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_f32_to_bf16(_p(v), v.size, _p(out))
    return out


def ffn(x_bits, g, eps, Wup, s_up, Wgate, s_gate, Wdown, s_down, threads=1):
    """Fused FFN; returns a dict with y and every intermediate stage."""
    x_bits = _c(x_bits, np.uint16)
    g = _c(g, np.float32)
    Wup, Wgate, Wdown = (_c(w, np.uint8) for w in (Wup, Wgate, Wdown))
    M, H = x_bits.shape
    F = Wup.shape[0]
    out = {
        "y": np.empty((M, H), np.float32),
        "xq": np.empty((M, H), np.int8),
        "sx": np.empty(M, np.float32),
        "u": np.empty((M, F), np.float32),
        "v": np.empty((M, F), np.float32),
        "h": np.empty((M, F), np.float32),
        "hq": np.empty((M, F), np.int8),
        "sh": np.empty(M, np.float32),
        "acc_down": np.empty((M, H), np.int32),
    }
    rc = lib().oracle_ffn(_p(x_bits), _p(g), float(eps), _p(Wup), float(s_up),
                          _p(Wgate), float(s_gate), _p(Wdown), float(s_down),
                          M, H, F, _p(out["y"]), _p(out["xq"]), _p(out["sx"]),
                          _p(out["u"]), _p(out["v"]), _p(out["h"]),
                          _p(out["hq"]), _p(out["sh"]), _p(out["acc_down"]),
                          int(threads))
    if rc != 0:
        raise ValueError("packed weights hold the unused 2-bit code 3")
    return out
