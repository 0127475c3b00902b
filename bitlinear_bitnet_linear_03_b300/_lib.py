"""ctypes binding over libbitnet_b300.so (include/bitnet_b300.h).

Argument marshalling only: every function here checks that it was handed
device tensors of the right dtype and shape, passes their pointers and the
current CUDA stream to the C function of the same name, and raises
BitnetError on a non-zero status.  No step of the computation runs in Python,
and there is no fallback: if the library is missing, loading it fails loudly.
"""
import ctypes
import os

import torch

from . import build as _build

BITNET_OK = 0
STATUS = {0: "BITNET_OK", 1: "BITNET_ERR_NULL", 2: "BITNET_ERR_SHAPE", 3: "BITNET_ERR_ALIGN",
          4: "BITNET_ERR_WORKSPACE", 5: "BITNET_ERR_UNSUPPORTED", 6: "BITNET_ERR_CUDA",
          7: "BITNET_ERR_ALIAS"}

# Every symbol the header declares, with its ctypes signature.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_INT = ctypes.c_int
_F = ctypes.c_float
SIGNATURES = {
    "bitnet_status_string": (ctypes.c_char_p, [_INT]),
    "bitnet_last_cuda_error": (_INT, []),
    "bitnet_abi_version": (_INT, []),
    "bitnet_device_error": (_INT, [_P, _P]),
    "bitnet_set_wait_limit": (None, [ctypes.c_longlong]),
    "bitnet_quantize_weights_workspace": (_SZ, [_I64, _I64]),
    "bitnet_quantize_weights": (_INT, [_P, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "bitnet_quantize_weights_noalloc": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "bitnet_quantize_act": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "bitnet_linear_workspace": (_SZ, [_I64, _I64, _I64]),
    "bitnet_linear": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "bitnet_linear_bf16": (_INT, [_P, _I64, _I64, _P, _INT, _P, _P, ctypes.c_uint, _P]),
    "bitnet_linear_lut": (_INT, [_P, _P, _P, _P, _I64, _I64, _P, _P, _INT, _P]),
    "bitnet_decode_chain_bytes": (_SZ, [_P, _INT, _I64]),
    "bitnet_decode_chain_build": (_INT, [_P, _INT, _I64, _P, _SZ, _P]),
    "bitnet_decode_chain_run": (_INT, [_P, _P]),
    "bitnet_ffn_workspace": (_SZ, [_I64, _I64, _I64]),
    "bitnet_ffn": (_INT, [_P, _P, _F, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _SZ,
                          _P]),
}


class BitnetError(RuntimeError):
    def __init__(self, fn, status, cuda_error=0):
        self.status = status
        msg = f"{fn}: {STATUS.get(status, status)} ({lib().bitnet_status_string(status).decode()})"
        if status == 6:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


class LinearTarget(ctypes.Structure):
    """bitnet_linear_target: one weight matrix of a grouped decode call."""
    _fields_ = [("Wq", _P), ("w_scale", _P), ("N", _I64), ("y", _P), ("acc_out", _P),
                ("y_bf16", _P)]


class DecodePhase(ctypes.Structure):
    """bitnet_decode_phase: one phase of a decode chain."""
    _fields_ = [("x", _P), ("K", _I64), ("targets", _P), ("count", _INT), ("flags", ctypes.c_uint),
                ("x_f32", _P), ("norm_gain", _P), ("norm_eps", _F), ("h", _P), ("xq_out", _P),
                ("x_scale_out", _P)]


class DecodeChain(ctypes.Structure):
    """bitnet_decode_chain: filled by bitnet_decode_chain_build."""
    _fields_ = [("table", _P), ("M", _I64), ("nphases", _INT), ("cfg", _INT * 12)]


class FfnDebug(ctypes.Structure):
    """bitnet_ffn_debug: optional destinations for the FFN's intermediates."""
    _fields_ = [("xq", _P), ("sx", _P), ("u", _P), ("v", _P), ("h", _P), ("hq", _P),
                ("sh", _P), ("acc_down", _P)]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Loads the CUDA library (building it first when sources are newer)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if os.environ.get("BITNET_NO_BUILD") != "1":
            path = _build.build()
        if not os.path.exists(path):
            raise ImportError(f"CUDA library {path} is missing; run build.py")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(fn, status):
    if status != BITNET_OK:
        raise BitnetError(fn, status, lib().bitnet_last_cuda_error())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _workspace(nbytes, device, ws):
    if nbytes == 0:
        return ws
    if ws is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError(f"workspace too small: need {nbytes} bytes")
    return ws


# ------------------------------------------------------------------ weights
def bitnet_quantize_weights_workspace(N, K) -> int:
    return int(lib().bitnet_quantize_weights_workspace(N, K))


def bitnet_quantize_weights(W, Wq=None, w_scale=None, ws=None, stream=None):
    """W float32 [N, K] (device) -> (Wq uint8 [N, K/4], w_scale float32 [1])."""
    N, K = W.shape
    if Wq is None:
        Wq = torch.empty((N, K // 4), dtype=torch.uint8, device=W.device)
    if w_scale is None:
        w_scale = torch.empty(1, dtype=torch.float32, device=W.device)
    nb = bitnet_quantize_weights_workspace(N, K)
    ws = _workspace(nb, W.device, ws)
    _check("bitnet_quantize_weights", lib().bitnet_quantize_weights(
        _ptr(W, torch.float32, "W"), N, K, _ptr(Wq, torch.uint8, "Wq"),
        _ptr(w_scale, torch.float32, "w_scale"), _ptr(ws, name="ws"), nb, _stream(stream)))
    return Wq, w_scale


def bitnet_quantize_weights_noalloc(W, Wq=None, w_scale=None, stream=None):
    """As bitnet_quantize_weights, with the library's own fixed scratch (no
    workspace argument).  Calls that overlap on the GPU must be serialised."""
    N, K = W.shape
    if Wq is None:
        Wq = torch.empty((N, K // 4), dtype=torch.uint8, device=W.device)
    if w_scale is None:
        w_scale = torch.empty(1, dtype=torch.float32, device=W.device)
    _check("bitnet_quantize_weights_noalloc", lib().bitnet_quantize_weights_noalloc(
        _ptr(W, torch.float32, "W"), N, K, _ptr(Wq, torch.uint8, "Wq"),
        _ptr(w_scale, torch.float32, "w_scale"), _stream(stream)))
    return Wq, w_scale


# ------------------------------------------------------------------ activations
def bitnet_quantize_act(x, xq=None, x_scale=None, stream=None):
    """x bfloat16 [M, K] (device) -> (xq int8 [M, K], x_scale float32 [M])."""
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if x_scale is None:
        x_scale = torch.empty(M, dtype=torch.float32, device=x.device)
    _check("bitnet_quantize_act", lib().bitnet_quantize_act(
        _ptr(x, torch.bfloat16, "x"), M, K, _ptr(xq, torch.int8, "xq"),
        _ptr(x_scale, torch.float32, "x_scale"), _stream(stream)))
    return xq, x_scale


# ------------------------------------------------------------------ linear
def bitnet_linear_workspace(M, N, K) -> int:
    return int(lib().bitnet_linear_workspace(M, N, K))


def bitnet_linear(Wq, w_scale, xq, x_scale, K=None, y=None, acc_out=None, ws=None,
                  stream=None, y_bf16=None):
    """Packed ternary Wq [N, K/4] x int8 xq [M, K] -> y float32 [M, N] and/or
    y_bf16 bfloat16 [M, N] (y rounded to nearest-even).  With neither given,
    y is allocated.  Returns y, or y_bf16 when y is None."""
    N = Wq.shape[0]
    M, Kx = xq.shape
    K = Kx if K is None else K
    if y is None and y_bf16 is None:
        y = torch.empty((M, N), dtype=torch.float32, device=xq.device)
    nb = bitnet_linear_workspace(M, N, K)
    ws = _workspace(nb, xq.device, ws)
    _check("bitnet_linear", lib().bitnet_linear(
        _ptr(Wq, torch.uint8, "Wq"), _ptr(w_scale, torch.float32, "w_scale"),
        _ptr(xq, torch.int8, "xq"), _ptr(x_scale, torch.float32, "x_scale"), M, N, K,
        _ptr(y, torch.float32, "y"), _ptr(y_bf16, torch.bfloat16, "y_bf16"),
        _ptr(acc_out, torch.int32, "acc_out"), _ptr(ws, name="ws"), nb, _stream(stream)))
    return y if y is not None else y_bf16


def bitnet_linear_lut(Wq, w_scale, xq, x_scale, variant=0, y=None, acc_out=None, stream=None):
    """One-token BitLinear with the table-lookup (variant 0) or dp4a (variant
    1) inner product: packed Wq [N, K/4] x int8 xq [1, K] (or [K]) -> y
    float32 [1, N]."""
    N = Wq.shape[0]
    K = xq.shape[-1]
    if y is None:
        y = torch.empty((1, N), dtype=torch.float32, device=xq.device)
    _check("bitnet_linear_lut", lib().bitnet_linear_lut(
        _ptr(Wq, torch.uint8, "Wq"), _ptr(w_scale, torch.float32, "w_scale"),
        _ptr(xq, torch.int8, "xq"), _ptr(x_scale, torch.float32, "x_scale"), N, K,
        _ptr(y, torch.float32, "y"), _ptr(acc_out, torch.int32, "acc_out"), int(variant),
        _stream(stream)))
    return y


BITNET_WEIGHTS_STATIC = 1


def _target(t):
    """(Wq, w_scale, y[, acc_out[, y_bf16]]) -> LinearTarget; y may be None
    when y_bf16 is given."""
    Wq, ws, y = t[0], t[1], t[2]
    acc = t[3] if len(t) > 3 else None
    yb = t[4] if len(t) > 4 else None
    return LinearTarget(_ptr(Wq, torch.uint8, "Wq"), _ptr(ws, torch.float32, "w_scale"),
                        Wq.shape[0], _ptr(y, torch.float32, "y"), _ptr(acc, torch.int32, "acc_out"),
                        _ptr(yb, torch.bfloat16, "y_bf16"))


def bitnet_linear_bf16(x, targets, xq_out=None, x_scale_out=None, weights_static=False,
                       stream=None):
    """Per-token int8 quantisation of bf16 x [M, K] and BitLinear with every
    (Wq, w_scale, y[, acc_out[, y_bf16]]) in `targets` (all sharing x), one
    launch.  weights_static: no work in flight on the stream writes the
    weights, so they may stream in before the previous kernel has finished."""
    M, K = x.shape
    arr = (LinearTarget * len(targets))()
    for i, t in enumerate(targets):
        arr[i] = _target(t)
    _check("bitnet_linear_bf16", lib().bitnet_linear_bf16(
        _ptr(x, torch.bfloat16, "x"), M, K, arr, len(targets),
        _ptr(xq_out, torch.int8, "xq_out"), _ptr(x_scale_out, torch.float32, "x_scale_out"),
        BITNET_WEIGHTS_STATIC if weights_static else 0, _stream(stream)))
    return [t[2] for t in targets]


BITNET_PHASE_GATED = 1


class DecodeChainHandle:
    """A built decode chain: its device table (a torch tensor) and the host
    description bitnet_decode_chain_run needs.  Keeps the target arrays and
    tensors it was built from alive."""

    def __init__(self, chain, table, keep):
        self.chain = chain
        self.table = table
        self._keep = keep


def _phase(spec):
    """A phase as a dict (keys: x | x_f32, targets, gated, h, norm_gain,
    norm_eps, xq_out, x_scale_out) or as a tuple (x, targets)."""
    if not isinstance(spec, dict):
        spec = {"x": spec[0], "targets": spec[1]}
    x, xf = spec.get("x"), spec.get("x_f32")
    src = x if x is not None else xf
    targets = spec["targets"]
    tarr = (LinearTarget * len(targets))()
    for j, t in enumerate(targets):
        tarr[j] = _target(t)
    ph = DecodePhase(_ptr(x, torch.bfloat16, "x"), src.shape[1], ctypes.cast(tarr, ctypes.c_void_p),
                     len(targets), BITNET_PHASE_GATED if spec.get("gated") else 0,
                     _ptr(xf, torch.float32, "x_f32"),
                     _ptr(spec.get("norm_gain"), torch.float32, "norm_gain"),
                     float(spec.get("norm_eps", 0.0)), _ptr(spec.get("h"), torch.float32, "h"),
                     _ptr(spec.get("xq_out"), torch.int8, "xq_out"),
                     _ptr(spec.get("x_scale_out"), torch.float32, "x_scale_out"))
    return ph, (tarr, spec), src.shape[0]


def bitnet_decode_chain_build(phases, device="cuda"):
    """phases: list of phase dicts (see _phase) or (x, targets) tuples.
    Builds the chain table in device memory (synchronous)."""
    n = len(phases)
    arr = (DecodePhase * n)()
    keep = []
    M = None
    for i, spec in enumerate(phases):
        arr[i], k, m = _phase(spec)
        keep.append(k)
        M = m if M is None else M
    nbytes = int(lib().bitnet_decode_chain_bytes(arr, n, M))
    if nbytes == 0:
        # the same checks give the status
        chain = DecodeChain()
        _check("bitnet_decode_chain_build", lib().bitnet_decode_chain_build(
            arr, n, M, None, 0, ctypes.byref(chain)))
        raise BitnetError("bitnet_decode_chain_bytes", 2)
    table = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
    base = (table.data_ptr() + 255) // 256 * 256
    chain = DecodeChain()
    _check("bitnet_decode_chain_build", lib().bitnet_decode_chain_build(
        arr, n, M, ctypes.c_void_p(base), nbytes, ctypes.byref(chain)))
    return DecodeChainHandle(chain, table, keep)


def bitnet_decode_chain_run(handle, stream=None):
    _check("bitnet_decode_chain_run", lib().bitnet_decode_chain_run(
        ctypes.byref(handle.chain), _stream(stream)))


def bitnet_set_wait_limit(cycles):
    """Test hook: bound of the kernels' waits in SM clocks (0 = default)."""
    lib().bitnet_set_wait_limit(int(cycles))


# ------------------------------------------------------------------ FFN
def bitnet_ffn_workspace(M, H, F) -> int:
    return int(lib().bitnet_ffn_workspace(M, H, F))


def bitnet_ffn(x, g, eps, Wup, s_up, Wgate, s_gate, Wdown, s_down, y=None, debug=None,
               ws=None, stream=None):
    """subln RMSNorm -> int8 -> up/gate BitLinear -> ReLU^2 gate -> int8 -> down.

    x bfloat16 [M, H]; returns y float32 [M, H].  `debug` may be a dict with
    any of xq, sx, u, v, h, hq, sh, acc_down (device tensors to receive them).
    """
    M, H = x.shape
    F = Wup.shape[0]
    if y is None:
        y = torch.empty((M, H), dtype=torch.float32, device=x.device)
    dbg = None
    if debug:
        types = dict(xq=torch.int8, sx=torch.float32, u=torch.float32, v=torch.float32,
                     h=torch.float32, hq=torch.int8, sh=torch.float32, acc_down=torch.int32)
        dbg = FfnDebug(**{k: _ptr(debug.get(k), types[k], k) for k in types})
    nb = bitnet_ffn_workspace(M, H, F)
    ws = _workspace(nb, x.device, ws)
    _check("bitnet_ffn", lib().bitnet_ffn(
        _ptr(x, torch.bfloat16, "x"), _ptr(g, torch.float32, "g"), float(eps),
        _ptr(Wup, torch.uint8, "Wup"), _ptr(s_up, torch.float32, "s_up"),
        _ptr(Wgate, torch.uint8, "Wgate"), _ptr(s_gate, torch.float32, "s_gate"),
        _ptr(Wdown, torch.uint8, "Wdown"), _ptr(s_down, torch.float32, "s_down"),
        M, H, F, _ptr(y, torch.float32, "y"), ctypes.byref(dbg) if dbg is not None else None,
        _ptr(ws, name="ws"), nb, _stream(stream)))
    return y


def bitnet_device_error(stream=None) -> int:
    code = ctypes.c_int(0)
    _check("bitnet_device_error", lib().bitnet_device_error(ctypes.byref(code), _stream(stream)))
    return code.value
