"""Helpers shared by the GPU parity tests: host<->device moves and the
comparison rules.  Holds none of the method's arithmetic."""
import numpy as np
import torch

# fp32 outputs: the gate is a relative error of 1e-5 (expected: bit-exact).
REL_TOL = 1e-5


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16)


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    bad = np.nonzero(got.view(np.uint8).reshape(got.shape + (-1,)) !=
                     want.view(np.uint8).reshape(want.shape + (-1,)))
    if bad[0].size:
        idx = tuple(b[0] for b in bad[:got.ndim])
        raise AssertionError(f"{what}: {bad[0].size} byte mismatches; first at {idx}: "
                             f"got {got[idx]!r}, want {want[idx]!r}")


def assert_f32_close(got: np.ndarray, want: np.ndarray, what: str):
    """fp32 gate: |got - want| <= REL_TOL * |want| element-wise (0 stays 0)."""
    assert got.shape == want.shape, (what, got.shape, want.shape)
    g = got.astype(np.float64)
    w = want.astype(np.float64)
    err = np.abs(g - w)
    lim = REL_TOL * np.abs(w)
    bad = ~(err <= lim)
    if bad.any():
        i = np.unravel_index(np.argmax(bad), bad.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond rel {REL_TOL}; first at "
                             f"{i}: got {got[i]!r}, want {want[i]!r}")
