"""Shared test helpers: device checks, tolerance checks and dtype conversions.

Tolerances for the mat-vecs are measured against the fp64 oracle in two ways, both
of which must hold (tol = 1e-3 for bf16, 1e-4 for q8_0):
  normwise       ||y - y64||_2 / ||y64||_2 <= tol
  componentwise  |y_r - y64_r| <= tol * sum_k |W_rk x_k|
The componentwise scale is the row's sum of term magnitudes, so rows whose terms
cancel are judged against the size of the terms, not the size of the result.
"""
import numpy as np
import pytest
import torch

TOL_BF16 = 1e-3
TOL_Q8 = 1e-4


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import weight_streaming_warp_gb300 as wsw
    wsw.load()  # raises if the library is missing: no silent fallback
    return wsw


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def f16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64_bf16(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_tol(y, y64, mag, tol, what=""):
    y = np.asarray(y, np.float64)
    y64 = np.asarray(y64, np.float64)
    mag = np.asarray(mag, np.float64)
    assert y.shape == y64.shape, (y.shape, y64.shape)
    assert np.isfinite(y).all(), what + ": non-finite output"
    nrm = np.linalg.norm(y64)
    if nrm > 0:
        rel = np.linalg.norm(y - y64) / nrm
        assert rel <= tol, "%s: normwise error %.3g > %.3g" % (what, rel, tol)
    err = np.abs(y - y64)
    bound = tol * mag + 1e-30
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, "%s: %d components over tolerance, first %d: %g vs %g (scale %g)" % (
        what, bad.size, bad[0], y[bad[0]], y64[bad[0]], mag[bad[0]])


def mag_bf16(W_bits: np.ndarray, x: np.ndarray, K=None):
    W = bits_to_f64_bf16(W_bits)
    if K is not None:
        W = W[:, :K]
    return np.abs(W) @ np.abs(np.asarray(x, np.float64)[:W.shape[1]])


def mag_q8(Wq, Wd_bits, xq, xd_bits):
    K = xq.shape[-1]
    wd = np.repeat(Wd_bits.view(np.float16).astype(np.float64), 32, axis=-1)[..., :K]
    xd = np.repeat(xd_bits.view(np.float16).astype(np.float64), 32, axis=-1)[..., :K]
    W = np.abs(Wq[..., :K].astype(np.float64) * wd)
    x = np.abs(xq.astype(np.float64) * xd)
    return W @ x


def u16_to_torch(a: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)
