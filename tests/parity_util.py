"""Comparison helpers for the GPU parity tests.

Tolerances, from the accuracy the kernels promise:
  - float32 K/V:          max |err| <= 1e-5 on out and lse;
  - float16 / bfloat16:   max |err| <= 2e-3 on out, <= 1e-3 on lse, with
    float32 accumulation;
  - a 16-bit *output* additionally carries its own final rounding: the bound
    is 2e-3 + half an ulp of the output dtype at |oracle| (round-to-nearest).
"""
from __future__ import annotations

import numpy as np
import torch

OUT_TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}
LSE_TOL = {"f32": 1e-5, "f16": 1e-3, "bf16": 1e-3}
MANT_BITS = {torch.float16: 10, torch.bfloat16: 7}
DTYPE_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def half_ulp(x: np.ndarray, dt: torch.dtype) -> np.ndarray:
    """Half an ulp of |x| in dtype dt (0 for float32 outputs)."""
    if dt == torch.float32:
        return np.zeros_like(x)
    mb = MANT_BITS[dt]
    ax = np.maximum(np.abs(x), 2.0 ** -14 if dt == torch.float16 else 2.0 ** -126)
    return 0.5 * 2.0 ** (np.floor(np.log2(ax)) - mb)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def check_out(out: torch.Tensor, ref: np.ndarray, in_dtype: str, what: str = "out") -> float:
    got = to_np(out)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values (NaN padding read?)"
    tol = OUT_TOL[in_dtype] + half_ulp(ref, out.dtype)
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: max err {err.max():.3e}, {int(bad.sum())} elements over "
                           f"tolerance (first at {np.argwhere(bad)[0].tolist()})")
    return float(err.max()) if err.size else 0.0


def check_lse(lse: torch.Tensor, ref: np.ndarray, in_dtype: str, what: str = "lse") -> float:
    got = to_np(lse)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: finite/-inf pattern differs"
    assert np.all(got[~fin] == -np.inf), f"{what}: empty rows must be -inf"
    if not fin.any():
        return 0.0
    err = np.abs(got[fin] - ref[fin])
    assert err.max() <= LSE_TOL[in_dtype], f"{what}: max err {err.max():.3e}"
    return float(err.max())
