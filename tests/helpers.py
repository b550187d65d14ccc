"""Shared test helpers: host <-> device transfer and the comparison rules.

Comparison rules (stated once here, used by every parity test):
  bf16 outputs (fp32 accumulation): per element |g - r_bf16| <= max(1e-2, 1 ulp_bf16(r_bf16))
      where r_bf16 is the oracle rounded to bf16 (RNE), and rel-L2
      ||g - r|| / ||r|| <= 1e-2 against the unrounded oracle.
  fp32 outputs of fp32 paths: max |g - r| <= 1e-5.
  fp32 weight gradient of bf16 inputs: |g - r| <= 2e-5 * sum_i |a_i b_i| per
      element (fp32 accumulation over a long reduction, bounded relative to
      the sum of absolute products), where the abs-sum comes from the oracle
      run on |dY|, |X|.
  byte / index work: bit-exact.
"""
from __future__ import annotations

import numpy as np

import oracle as O
import synthetic as S

BF16_ABS = 1e-2
BF16_REL_L2 = 1e-2
F32_ABS = 1e-5
DW_REL_ABS_SUM = 2e-5


def to_dev(a: np.ndarray, device="cuda"):
    """numpy (uint16 = bf16 bits, float32, int32) -> torch tensor on device."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_f64(t) -> np.ndarray:
    """torch tensor (bf16 or fp32, any device) -> float64 numpy (exact)."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return S.bf16_bits_to_f32(t.contiguous().view(torch.int16).numpy().view(np.uint16)).astype(np.float64)
    return t.contiguous().numpy().astype(np.float64)


def ulp_bf16(r: np.ndarray) -> np.ndarray:
    a = np.abs(r)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def assert_bf16_close(g: np.ndarray, r: np.ndarray, what: str = "") -> dict:
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    rb = O.round_bf16(r)
    err = np.abs(g - rb)
    bound = np.maximum(BF16_ABS, ulp_bf16(rb))
    bad = err > bound
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    stats = {"max_abs_vs_rounded": float(err.max(initial=0.0)),
             "max_abs_vs_exact": float(np.abs(g - r).max(initial=0.0)), "rel_l2": rel}
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {idx}: "
                             f"gpu={g[idx]!r} oracle={r[idx]!r} ({stats})")
    assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel} ({stats})"
    return stats


def assert_f32_close(g: np.ndarray, r: np.ndarray, what: str = "", tol: float = F32_ABS) -> float:
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    m = float(np.abs(g - r).max(initial=0.0))
    assert m <= tol, f"{what}: max abs {m} > {tol}"
    return m


def assert_dw_close(g: np.ndarray, r: np.ndarray, abs_sum: np.ndarray, what: str = "") -> float:
    g = np.asarray(g, np.float64)
    err = np.abs(g - r)
    bound = DW_REL_ABS_SUM * abs_sum + 1e-6
    assert np.all(np.isfinite(g)), f"{what}: non-finite dW"
    worst = float((err / bound).max())
    assert worst <= 1.0, f"{what}: dW error {err.max()} exceeds bound (ratio {worst})"
    return worst


def abs_bits(a: np.ndarray) -> np.ndarray:
    """|a| for bf16 bit patterns (clear the sign bit) or floats."""
    if a.dtype == np.uint16:
        return a & np.uint16(0x7FFF)
    return np.abs(a)
