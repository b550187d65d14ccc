"""Shared test helpers: host <-> device transfer and the comparison rules.

Comparison rules (stated once here, used by every parity test):
  bf16 outputs (fp32 accumulation): per element |g - r_bf16| <= max(1e-2, 1 ulp_bf16(r_bf16))
      where r_bf16 is the oracle rounded to bf16 (RNE), and rel-L2
      ||g - r|| / ||r|| <= 1e-2 against the unrounded oracle (RMS |g| <= 1e-2
      when the oracle is identically zero, e.g. dK under a window of one key).
  fp32 outputs of fp32 paths: max |g - r| <= 1e-5.
  fp32 weight gradient (both dtypes): per element the first-order bound of
      recursive fp32 summation, |g - r| <= u (L + n) sum_i |a_i b_i|, with
      u = 2^-23 (one fp32 rounding, truncation allowed in the tensor-core
      adder), L the longest chain of additions into one running sum and n
      the partial sums one element receives by atomics (dw_chain, from each
      kernel's blocking), plus the bf16 hi + lo split of R X (2^-17) and the
      fp32 rotation (2^-22) with RoPE; sum_i |a_i b_i| comes from the oracle
      on |dY| and |X| (and |X| with partner features swapped, for RoPE).
      That bound is a guarantee, and loose; the sharp check is rel-L2
      ||g - r|| / ||r|| <= 1e-5 (typical blocked fp32 error ~1e-6).
  bf16 attention gradients: per element |g - r_bf16| <= max(1e-2, 1 ulp) +
      (2^-8 + (L + 16) 2^-23) sum_i |t_i|: each term t_i of a gradient's sum
      carries the bf16 rounding (unit roundoff 2^-8) of the MMA operand it
      multiplies (dS for dQ and dK, P for dV) plus fp32 accumulation over at
      most L = N terms; sum_i |t_i| is the oracle run on absolute terms.  And
      rel-L2 <= 1e-2.
  byte / index work: bit-exact.
"""
from __future__ import annotations

import numpy as np

import oracle as O
import synthetic as S

BF16_ABS = 1e-2
BF16_REL_L2 = 1e-2
F32_ABS = 1e-5
U_ACC = 2.0 ** -23
DW_REL_L2 = 1e-5
DW_TT = 4  # tokens per shared-memory chunk of the mma.sync weight-gradient kernel


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
    nr = float(np.linalg.norm(r))
    if nr > 0.0:
        rel = float(np.linalg.norm(g - r) / nr)
    else:  # an all-zero reference: hold the RMS error to the same 1e-2
        rel = float(np.linalg.norm(g) / np.sqrt(max(g.size, 1)))
    stats = {"max_abs_vs_rounded": float(err.max(initial=0.0)),
             "max_abs_vs_exact": float(np.abs(g - r).max(initial=0.0)), "rel_l2": rel}
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {idx}: "
                             f"gpu={g[idx]!r} oracle={r[idx]!r} ({stats})")
    assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel} ({stats})"
    return stats


def assert_grad_close(g: np.ndarray, r: np.ndarray, abs_terms: np.ndarray, L: int,
                      what: str = "") -> dict:
    """Gradient rule (module docstring): the bf16 output rule widened by the
    rounding of bf16 MMA operands, scaled by the sum of absolute terms."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    assert g.shape == r.shape == abs_terms.shape, (g.shape, r.shape, abs_terms.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    rb = O.round_bf16(r)
    err = np.abs(g - rb)
    bound = np.maximum(BF16_ABS, ulp_bf16(rb)) + (2.0 ** -8 + (L + 16) * 2.0 ** -23) * abs_terms
    nr = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / nr) if nr > 0 else float(
        np.linalg.norm(g) / np.sqrt(max(g.size, 1)))
    stats = {"max_abs_vs_rounded": float(err.max(initial=0.0)),
             "max_abs_vs_exact": float(np.abs(g - r).max(initial=0.0)), "rel_l2": rel,
             "worst_over_bound": float((err / bound).max(initial=0.0))}
    bad = err > bound
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


def n_sms() -> int:
    import torch
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def dw_chain(B: int, N: int, H: int, P: int, d: int, dtype: str = "bf16", rope: bool = False,
             n_sm: int | None = None) -> tuple[int, int]:
    """(L, n): the longest chain of fp32 additions into one running sum, and the
    number of partial sums combined by atomics, over the weight-gradient
    kernels that can run for this shape:
      tensor-core kernel (bf16, d = 128): CTA c of min(SMs, tokens) owns tokens
        c, c + grid, ...; each token adds d/16 MMA K-steps of 16 products to the
        TMEM accumulator (the 16 products of one K-step add inside the tensor
        core: 16 more); with RoPE the hi and lo columns add once at the end;
      mma.sync kernel (other bf16 shapes): 4 blocks per SM over slabs of whole
        4-token chunks, d/16 K-steps per token, twice with RoPE (hi and lo);
      fp32 kernel: 256 threads stride over tokens x features, then an 8-level
        tree; plain store."""
    ntok = B * N
    if n_sm is None:
        n_sm = n_sms()
    if dtype == "f32":
        return -(-ntok * d // 256) + 8, 0
    ks = -(-d // 16)
    grid = min(n_sm, ntok)
    tc = -(-ntok // grid) * ks + 16 + (1 if rope else 0)
    blocks = n_sm * 4
    per = -(-ntok // blocks)
    per = -(-per // DW_TT) * DW_TT
    blocks = -(-ntok // per)
    ms = per * ks * (2 if rope else 1) + 16
    return max(tc, ms), max(grid, blocks)


def dw_abs_sum(dy: np.ndarray, x: np.ndarray, P: int, rope: bool = False) -> np.ndarray:
    """sum over (tokens, features) of |g_f| |x'_f| bounding every product the
    kernels add: |dY| |X|, and with RoPE also |dY| times |X| with each feature
    swapped for its rotation partner (R X mixes f with f +- d/2)."""
    a = O.premix_bwd_dw(abs_bits(dy), abs_bits(x), P)
    if rope:
        d = x.shape[-1]
        xs = np.concatenate([x[..., d // 2:], x[..., : d // 2]], axis=-1)
        a = a + O.premix_bwd_dw(abs_bits(dy), abs_bits(np.ascontiguousarray(xs)), P)
    return a


def assert_dw_close(g: np.ndarray, r: np.ndarray, abs_sum: np.ndarray, chain: tuple[int, int],
                    rope: bool = False, what: str = "") -> dict:
    """Weight-gradient rule (module docstring): per-element blocked-summation
    bound and rel-L2 <= 1e-5 against the exact (float64) oracle."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite dW"
    L, n = chain
    coef = U_ACC * (L + n) + ((2.0 ** -17 + 2.0 ** -22) if rope else 0.0)
    bound = coef * abs_sum + 1e-30
    err = np.abs(g - r)
    worst = float((err / bound).max())
    nr = float(np.linalg.norm(r))
    if nr > 0.0:
        rel = float(np.linalg.norm(g - r) / nr)
    else:  # an all-zero reference: hold the RMS error to the same 1e-2
        rel = float(np.linalg.norm(g) / np.sqrt(max(g.size, 1)))
    stats = {"max_abs": float(err.max()), "worst_over_bound": worst, "rel_l2": rel}
    assert worst <= 1.0, f"{what}: dW error exceeds the blocked-summation bound ({stats})"
    assert rel <= DW_REL_L2, f"{what}: dW rel-L2 {rel} > {DW_REL_L2} ({stats})"
    return stats


def abs_bits(a: np.ndarray) -> np.ndarray:
    """|a| for bf16 bit patterns (clear the sign bit) or floats."""
    if a.dtype == np.uint16:
        return a & np.uint16(0x7FFF)
    return np.abs(a)
