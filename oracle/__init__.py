"""Oracle for the IHA attention-layer hot path (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it.

The arithmetic lives in ``iha_oracle.c`` (plain loops, double accumulation,
OpenMP over independent rows).  This wrapper only marshals numpy arrays:
bf16 inputs (uint16 bit patterns) are widened to float32 exactly before the
call; results come back as float64.

Sources: "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs",
sections "Pseudo-Token Mixing (Triton Premix Kernels)" and "FLOP Matching",
and "Repository Structure" / "End-to-End Training Benchmark" (the attention
backward of the training step);
"hiera-optim 0.1.0", README item 2 (gather / scatter) and
hiera_optim/attention/mask_unit.py (MaskUnitAttentionFast.forward).
Every oracle function is pinned by a CPU test against values the pages or the
mathematics fix (tests/test_oracle.py); none is marked "parity unpinned".
"""
from __future__ import annotations

import ctypes as C
import math

import numpy as np

from . import build as _build

_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        dp, fp, lp, i32p, u8p = (C.POINTER(C.c_double), C.POINTER(C.c_float),
                                 C.POINTER(C.c_long), C.POINTER(C.c_int32),
                                 C.POINTER(C.c_uint8))
        l, i, d = C.c_long, C.c_int, C.c_double
        L.oracle_num_threads.restype = C.c_int
        L.oracle_rope.argtypes = [dp, dp, l, l, l, l, d, i]
        for name in ("oracle_premix_fwd", "oracle_premix_bwd_dx"):
            getattr(L, name).argtypes = [fp, fp, dp, l, l, l, l, l, i, d, l]
        L.oracle_premix_bwd_dw.argtypes = [fp, fp, dp, l, l, l, l, l, i, d]
        L.oracle_attention.argtypes = [fp, fp, fp, dp, dp, l, l, l, l, l, l,
                                       lp, lp, lp, d, i, l]
        L.oracle_attention_rows.argtypes = [fp, fp, fp, lp, l, dp, dp, l, l,
                                            lp, lp, lp, d, i, l]
        L.oracle_attention_bwd.argtypes = [fp, fp, fp, fp, dp, dp, dp, l, l, l, l, d, i, l, i]
        L.oracle_tile_visits.argtypes = [l, l, i, l, l, l]
        L.oracle_tile_visits.restype = l
        for name in ("oracle_mu_gather", "oracle_mu_scatter"):
            getattr(L, name).argtypes = [u8p, i32p, u8p, l, l, l, l, l, l, l, l]
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


# ------------------------------------------------------------------ helpers
def _as_f32(a: np.ndarray) -> np.ndarray:
    """Exact float32 view of the input: bf16 bit patterns are widened."""
    if a.dtype == np.uint16:
        return (np.ascontiguousarray(a).astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.ascontiguousarray(a, dtype=np.float32)


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(C.POINTER(ct))


MASK_NONE, MASK_CAUSAL, MASK_CAUSAL_WINDOW = 0, 1, 2


# ------------------------------------------------------------------ premix
def premix_fwd(x: np.ndarray, w: np.ndarray, P: int, rope: bool = False,
               rope_base: float = 10000.0, pos0: int = 0) -> np.ndarray:
    """Y[B,N,H*P,d] (float64) from X[B,N,H,d] and W[H,P,H].

    pos0: RoPE position of the first row (for a window of a longer sequence).
    """
    B, N, H, d = x.shape
    xf, wf = _as_f32(x), _as_f32(w)
    assert wf.shape == (H, P, H)
    y = np.empty((B, N, H * P, d), dtype=np.float64)
    lib().oracle_premix_fwd(_p(xf, C.c_float), _p(wf, C.c_float), _p(y, C.c_double),
                            B, N, H, P, d, int(rope), float(rope_base), int(pos0))
    return y


def premix_bwd_dx(dy: np.ndarray, w: np.ndarray, rope: bool = False,
                  rope_base: float = 10000.0, pos0: int = 0) -> np.ndarray:
    """dX[B,N,H,d] (float64) from dY[B,N,H*P,d] and W[H,P,H]."""
    B, N, HP, d = dy.shape
    H, P, _ = w.shape
    assert HP == H * P
    gf, wf = _as_f32(dy), _as_f32(w)
    dx = np.empty((B, N, H, d), dtype=np.float64)
    lib().oracle_premix_bwd_dx(_p(gf, C.c_float), _p(wf, C.c_float), _p(dx, C.c_double),
                               B, N, H, P, d, int(rope), float(rope_base), int(pos0))
    return dx


def premix_bwd_dw(dy: np.ndarray, x: np.ndarray, P: int, rope: bool = False,
                  rope_base: float = 10000.0) -> np.ndarray:
    """dW[H,P,H] (float64) from dY[B,N,H*P,d] and X[B,N,H,d]."""
    B, N, H, d = x.shape
    assert dy.shape == (B, N, H * P, d)
    gf, xf = _as_f32(dy), _as_f32(x)
    dw = np.empty((H, P, H), dtype=np.float64)
    lib().oracle_premix_bwd_dw(_p(gf, C.c_float), _p(xf, C.c_float), _p(dw, C.c_double),
                               B, N, H, P, d, int(rope), float(rope_base))
    return dw


def rope(x: np.ndarray, base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """Rotate-half RoPE of x[B,N,heads,d] (float64) at positions n = 0..N-1."""
    B, N, heads, d = x.shape
    xi = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(xi)
    lib().oracle_rope(_p(xi, C.c_double), _p(y, C.c_double), B, N, heads, d,
                      float(base), int(inverse))
    return y


# ------------------------------------------------------------------ attention
def _strides5(a: np.ndarray) -> np.ndarray:
    """Element strides (b_outer, b_inner, seq, head) of a [Bo,Bi,N,Hh,d] view."""
    s = [st // a.itemsize for st in a.strides]
    assert s[4] == 1, "last dim must be dense"
    return np.array(s[:4], dtype=np.int64)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: int = 0,
              window: int = 0, scale: float | None = None):
    """Attention over [Bo,Bi,N,Hh,d] views (float32 or bf16 bits).

    Returns O [Bo,Bi,Nq,Hh,d] float64 and lse [Bo,Bi,Hh,Nq] float64.
    """
    qf, kf, vf = _as_f32(q), _as_f32(k), _as_f32(v)
    Bo, Bi, Nq, Hh, d = qf.shape
    Nk = kf.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.empty((Bo, Bi, Nq, Hh, d), dtype=np.float64)
    lse = np.empty((Bo, Bi, Hh, Nq), dtype=np.float64)
    sq, sk, sv = _strides5(qf), _strides5(kf), _strides5(vf)
    lib().oracle_attention(_p(qf, C.c_float), _p(kf, C.c_float), _p(vf, C.c_float),
                           _p(o, C.c_double), _p(lse, C.c_double),
                           Bo, Bi, Hh, Nq, Nk, d, _p(sq, C.c_long), _p(sk, C.c_long),
                           _p(sv, C.c_long), float(scale), int(mask), int(window))
    return o, lse


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: np.ndarray,
                   mask: int = 0, window: int = 0, scale: float | None = None):
    """Selected rows (n, 4) = (bo, bi, head, i) of the attention above.

    Returns O rows [n, d] and lse [n] (float64).  Inputs as in ``attention``.
    """
    qf, kf, vf = _as_f32(q), _as_f32(k), _as_f32(v)
    Bo, Bi, Nq, Hh, d = qf.shape
    Nk = kf.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rr = np.ascontiguousarray(rows, dtype=np.int64)
    n = rr.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    sq, sk, sv = _strides5(qf), _strides5(kf), _strides5(vf)
    lib().oracle_attention_rows(_p(qf, C.c_float), _p(kf, C.c_float), _p(vf, C.c_float),
                                _p(rr, C.c_long), n, _p(o, C.c_double), _p(lse, C.c_double),
                                Nk, d, _p(sq, C.c_long), _p(sk, C.c_long), _p(sv, C.c_long),
                                float(scale), int(mask), int(window))
    return o, lse


def attention_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray,
                  mask: int = 0, window: int = 0, scale: float | None = None,
                  absolute: bool = False):
    """Gradients (dQ, dK, dV) of attention over dense [B, N, Hh, d] tensors
    (float32 or bf16 bits) for the upstream gradient dout; float64 results.
    absolute=True returns the same sums over absolute values of their terms
    (sum |dS||k|, sum |dS||q|, sum P|dO|), the scale of rounding errors."""
    qf, kf, vf, gf = _as_f32(q), _as_f32(k), _as_f32(v), _as_f32(dout)
    B, N, Hh, d = qf.shape
    assert kf.shape == vf.shape == gf.shape == qf.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.empty(qf.shape, dtype=np.float64)
    dk = np.empty(qf.shape, dtype=np.float64)
    dv = np.empty(qf.shape, dtype=np.float64)
    lib().oracle_attention_bwd(_p(qf, C.c_float), _p(kf, C.c_float), _p(vf, C.c_float),
                               _p(gf, C.c_float), _p(dq, C.c_double), _p(dk, C.c_double),
                               _p(dv, C.c_double), B, Hh, N, d, float(scale), int(mask),
                               int(window), int(absolute))
    return dq, dk, dv


def tile_visits(N: int, heads: int, mask: int, window: int, tile_q: int = 128,
                tile_k: int = 128) -> int:
    """(head, query tile, key tile) triples holding at least one visible pair."""
    return int(lib().oracle_tile_visits(N, heads, mask, window, tile_q, tile_k))


# ------------------------------------------------------------------ gather / scatter
def mu_gather(x: np.ndarray, keep: np.ndarray, grid_h: int, grid_w: int,
              mu_h: int, mu_w: int) -> np.ndarray:
    """x [B, grid_h*grid_w, C] -> out [B, n_keep, mu_h*mu_w, C] (same dtype)."""
    x = np.ascontiguousarray(x)
    keep = np.ascontiguousarray(keep, dtype=np.int32)
    B, G, Cc = x.shape
    n_keep = keep.shape[1]
    out = np.empty((B, n_keep, mu_h * mu_w, Cc), dtype=x.dtype)
    lib().oracle_mu_gather(_p(x.view(np.uint8), C.c_uint8), _p(keep, C.c_int32),
                           _p(out.view(np.uint8), C.c_uint8), B, grid_h, grid_w,
                           mu_h, mu_w, n_keep, Cc, x.itemsize)
    return out


def mu_scatter(src: np.ndarray, keep: np.ndarray, x: np.ndarray, grid_h: int,
               grid_w: int, mu_h: int, mu_w: int) -> np.ndarray:
    """Copy of x with the kept units' tokens overwritten from src."""
    out = np.array(x, copy=True, order="C")
    src = np.ascontiguousarray(src, dtype=out.dtype)
    keep = np.ascontiguousarray(keep, dtype=np.int32)
    B, G, Cc = out.shape
    n_keep = keep.shape[1]
    lib().oracle_mu_scatter(_p(src.view(np.uint8), C.c_uint8), _p(keep, C.c_int32),
                            _p(out.view(np.uint8), C.c_uint8), B, grid_h, grid_w,
                            mu_h, mu_w, n_keep, Cc, out.itemsize)
    return out


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float64 results to the bf16 grid (RNE, via float32) -> float64.

    Used to compare a bf16-output kernel with the oracle at the output dtype.
    Double rounding (f64 -> f32 -> bf16) can differ from direct rounding only
    on exact ties at the f32 step, which the tolerances absorb.
    """
    f = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (f >> np.uint32(16)) & np.uint32(1)
    r = ((f + np.uint32(0x7FFF) + lsb) >> np.uint32(16)) << np.uint32(16)
    return r.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- interleaved pseudo-tokens
def interleave_heads(y: np.ndarray, H: int, P: int) -> np.ndarray:
    """Premix output [B, N, H*P, d] (rows h*P + p) -> [B, N, P, H, d].

    The interleaved pseudo-token layout of the joint-softmax reading of IHA
    ("IHA-CUDA", the "interleaved" heads and the softmax "joint" across the
    P pseudo-heads): pseudo-token n*P + p of head h carries Y[b, n, h*P + p].
    A pure reordering; no arithmetic.
    """
    B, N, HP, d = y.shape
    assert HP == H * P
    return np.ascontiguousarray(y.reshape(B, N, H, P, d).transpose(0, 1, 3, 2, 4))


def joint_attention(yq: np.ndarray, yk: np.ndarray, yv: np.ndarray, causal: bool = True,
                    scale: float | None = None):
    """Attention of each head h over the N*P interleaved pseudo-tokens
    m = n*P + p of [B, N, P, H, d] inputs (causal on m when `causal`), by
    the plain two-pass softmax of ``attention`` on the [B, 1, N*P, H, d] view.

    Returns O [B, N, P, H, d] float64 and lse [B, H, N*P] float64.
    """
    B, N, P, H, d = yq.shape
    view = lambda a: np.ascontiguousarray(a).reshape(B, 1, N * P, H, d)
    o, lse = attention(view(yq), view(yk), view(yv), MASK_CAUSAL if causal else MASK_NONE, 0,
                       scale)
    return o.reshape(B, N, P, H, d), lse.reshape(B, H, N * P)


# ---------------------------------------------------------------- Hiera q_pool
def q_pool(q: np.ndarray, q_stride: int) -> np.ndarray:
    """Max-pooled queries of each mask unit ("hiera-optim 0.1.0",
    hiera_optim/attention/mask_unit.py, MaskUnitAttentionFast.forward with
    q_stride > 1): a unit's T query rows form q_stride blocks of
    Tq = T / q_stride rows, the block index being the slow axis, and pooled
    row t is the elementwise maximum over the blocks of row t of each block
    (rows t, Tq + t, ..., (q_stride - 1) * Tq + t).

    q [Bo, Bi, T, Hh, d] (float32 or bf16 bits) -> float32 [Bo, Bi, Tq, Hh, d];
    a maximum picks one of its inputs, so bf16 values stay exact.
    """
    qf = _as_f32(q)
    Bo, Bi, T, Hh, d = qf.shape
    assert q_stride >= 1 and T % q_stride == 0
    Tq = T // q_stride
    return np.ascontiguousarray(qf.reshape(Bo, Bi, q_stride, Tq, Hh, d).max(axis=2))


def attention_qpool(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_stride: int,
                    scale: float | None = None):
    """Unmasked attention of the pooled queries over all T keys of the unit:
    ``attention(q_pool(q, q_stride), k, v)`` (the same page and function).

    Returns O [Bo,Bi,Tq,Hh,d] float64 and lse [Bo,Bi,Hh,Tq] float64.
    """
    return attention(q_pool(q, q_stride), k, v, MASK_NONE, 0, scale)
