"""GB300 (sm_103a) library for the Interleaved Head Attention hot path.

Thin ctypes binding over ``libiha.so``: argument marshalling only.  Every
step runs in the library's CUDA kernels; there is no CPU or PyTorch fallback.
If the library is missing, ``lib()`` raises instead of degrading.

Entry points (same names as the C ABI in include/iha.h):
  premix_fwd, premix_bwd_dx, premix_bwd_dw,
  premix_bwd (both gradients, one pass)     -- "IHA-CUDA", section
      "Pseudo-Token Mixing (Triton Premix Kernels)"
  mha_fwd                                   -- "IHA-CUDA", sections "Kernel
      Design" and "FLOP Matching"; hiera-optim MaskUnitAttentionFast.forward
  mu_gather, mu_scatter                     -- "hiera-optim 0.1.0", README,
      item 2 of what optimize(model) does
PyTorch supplies device memory and the current stream only.
"""
from __future__ import annotations

import ctypes as C
import os

from . import _build

__all__ = ["build", "lib", "premix_fwd", "premix_bwd_dx", "premix_bwd_dw", "premix_bwd", "mha_fwd",
           "mha_bwd", "mha_bwd_workspace_bytes",
           "mu_gather", "mu_scatter", "device_error", "IHAError", "Strides", "MASK_NONE",
           "MASK_CAUSAL", "MASK_CAUSAL_WINDOW", "F32", "BF16"]

IHA_OK, IHA_ERR_INVALID_ARG, IHA_ERR_UNSUPPORTED, IHA_ERR_ALIGNMENT, IHA_ERR_CUDA = range(5)
F32, BF16 = 0, 1
MASK_NONE, MASK_CAUSAL, MASK_CAUSAL_WINDOW = 0, 1, 2

SYMBOLS = ("iha_premix_fwd", "iha_premix_bwd_dx", "iha_premix_bwd_dw", "iha_premix_bwd",
           "mha_fwd", "mu_gather", "mu_scatter", "iha_status_string", "iha_last_error",
           "iha_device_error", "iha_test_fail_next_wait", "mha_bwd", "mha_bwd_workspace_bytes",
           "mha_bwd_noalloc", "iha_premix_fwd_qkv", "mu_attention_fused",
           "iha_premix_fwd_qkv_interleaved", "iha_premix_bwd_qkv", "mha_fwd_qpool")


class IHAError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status} ({detail})")
        self.status = status


class Strides(C.Structure):
    """Element strides (b_outer, b_inner, seq, head) of a [Bo, Bi, N, Hh, d] view."""
    _fields_ = [("b_outer", C.c_int64), ("b_inner", C.c_int64), ("seq", C.c_int64),
                ("head", C.c_int64)]


_lib = None


def build(force: bool = False) -> str:
    """Compile libiha.so for sm_103a (in-tree)."""
    return _build.build(force=force)


def lib() -> C.CDLL:
    """The loaded C-ABI library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"{_build.LIB} is missing: run transformer_attention_iha_gb300.build()")
    L = C.CDLL(_build.LIB)
    vp, i, f = C.c_void_p, C.c_int, C.c_float
    L.iha_premix_fwd.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    L.iha_premix_fwd_qkv.argtypes = [vp] * 9 + [i, i, i, i, i, i, i, f, vp]
    L.iha_premix_fwd_qkv_interleaved.argtypes = [vp] * 9 + [i, i, i, i, i, i, i, f, vp]
    L.iha_premix_bwd_dx.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    L.iha_premix_bwd_dw.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    L.iha_premix_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    L.mha_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, Strides, Strides, Strides,
                          Strides, f, i, i, i, vp]
    L.mha_bwd_workspace_bytes.argtypes = [i, i, i, i]
    L.mha_bwd_workspace_bytes.restype = C.c_size_t
    L.mha_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, C.c_size_t, i, i, i, i, f, i,
                          i, i, vp]
    L.mha_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp]
    L.mha_bwd_noalloc.restype = C.c_int
    L.mu_gather.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, i, vp]
    L.mu_scatter.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, i, vp]
    L.mu_attention_fused.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    L.iha_premix_bwd_qkv.argtypes = [vp] * 15 + [i, i, i, i, i, i, i, f, vp]
    L.mha_fwd_qpool.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, Strides, Strides, Strides,
                                Strides, f, i, vp]
    for name in ("iha_premix_fwd", "iha_premix_fwd_qkv", "iha_premix_fwd_qkv_interleaved",
                 "iha_premix_bwd_dx",
                 "iha_premix_bwd_dw", "iha_premix_bwd", "mha_fwd", "mha_bwd", "mu_gather",
                 "mu_scatter", "mu_attention_fused", "iha_premix_bwd_qkv", "mha_fwd_qpool"):
        getattr(L, name).restype = C.c_int
    L.iha_status_string.argtypes = [i]
    L.iha_status_string.restype = C.c_char_p
    L.iha_last_error.argtypes = []
    L.iha_last_error.restype = C.c_char_p
    L.iha_device_error.argtypes = [i]
    L.iha_device_error.restype = C.c_int
    L.iha_test_fail_next_wait.argtypes = [i]
    L.iha_test_fail_next_wait.restype = C.c_int
    _lib = L
    return L


def check(status: int, where: str) -> None:
    if status != IHA_OK:
        L = lib()
        detail = L.iha_last_error().decode() or L.iha_status_string(status).decode()
        raise IHAError(status, where, detail)


def device_error(clear: bool = True) -> int:
    """Device error word (0 = none); synchronises the device."""
    return int(lib().iha_device_error(int(clear)))


# ---------------------------------------------------------------- torch helpers
def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _dt(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return C.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


def _expect(t, name: str, shape=None, dtype=None, device=None, contiguous: bool = True):
    """Host-side argument check: raises before anything reaches the library."""
    if not t.is_cuda:
        raise ValueError(f"{name}: must live on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


# ---------------------------------------------------------------- premix
def premix_fwd(x, w, P: int, rope: bool = False, rope_base: float = 10000.0, out=None,
               stream=None):
    """Y[B,N,H*P,d] = premix of X[B,N,H,d] with W[H,P,H] (fp32), optional RoPE."""
    torch = _torch()
    _expect(x, "x")
    if x.dim() != 4:
        raise ValueError("x must be [B, N, H, d]")
    B, N, H, d = x.shape
    _expect(w, "w", (H, P, H), torch.float32, x.device)
    if out is None:
        out = torch.empty((B, N, H * P, d), dtype=x.dtype, device=x.device)
    _expect(out, "out", (B, N, H * P, d), x.dtype, x.device)
    check(lib().iha_premix_fwd(_ptr(x), _ptr(w), _ptr(out), B, N, H, P, d, _dt(x), int(rope),
                               float(rope_base), _stream(stream)), "iha_premix_fwd")
    return out


def premix_fwd_qkv(xs, ws, P: int, rope: bool = False, rope_base: float = 10000.0, out=None,
                   stream=None):
    """(Y_q, Y_k, Y_v) = premix of (X_q, X_k, X_v) with (W_q, W_k, W_v) in one
    launch; RoPE (when rope) on Q and K only."""
    torch = _torch()
    if len(xs) != 3 or len(ws) != 3:
        raise ValueError("xs and ws must hold three tensors (q, k, v)")
    x0 = xs[0]
    _expect(x0, "xq")
    if x0.dim() != 4:
        raise ValueError("x must be [B, N, H, d]")
    B, N, H, d = x0.shape
    for t, (x, w) in enumerate(zip(xs, ws)):
        _expect(x, f"x[{t}]", (B, N, H, d), x0.dtype, x0.device)
        _expect(w, f"w[{t}]", (H, P, H), torch.float32, x0.device)
    if out is None:
        out = tuple(torch.empty((B, N, H * P, d), dtype=x0.dtype, device=x0.device)
                    for _ in range(3))
    if len(out) != 3:
        raise ValueError("out must hold three tensors")
    for t, y in enumerate(out):
        _expect(y, f"out[{t}]", (B, N, H * P, d), x0.dtype, x0.device)
    check(lib().iha_premix_fwd_qkv(*(_ptr(x) for x in xs), *(_ptr(w) for w in ws),
                                   *(_ptr(y) for y in out), B, N, H, P, d, _dt(x0), int(rope),
                                   float(rope_base), _stream(stream)), "iha_premix_fwd_qkv")
    return tuple(out)


def premix_fwd_qkv_interleaved(xs, ws, P: int, rope: bool = False, rope_base: float = 10000.0,
                               out=None, stream=None):
    """(Y_q, Y_k, Y_v) as [B, N, P, H, d]: the premix of (X_q, X_k, X_v) with
    rows ordered p * H + h (the interleaved pseudo-token layout); RoPE on Q, K."""
    torch = _torch()
    if len(xs) != 3 or len(ws) != 3:
        raise ValueError("xs and ws must hold three tensors (q, k, v)")
    x0 = xs[0]
    _expect(x0, "xq")
    if x0.dim() != 4:
        raise ValueError("x must be [B, N, H, d]")
    B, N, H, d = x0.shape
    for t, (x, w) in enumerate(zip(xs, ws)):
        _expect(x, f"x[{t}]", (B, N, H, d), x0.dtype, x0.device)
        _expect(w, f"w[{t}]", (H, P, H), torch.float32, x0.device)
    if out is None:
        out = tuple(torch.empty((B, N, P, H, d), dtype=x0.dtype, device=x0.device)
                    for _ in range(3))
    if len(out) != 3:
        raise ValueError("out must hold three tensors")
    for t, y in enumerate(out):
        _expect(y, f"out[{t}]", (B, N, P, H, d), x0.dtype, x0.device)
    check(lib().iha_premix_fwd_qkv_interleaved(*(_ptr(x) for x in xs), *(_ptr(w) for w in ws),
                                               *(_ptr(y) for y in out), B, N, H, P, d, _dt(x0),
                                               int(rope), float(rope_base), _stream(stream)),
          "iha_premix_fwd_qkv_interleaved")
    return tuple(out)


def premix_bwd_dx(dy, w, rope: bool = False, rope_base: float = 10000.0, out=None,
                  stream=None):
    """dX[B,N,H,d] = W^T dY (with the inverse RoPE when rope)."""
    torch = _torch()
    _expect(w, "w", dtype=torch.float32)
    if w.dim() != 3 or w.shape[0] != w.shape[2]:
        raise ValueError("w must be [H, P, H]")
    H, P, _ = w.shape
    _expect(dy, "dy", device=w.device)
    if dy.dim() != 4 or dy.shape[2] != H * P:
        raise ValueError(f"dy must be [B, N, H*P={H * P}, d], got {tuple(dy.shape)}")
    B, N, _, d = dy.shape
    if out is None:
        out = torch.empty((B, N, H, d), dtype=dy.dtype, device=dy.device)
    _expect(out, "out", (B, N, H, d), dy.dtype, dy.device)
    check(lib().iha_premix_bwd_dx(_ptr(dy), _ptr(w), _ptr(out), B, N, H, P, d, _dt(dy),
                                  int(rope), float(rope_base), _stream(stream)),
          "iha_premix_bwd_dx")
    return out


def premix_bwd_dw(dy, x, P: int, rope: bool = False, rope_base: float = 10000.0, out=None,
                  stream=None):
    """dW[H,P,H] (fp32, overwritten) = sum over tokens and features of dY X^T."""
    torch = _torch()
    _expect(x, "x")
    if x.dim() != 4:
        raise ValueError("x must be [B, N, H, d]")
    B, N, H, d = x.shape
    _expect(dy, "dy", (B, N, H * P, d), x.dtype, x.device)
    if out is None:
        out = torch.empty((H, P, H), dtype=torch.float32, device=x.device)
    _expect(out, "out", (H, P, H), torch.float32, x.device)
    check(lib().iha_premix_bwd_dw(_ptr(dy), _ptr(x), _ptr(out), B, N, H, P, d, _dt(x),
                                  int(rope), float(rope_base), _stream(stream)),
          "iha_premix_bwd_dw")
    return out


def premix_bwd(dy, x, w, rope: bool = False, rope_base: float = 10000.0, dx=None, dw=None,
               stream=None):
    """(dX, dW) in one pass over dY: dX = W^T dY (inverse RoPE when rope), dW = sum dY X^T."""
    torch = _torch()
    _expect(x, "x")
    if x.dim() != 4:
        raise ValueError("x must be [B, N, H, d]")
    B, N, H, d = x.shape
    if w.dim() != 3:
        raise ValueError("w must be [H, P, H]")
    P = w.shape[1]
    _expect(w, "w", (H, P, H), torch.float32, x.device)
    _expect(dy, "dy", (B, N, H * P, d), x.dtype, x.device)
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty((H, P, H), dtype=torch.float32, device=x.device)
    _expect(dx, "dx", (B, N, H, d), x.dtype, x.device)
    _expect(dw, "dw", (H, P, H), torch.float32, x.device)
    check(lib().iha_premix_bwd(_ptr(dy), _ptr(x), _ptr(w), _ptr(dx), _ptr(dw), B, N, H, P, d,
                               _dt(x), int(rope), float(rope_base), _stream(stream)),
          "iha_premix_bwd")
    return dx, dw


def premix_bwd_qkv(dys, xs, ws, rope: bool = False, rope_base: float = 10000.0, dxs=None,
                   dws=None, stream=None):
    """((dX_q, dX_k, dX_v), (dW_q, dW_k, dW_v)) of the three premixes in one
    backward launch; inverse RoPE (when rope) on Q and K only."""
    torch = _torch()
    if len(dys) != 3 or len(xs) != 3 or len(ws) != 3:
        raise ValueError("dys, xs and ws must hold three tensors (q, k, v)")
    x0 = xs[0]
    _expect(x0, "xq")
    if x0.dim() != 4:
        raise ValueError("x must be [B, N, H, d]")
    B, N, H, d = x0.shape
    if ws[0].dim() != 3:
        raise ValueError("w must be [H, P, H]")
    P = ws[0].shape[1]
    for t in range(3):
        _expect(xs[t], f"x[{t}]", (B, N, H, d), x0.dtype, x0.device)
        _expect(ws[t], f"w[{t}]", (H, P, H), torch.float32, x0.device)
        _expect(dys[t], f"dy[{t}]", (B, N, H * P, d), x0.dtype, x0.device)
    if dxs is None:
        dxs = tuple(torch.empty_like(x0) for _ in range(3))
    if dws is None:
        dws = tuple(torch.empty((H, P, H), dtype=torch.float32, device=x0.device)
                    for _ in range(3))
    if len(dxs) != 3 or len(dws) != 3:
        raise ValueError("dxs and dws must hold three tensors")
    for t in range(3):
        _expect(dxs[t], f"dx[{t}]", (B, N, H, d), x0.dtype, x0.device)
        _expect(dws[t], f"dw[{t}]", (H, P, H), torch.float32, x0.device)
    check(lib().iha_premix_bwd_qkv(*(_ptr(t) for t in dys), *(_ptr(t) for t in xs),
                                   *(_ptr(t) for t in ws), *(_ptr(t) for t in dxs),
                                   *(_ptr(t) for t in dws), B, N, H, P, d, _dt(x0), int(rope),
                                   float(rope_base), _stream(stream)), "iha_premix_bwd_qkv")
    return tuple(dxs), tuple(dws)


# ---------------------------------------------------------------- attention
def _as5(t):
    """View a [B, N, Hh, d] or [Bo, Bi, N, Hh, d] tensor as 5-D (no copy)."""
    if t.dim() == 4:
        return t.unsqueeze(1)
    if t.dim() == 5:
        return t
    raise ValueError("attention tensors must be [B,N,Hh,d] or [Bo,Bi,N,Hh,d]")


def _strides(t5) -> Strides:
    s = t5.stride()
    if s[4] != 1:
        raise ValueError("the head dimension must be dense")
    return Strides(s[0], s[1], s[2], s[3])


def mha_fwd(q, k, v, mask: int = MASK_NONE, window: int = 0, scale: float = 0.0, out=None,
            lse=None, return_lse: bool = False, stream=None):
    """Softmax attention over [B,N,Hh,d] or [Bo,Bi,N,Hh,d] views (strided allowed).

    Returns O shaped like q (dense unless `out` is given); with return_lse,
    also lse [Bo, Bi, Hh, Nq] fp32 (natural log, scale included).
    """
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _expect(t, name, dtype=q.dtype, device=q.device, contiguous=False)
    q5, k5, v5 = _as5(q), _as5(k), _as5(v)
    Bo, Bi, Nq, Hh, d = q5.shape
    Nk = k5.shape[2]
    if tuple(k5.shape) != (Bo, Bi, Nk, Hh, d) or tuple(v5.shape) != (Bo, Bi, Nk, Hh, d):
        raise ValueError(f"k {tuple(k5.shape)} / v {tuple(v5.shape)} do not match q "
                         f"{tuple(q5.shape)}")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    _expect(out, "out", q.shape, q.dtype, q.device, contiguous=False)
    o5 = _as5(out)
    if lse is None and return_lse:
        lse = torch.empty((Bo, Bi, Hh, Nq), dtype=torch.float32, device=q.device)
    if lse is not None:
        if lse.numel() != Bo * Bi * Hh * Nq:
            raise ValueError(f"lse: {lse.numel()} elements, expected [Bo, Bi, Hh, Nq] = "
                             f"{(Bo, Bi, Hh, Nq)}")
        _expect(lse, "lse", dtype=torch.float32, device=q.device)
    check(lib().mha_fwd(_ptr(q5), _ptr(k5), _ptr(v5), _ptr(o5),
                        C.c_void_p(lse.data_ptr() if lse is not None else 0), Bo, Bi, Hh, Nq,
                        Nk, d, _strides(q5), _strides(k5), _strides(v5), _strides(o5),
                        float(scale), int(mask), int(window), _dt(q), _stream(stream)),
          "mha_fwd")
    return (out, lse) if return_lse else out


def mha_fwd_qpool(q, k, v, q_stride: int, scale: float = 0.0, out=None, lse=None,
                  return_lse: bool = False, stream=None):
    """Mask-unit attention with Hiera's pooled queries: q, k, v are [Bo,Bi,T,Hh,d]
    (or [B,T,Hh,d]) bf16 views; the T query rows are max-pooled over q_stride
    blocks (block index slow) inside the kernel.  Returns O [Bo,Bi,T/q_stride,Hh,d]
    (4-D in, 4-D out); with return_lse, also lse [Bo, Bi, Hh, T/q_stride]."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _expect(t, name, q.shape, q.dtype, q.device, contiguous=False)
    q5, k5, v5 = _as5(q), _as5(k), _as5(v)
    Bo, Bi, T, Hh, d = q5.shape
    if q_stride <= 0 or T % q_stride:
        raise ValueError(f"q_stride {q_stride} must divide T = {T}")
    Tq = T // q_stride
    oshape = tuple(q.shape[:-3]) + (Tq, Hh, d)
    if out is None:
        out = torch.empty(oshape, dtype=q.dtype, device=q.device)
    _expect(out, "out", oshape, q.dtype, q.device, contiguous=False)
    o5 = _as5(out)
    if lse is None and return_lse:
        lse = torch.empty((Bo, Bi, Hh, Tq), dtype=torch.float32, device=q.device)
    if lse is not None:
        if lse.numel() != Bo * Bi * Hh * Tq:
            raise ValueError(f"lse: {lse.numel()} elements, expected {(Bo, Bi, Hh, Tq)}")
        _expect(lse, "lse", dtype=torch.float32, device=q.device)
    check(lib().mha_fwd_qpool(_ptr(q5), _ptr(k5), _ptr(v5), _ptr(o5),
                              C.c_void_p(lse.data_ptr() if lse is not None else 0), Bo, Bi, Hh,
                              T, d, int(q_stride), _strides(q5), _strides(k5), _strides(v5),
                              _strides(o5), float(scale), _dt(q), _stream(stream)),
          "mha_fwd_qpool")
    return (out, lse) if return_lse else out


def mha_bwd_workspace_bytes(B: int, Hh: int, N: int, d: int) -> int:
    """Bytes of device scratch mha_bwd needs for [B, N, Hh, d] tensors."""
    return int(lib().mha_bwd_workspace_bytes(B, Hh, N, d))


def mha_bwd(q, k, v, o, dout, lse, mask: int = MASK_NONE, window: int = 0, scale: float = 0.0,
            dq=None, dk=None, dv=None, workspace=None, stream=None):
    """(dQ, dK, dV) of attention over dense [B, N, Hh, d] bf16 tensors, given the
    forward's output o and lse [B, Hh, N] (or [B, 1, Hh, N]) fp32 and the upstream
    gradient dout.  `workspace` (uint8 CUDA tensor of mha_bwd_workspace_bytes) is
    allocated here when not given."""
    torch = _torch()
    _expect(q, "q", dtype=torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, N, Hh, d]")
    B, N, Hh, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _expect(t, name, (B, N, Hh, d), torch.bfloat16, q.device)
    if lse.numel() != B * Hh * N:
        raise ValueError(f"lse: {lse.numel()} elements, expected [B, Hh, N] = {(B, Hh, N)}")
    _expect(lse, "lse", dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _expect(t, name, (B, N, Hh, d), torch.bfloat16, q.device)
    need = mha_bwd_workspace_bytes(B, Hh, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _expect(workspace, "workspace", dtype=torch.uint8, device=q.device)
    check(lib().mha_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                        _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, Hh, N, d,
                        float(scale), int(mask), int(window), _dt(q), _stream(stream)),
          "mha_bwd")
    return dq, dk, dv


# ---------------------------------------------------------------- gather / scatter
def _mu_check(x, keep, grid_h: int, grid_w: int, mu_h: int, mu_w: int):
    torch = _torch()
    _expect(x, "x")
    if x.dim() != 3 or x.shape[1] != grid_h * grid_w:
        raise ValueError(f"x must be [B, grid_h*grid_w={grid_h * grid_w}, C], got "
                         f"{tuple(x.shape)}")
    _expect(keep, "keep", dtype=torch.int32, device=x.device)
    if keep.dim() != 2 or keep.shape[0] != x.shape[0]:
        raise ValueError(f"keep must be [B={x.shape[0]}, n_keep] int32, got {tuple(keep.shape)}")


def mu_gather(x, keep, grid_h: int, grid_w: int, mu_h: int, mu_w: int, out=None, stream=None):
    """x [B, grid_h*grid_w, C] -> [B, n_keep, mu_h*mu_w, C] (bit-exact copy)."""
    torch = _torch()
    _mu_check(x, keep, grid_h, grid_w, mu_h, mu_w)
    B, G, Cc = x.shape
    n_keep = keep.shape[1]
    if out is None:
        out = torch.empty((B, n_keep, mu_h * mu_w, Cc), dtype=x.dtype, device=x.device)
    _expect(out, "out", (B, n_keep, mu_h * mu_w, Cc), x.dtype, x.device)
    check(lib().mu_gather(_ptr(x), _ptr(keep), _ptr(out), B, grid_h, grid_w, mu_h, mu_w, n_keep,
                          Cc, x.element_size(), _stream(stream)), "mu_gather")
    return out


def mu_attention_fused(x, keep, canvas, grid_h: int, grid_w: int, mu_h: int, mu_w: int,
                       scale: float = 0.0, stream=None):
    """Gather -> mask-unit attention (Q = K = V = the unit's tokens) -> scatter
    into `canvas` (in place; tokens of units not kept are untouched)."""
    torch = _torch()
    _mu_check(x, keep, grid_h, grid_w, mu_h, mu_w)
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bfloat16")
    B, G, Cc = x.shape
    _expect(canvas, "canvas", (B, G, Cc), x.dtype, x.device)
    check(lib().mu_attention_fused(_ptr(x), _ptr(keep), _ptr(canvas), B, grid_h, grid_w, mu_h,
                                   mu_w, keep.shape[1], Cc, float(scale), BF16, _stream(stream)),
          "mu_attention_fused")
    return canvas


def mu_scatter(src, keep, x, grid_h: int, grid_w: int, mu_h: int, mu_w: int, stream=None):
    """In place: x[b, tok(keep[b,k], t), :] = src[b, k, t, :]."""
    _mu_check(x, keep, grid_h, grid_w, mu_h, mu_w)
    B, G, Cc = x.shape
    n_keep = keep.shape[1]
    _expect(src, "src", (B, n_keep, mu_h * mu_w, Cc), x.dtype, x.device)
    check(lib().mu_scatter(_ptr(src), _ptr(keep), _ptr(x), B, grid_h, grid_w, mu_h, mu_w, n_keep,
                           Cc, x.element_size(), _stream(stream)), "mu_scatter")
    return x
