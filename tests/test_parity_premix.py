"""GPU parity: premix forward / input gradient / weight gradient vs the oracle.

Small shapes run the whole oracle (several blocks and a ragged tail); the
LLaMA-2.4B layer shape (B=1, N=8192, H=20, P=4, d=128) checks sampled token
windows for the forward and input gradient and the full weight gradient; the
long-context shape (B=2, N=16384) checks RoPE at late positions.
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from helpers import (assert_bf16_close, assert_dw_close, assert_f32_close, dw_abs_sum, dw_chain,
                     to_dev, to_f64)

pytestmark = pytest.mark.gpu

SHAPES = [  # (B, N, H, P, d)
    (2, 37, 20, 4, 128),
    (1, 5, 4, 2, 32),
    (3, 9, 3, 3, 64),
    (1, 33, 7, 5, 96),
    (2, 17, 32, 4, 16),
    (1, 3, 1, 1, 8),
]

# Edges of the tensor-core kernels' range (bf16, d in {64, 128}, H <= 32,
# H*P <= 128): full M = 128 tiles, padded pseudo-head counts, K = 32 source
# heads, and small H*P at d = 128 (one or two 16-row K-steps of dY).
TC_EDGE_SHAPES = [  # (B, N, H, P, d)
    (1, 19, 24, 4, 128),   # H*P = 96
    (1, 19, 32, 4, 128),   # H*P = 128, H = 32
    (1, 23, 16, 8, 128),   # H*P = 128, P = 8
    (1, 23, 19, 5, 128),   # H*P = 95 (padded to 96), P = 5
    (2, 11, 24, 5, 64),    # H*P = 120, d = 64
    (1, 13, 32, 4, 64),    # H*P = 128, d = 64
    (2, 21, 4, 4, 128),    # H*P = 16
    (1, 25, 12, 4, 128),   # H*P = 48
    (1, 9, 4, 2, 128),     # H*P = 8
    (1, 7, 1, 1, 128),     # H = P = 1
]


@pytest.fixture(scope="module")
def T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_iha_gb300 as T
    T.lib()
    return T


def _inputs(B, N, H, P, d, seed, dtype="bf16"):
    x = S.normal((B, N, H, d), seed, 0, dtype=dtype)
    dy = S.normal((B, N, H * P, d), seed, 1, dtype=dtype)
    w = S.premix_weight(H, P, seed, 2)
    return x, dy, w


def _rope_ok(d):
    return d >= 16 and d <= 128 and (d & (d - 1)) == 0


def _check_all_ops(T, shape, rope, seed, base=100.0):
    B, N, H, P, d = shape
    x, dy, w = _inputs(B, N, H, P, d, seed=seed)
    y = T.premix_fwd(to_dev(x), to_dev(w), P, rope=rope, rope_base=base)
    assert_bf16_close(to_f64(y), O.premix_fwd(x, w, P, rope=rope, rope_base=base), "fwd")
    rdx = O.premix_bwd_dx(dy, w, rope=rope, rope_base=base)
    dx = T.premix_bwd_dx(to_dev(dy), to_dev(w), rope=rope, rope_base=base)
    assert_bf16_close(to_f64(dx), rdx, "dx")
    dw = T.premix_bwd_dw(to_dev(dy), to_dev(x), P, rope=rope, rope_base=base)
    absum = dw_abs_sum(dy, x, P, rope)
    chain = dw_chain(B, N, H, P, d, rope=rope)
    rdw = O.premix_bwd_dw(dy, x, P, rope=rope, rope_base=base)
    assert_dw_close(to_f64(dw), rdw, absum, chain, rope, "dw")
    # both gradients from one pass over dY
    dx2, dw2 = T.premix_bwd(to_dev(dy), to_dev(x), to_dev(w), rope=rope, rope_base=base)
    assert_bf16_close(to_f64(dx2), rdx, "fused dx")
    assert_dw_close(to_f64(dw2), rdw, absum, chain, rope, "fused dw")
    assert T.device_error() == 0


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("rope", [False, True])
def test_premix_bf16_small(T, shape, rope):
    if rope and not _rope_ok(shape[4]):
        pytest.skip("RoPE needs d a power of two")
    _check_all_ops(T, shape, rope, seed=11 + shape[4])


@pytest.mark.parametrize("shape", TC_EDGE_SHAPES)
@pytest.mark.parametrize("rope", [False, True])
def test_premix_bf16_tensor_core_edges(T, shape, rope):
    _check_all_ops(T, shape, rope, seed=3 + shape[2] * shape[3])


def _check_qkv_fwd(T, shape, rope, seed, dtype="bf16", base=100.0):
    """Q, K, V in one launch: every tensor against the oracle (RoPE on Q and K
    only), and bit-equal to its own single-tensor launch."""
    B, N, H, P, d = shape
    xs = [S.normal((B, N, H, d), seed, 10 + t, dtype=dtype) for t in range(3)]
    ws = [S.premix_weight(H, P, seed, 20 + t) for t in range(3)]
    ys = T.premix_fwd_qkv([to_dev(x) for x in xs], [to_dev(w) for w in ws], P, rope=rope,
                          rope_base=base)
    for t, (x, w, y) in enumerate(zip(xs, ws, ys)):
        r = O.premix_fwd(x, w, P, rope=rope and t < 2, rope_base=base)
        if dtype == "bf16":
            assert_bf16_close(to_f64(y), r, f"qkv fwd tensor {t}")
        else:
            assert_f32_close(to_f64(y), r, f"qkv fwd tensor {t}")
        one = T.premix_fwd(to_dev(x), to_dev(w), P, rope=rope and t < 2, rope_base=base)
        assert bool((one.view(-1) == y.view(-1)).all()), f"tensor {t}: differs from its own launch"
    assert T.device_error() == 0


@pytest.mark.parametrize("shape", SHAPES[:3] + TC_EDGE_SHAPES)
@pytest.mark.parametrize("rope", [False, True])
def test_premix_qkv_fwd_one_launch(T, shape, rope):
    if rope and not _rope_ok(shape[4]):
        pytest.skip("RoPE needs d a power of two")
    _check_qkv_fwd(T, shape, rope, seed=5 + shape[1])


def _check_qkv_bwd(T, shape, rope, seed, base=100.0):
    """Q, K, V backward in one launch: every tensor's dX and dW against the
    oracle (inverse RoPE on Q and K only); dX bit-equal to the tensor's own
    single-tensor backward (dW sums in a different atomic order)."""
    B, N, H, P, d = shape
    xs = [S.normal((B, N, H, d), seed, 30 + t) for t in range(3)]
    dys = [S.normal((B, N, H * P, d), seed, 40 + t) for t in range(3)]
    ws = [S.premix_weight(H, P, seed, 50 + t) for t in range(3)]
    dxs, dws = T.premix_bwd_qkv([to_dev(a) for a in dys], [to_dev(a) for a in xs],
                                [to_dev(a) for a in ws], rope=rope, rope_base=base)
    for t in range(3):
        r = rope and t < 2
        rdx = O.premix_bwd_dx(dys[t], ws[t], rope=r, rope_base=base)
        assert_bf16_close(to_f64(dxs[t]), rdx, f"qkv dx tensor {t}")
        rdw = O.premix_bwd_dw(dys[t], xs[t], P, rope=r, rope_base=base)
        assert_dw_close(to_f64(dws[t]), rdw, dw_abs_sum(dys[t], xs[t], P, r),
                        dw_chain(B, N, H, P, d, rope=r), r, f"qkv dw tensor {t}")
        dx1, _ = T.premix_bwd(to_dev(dys[t]), to_dev(xs[t]), to_dev(ws[t]), rope=r,
                              rope_base=base)
        assert bool((dx1.view(-1) == dxs[t].view(-1)).all()), f"tensor {t}: dx differs"
    assert T.device_error() == 0


@pytest.mark.parametrize("shape", SHAPES[:3] + TC_EDGE_SHAPES)
@pytest.mark.parametrize("rope", [False, True])
def test_premix_qkv_bwd_one_launch(T, shape, rope):
    if rope and not _rope_ok(shape[4]):
        pytest.skip("RoPE needs d a power of two")
    _check_qkv_bwd(T, shape, rope, seed=7 + shape[1])


def test_premix_qkv_bwd_llama_shape(T):
    """B=1, N=8192, H=20, P=4, d=128, RoPE on Q and K, one backward launch:
    dX on token windows at the start, middle and end, every full dW."""
    sh = S.LLAMA_PREMIX
    B, N, H, P, d = sh.B, sh.N, sh.H, sh.P, sh.d
    xs = [S.normal((B, N, H, d), 4, 30 + t) for t in range(3)]
    dys = [S.normal((B, N, H * P, d), 4, 40 + t) for t in range(3)]
    ws = [S.premix_weight(H, P, 4, 50 + t) for t in range(3)]
    dxs, dws = T.premix_bwd_qkv([to_dev(a) for a in dys], [to_dev(a) for a in xs],
                                [to_dev(a) for a in ws], rope=True, rope_base=S.ROPE_BASE)
    for t in range(3):
        r = t < 2
        dx = to_f64(dxs[t])
        for n0 in (0, 4093, N - 131):
            sl = slice(n0, n0 + 131)
            rdx = O.premix_bwd_dx(dys[t][:, sl], ws[t], rope=r, rope_base=S.ROPE_BASE, pos0=n0)
            assert_bf16_close(dx[:, sl], rdx, f"tensor {t} dx@{n0}")
        rdw = O.premix_bwd_dw(dys[t], xs[t], P, rope=r, rope_base=S.ROPE_BASE)
        assert_dw_close(to_f64(dws[t]), rdw, dw_abs_sum(dys[t], xs[t], P, r),
                        dw_chain(B, N, H, P, d, rope=r), r, f"tensor {t} dw full")
    assert T.device_error() == 0


def test_premix_qkv_fwd_f32_tiny_layer(T):
    sh = S.TINY
    _check_qkv_fwd(T, (sh.B, sh.N, sh.H, sh.P, sh.d), True, seed=9, dtype="f32")


def test_premix_qkv_fwd_llama_shape_sampled(T):
    """B=1, N=8192, H=20, P=4, d=128 in one launch: sampled token windows of
    each tensor against the oracle (positions enter through RoPE)."""
    import torch
    B, N, H, P, d = 1, 8192, 20, 4, 128
    xs = [S.normal((B, N, H, d), 31, t) for t in range(3)]
    ws = [S.premix_weight(H, P, 31, 10 + t) for t in range(3)]
    ys = T.premix_fwd_qkv([to_dev(x) for x in xs], [to_dev(w) for w in ws], P, rope=True)
    torch.cuda.synchronize()
    for n0 in (0, 4093, N - 64):
        for t in range(3):
            r = O.premix_fwd(np.ascontiguousarray(xs[t][:, n0:n0 + 64]), ws[t], P, rope=t < 2,
                             pos0=n0)
            assert_bf16_close(to_f64(ys[t][:, n0:n0 + 64]), r, f"qkv llama tensor {t} @{n0}")
    assert T.device_error() == 0


@pytest.mark.parametrize("rope", [False, True])
def test_premix_f32_tiny_layer(T, rope):
    """fp32 path at the tiny-layer shape (B=1, N=128, H=4, P=2, d=32): 1e-5."""
    sh = S.TINY
    x, dy, w = _inputs(sh.B, sh.N, sh.H, sh.P, sh.d, seed=0, dtype="f32")
    y = T.premix_fwd(to_dev(x), to_dev(w), sh.P, rope=rope)
    assert_f32_close(to_f64(y), O.premix_fwd(x, w, sh.P, rope=rope), "fwd f32")
    dx = T.premix_bwd_dx(to_dev(dy), to_dev(w), rope=rope)
    assert_f32_close(to_f64(dx), O.premix_bwd_dx(dy, w, rope=rope), "dx f32")
    dw = T.premix_bwd_dw(to_dev(dy), to_dev(x), sh.P, rope=rope)
    r = O.premix_bwd_dw(dy, x, sh.P, rope=rope)
    # fp32 reduction over B*N*d = 4096 products of N(0,1) values
    assert_f32_close(to_f64(dw), r, "dw f32", tol=1e-5 * max(1.0, float(np.abs(r).max())))


def test_premix_llama_shape_sampled(T):
    """B=1, N=8192, H=20, P=4, d=128 (the bench shape): token windows at the
    start, middle and end for fwd / dx; the full dW."""
    sh = S.LLAMA_PREMIX
    x, dy, w = _inputs(sh.B, sh.N, sh.H, sh.P, sh.d, seed=0)
    y = to_f64(T.premix_fwd(to_dev(x), to_dev(w), sh.P))
    dx = to_f64(T.premix_bwd_dx(to_dev(dy), to_dev(w)))
    for n0 in (0, 4093, sh.N - 131):
        sl = slice(n0, n0 + 131)
        assert_bf16_close(y[:, sl], O.premix_fwd(x[:, sl], w, sh.P), f"fwd@{n0}")
        assert_bf16_close(dx[:, sl], O.premix_bwd_dx(dy[:, sl], w), f"dx@{n0}")
    dw = to_f64(T.premix_bwd_dw(to_dev(dy), to_dev(x), sh.P))
    absum = dw_abs_sum(dy, x, sh.P)
    chain = dw_chain(sh.B, sh.N, sh.H, sh.P, sh.d)
    rdw = O.premix_bwd_dw(dy, x, sh.P)
    assert_dw_close(dw, rdw, absum, chain, False, "dw full")
    dx2, dw2 = T.premix_bwd(to_dev(dy), to_dev(x), to_dev(w))
    dx2 = to_f64(dx2)
    for n0 in (0, sh.N - 131):
        sl = slice(n0, n0 + 131)
        assert_bf16_close(dx2[:, sl], O.premix_bwd_dx(dy[:, sl], w), f"fused dx@{n0}")
    assert_dw_close(to_f64(dw2), rdw, absum, chain, False, "fused dw full")


def test_premix_long_context_rope_sampled(T):
    """B=2, N=16384 with RoPE (base 10000): windows near the end of each
    sequence, where angles are largest."""
    sh = S.LONG_CTX
    x = S.normal((sh.B, sh.N, sh.H, sh.d), 5, 0)
    w = S.premix_weight(sh.H, sh.P, 5, 1)
    y = to_f64(T.premix_fwd(to_dev(x), to_dev(w), sh.P, rope=True, rope_base=S.ROPE_BASE))
    for n0 in (0, 9001, sh.N - 67):
        sl = slice(n0, n0 + 67)
        ref = O.premix_fwd(x[:, sl], w, sh.P, rope=True, rope_base=S.ROPE_BASE, pos0=n0)
        assert_bf16_close(y[:, sl], ref, f"fwd rope@{n0}")
    dy = S.normal((sh.B, sh.N, sh.HP, sh.d), 5, 2)
    dx = to_f64(T.premix_bwd_dx(to_dev(dy), to_dev(w), rope=True, rope_base=S.ROPE_BASE))
    dx2, dw2 = T.premix_bwd(to_dev(dy), to_dev(x), to_dev(w), rope=True, rope_base=S.ROPE_BASE)
    dx2 = to_f64(dx2)
    for n0 in (0, sh.N - 67):
        sl = slice(n0, n0 + 67)
        ref = O.premix_bwd_dx(dy[:, sl], w, rope=True, rope_base=S.ROPE_BASE, pos0=n0)
        assert_bf16_close(dx[:, sl], ref, f"dx rope@{n0}")
        assert_bf16_close(dx2[:, sl], ref, f"fused dx rope@{n0}")
    # dW with RoPE at this size: the full oracle reduction over 32768 tokens
    assert_dw_close(to_f64(dw2), O.premix_bwd_dw(dy, x, sh.P, rope=True, rope_base=S.ROPE_BASE),
                    dw_abs_sum(dy, x, sh.P, True), dw_chain(sh.B, sh.N, sh.H, sh.P, sh.d, rope=True),
                    True, "fused dw rope")


def test_premix_one_hot_copies_are_bit_exact(T):
    """One-hot W makes every pseudo-head an exact copy of a source head."""
    B, N, H, P, d = 2, 19, 5, 3, 64
    x = S.normal((B, N, H, d), 3, 0)
    w = np.zeros((H, P, H), np.float32)
    for h in range(H):
        for p in range(P):
            w[h, p, (2 * h + p) % H] = 1.0
    y = T.premix_fwd(to_dev(x), to_dev(w), P)
    yb = y.view(__import__("torch").int16).cpu().numpy().view(np.uint16)
    for h in range(H):
        for p in range(P):
            np.testing.assert_array_equal(yb[:, :, h * P + p], x[:, :, (2 * h + p) % H])


def test_premix_rejects_bad_args(T):
    import torch
    x = torch.zeros((1, 4, 3, 10), dtype=torch.bfloat16, device="cuda")   # d % 8 != 0
    w = torch.zeros((3, 2, 3), dtype=torch.float32, device="cuda")
    with pytest.raises(T.IHAError) as e:
        T.premix_fwd(x, w, 2)
    assert e.value.status == 2
    x = torch.zeros((1, 4, 33, 16), dtype=torch.bfloat16, device="cuda")  # H > 32
    w = torch.zeros((33, 1, 33), dtype=torch.float32, device="cuda")
    with pytest.raises(T.IHAError):
        T.premix_fwd(x, w, 1)
    assert T.device_error() == 0
