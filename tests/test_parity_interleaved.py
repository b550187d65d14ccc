"""GPU parity: the joint-softmax (interleaved pseudo-token) variant of the
IHA layer.  The premix writes [B, N, P, H, d] (pseudo-token n*P + p of head
h); mha_fwd attends over the [B, N*P, H, d] view of it in place, causal on
n*P + p.  Each stage against the oracle, and the premix bit-equal to the
head-major premix reordered."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from helpers import assert_bf16_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

SHAPES = [  # (B, N, H, P, d)
    (1, 37, 20, 4, 128),
    (2, 19, 8, 2, 64),
    (1, 23, 24, 5, 128),   # H*P = 120
]


@pytest.fixture(scope="module")
def T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_iha_gb300 as T
    T.lib()
    return T


def _bits(t):
    import torch
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("rope", [False, True])
def test_interleaved_premix(T, shape, rope):
    B, N, H, P, d = shape
    xs = [S.normal((B, N, H, d), 41 + N, t) for t in range(3)]
    ws = [S.premix_weight(H, P, 41 + N, 10 + t) for t in range(3)]
    ys = T.premix_fwd_qkv_interleaved([to_dev(x) for x in xs], [to_dev(w) for w in ws], P,
                                      rope=rope, rope_base=100.0)
    head_major = T.premix_fwd_qkv([to_dev(x) for x in xs], [to_dev(w) for w in ws], P, rope=rope,
                                  rope_base=100.0)
    for t in range(3):
        r = O.interleave_heads(O.premix_fwd(xs[t], ws[t], P, rope=rope and t < 2,
                                            rope_base=100.0), H, P)
        assert_bf16_close(to_f64(ys[t]), r, f"interleaved premix tensor {t}")
        hm = _bits(head_major[t]).reshape(B, N, H * P, d)
        np.testing.assert_array_equal(_bits(ys[t]), O.interleave_heads(hm, H, P))
    assert T.device_error() == 0


@pytest.mark.parametrize("shape", SHAPES[:2])
def test_joint_attention_over_interleaved_pseudo_tokens(T, shape):
    """mha_fwd over the [B, N*P, H, d] view (strides of the interleaved
    premix output), causal on n*P + p, against the oracle's joint attention
    on the same bf16 inputs."""
    import torch
    B, N, H, P, d = shape
    xs = [S.normal((B, N, H, d), 51 + N, t) for t in range(3)]
    ws = [S.premix_weight(H, P, 51 + N, 10 + t) for t in range(3)]
    yq, yk, yv = T.premix_fwd_qkv_interleaved([to_dev(x) for x in xs], [to_dev(w) for w in ws], P,
                                              rope=True)
    view = lambda y: y.view(B, N * P, H, d)
    o, lse = T.mha_fwd(view(yq), view(yk), view(yv), mask=T.MASK_CAUSAL, return_lse=True)
    torch.cuda.synchronize()
    ro, rl = O.joint_attention(_bits(yq), _bits(yk), _bits(yv), causal=True)
    assert_bf16_close(to_f64(o).reshape(B, N, P, H, d), ro, "joint attention")
    np.testing.assert_allclose(lse.cpu().numpy().reshape(B, H, N * P), rl, rtol=0, atol=2e-3)
    assert T.device_error() == 0


def test_joint_attention_llama_shape_sampled(T):
    """B=1, N=2048, H=20, P=4, d=128: 8192 pseudo-tokens per head, causal;
    sampled query rows against the oracle."""
    import torch
    B, N, H, P, d = 1, 2048, 20, 4, 128
    xs = [S.normal((B, N, H, d), 61, t) for t in range(3)]
    ws = [S.premix_weight(H, P, 61, 10 + t) for t in range(3)]
    ys = T.premix_fwd_qkv_interleaved([to_dev(x) for x in xs], [to_dev(w) for w in ws], P,
                                      rope=True)
    yq, yk, yv = (y.view(B, N * P, H, d) for y in ys)
    o = T.mha_fwd(yq, yk, yv, mask=T.MASK_CAUSAL)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    M = N * P
    m = np.concatenate([[0, 1, M - 1], rng.integers(0, M, 29)])
    h = rng.integers(0, H, m.size)
    rows = np.stack([np.zeros_like(m), np.zeros_like(m), h, m], axis=1).astype(np.int64)
    qb, kb, vb = (_bits(y).reshape(B, 1, M, H, d) for y in (yq, yk, yv))
    ro, _ = O.attention_rows(qb, kb, vb, rows, O.MASK_CAUSAL, 0)
    got = to_f64(o)[0][m, h]
    assert_bf16_close(got, ro, "joint attention rows")
    assert T.device_error() == 0
