"""GPU parity: the tiny IHA layer forward end to end (fp32): premix Q, K, V into
8 pseudo-heads, then unmasked softmax attention with scale 1/sqrt(d) — against
the oracle chain at 1e-5."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from helpers import assert_f32_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def test_tiny_iha_layer_forward_f32():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_iha_gb300 as T
    sh = S.TINY
    xs = [S.normal((sh.B, sh.N, sh.H, sh.d), 0, c, dtype="f32") for c in range(3)]
    ws = [S.premix_weight(sh.H, sh.P, 0, 10 + c) for c in range(3)]
    ys = [T.premix_fwd(to_dev(x), to_dev(w), sh.P) for x, w in zip(xs, ws)]
    o, lse = T.mha_fwd(*ys, return_lse=True)
    ry = [O.premix_fwd(x, w, sh.P) for x, w in zip(xs, ws)]
    for g, r in zip(ys, ry):
        assert_f32_close(to_f64(g), r, "premix")
    # the oracle attention consumes the oracle premix, rounded to fp32 storage
    r32 = [r.astype(np.float32)[:, None] for r in ry]
    ro, rl = O.attention(*r32)
    assert_f32_close(to_f64(o), ro[:, 0], "attention")
    assert_f32_close(to_f64(lse)[:, 0], rl[:, 0], "lse")
    assert T.device_error() == 0
