"""GPU parity: mask-unit attention with Hiera's pooled queries (q_pool,
"hiera-optim 0.1.0", hiera_optim/attention/mask_unit.py,
MaskUnitAttentionFast.forward with q_stride > 1) against the oracle.

Cases: the stage-2 pooling block of Hiera (T = 64 tokens per unit pooled 4:1,
d = 96, 2 heads) in the in-place (T outer, units inner) layout, ragged and odd
unit counts (the last 128-row tile holds one unit), T < 64, Tq = 1, d in
{16, 32, 64, 96, 128}, and q_stride = 1 against plain attention.
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from helpers import assert_bf16_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_iha_gb300 as T
    T.lib()
    return T


def _lse_close(g, r, what):
    m = float(np.abs(np.asarray(g) - np.asarray(r)).max(initial=0.0))
    assert m <= 2e-3, f"{what}: lse max abs {m}"


CASES = [  # (Bo, Bi, T, Hh, d, q_stride)
    (3, 1, 64, 2, 96, 4),
    (2, 3, 16, 1, 64, 4),
    (1, 5, 64, 1, 128, 2),
    (2, 2, 49, 1, 96, 7),
    (1, 3, 8, 2, 32, 8),
    (3, 3, 64, 1, 16, 16),
    (7, 1, 36, 1, 96, 4),
]


@pytest.mark.parametrize("case", CASES)
def test_qpool_attention_small(T, case):
    Bo, Bi, Tn, Hh, d, qs = case
    seed = Tn + d + qs
    q, k, v = (S.normal((Bo, Bi, Tn, Hh, d), seed, c) for c in range(3))
    o, lse = T.mha_fwd_qpool(to_dev(q), to_dev(k), to_dev(v), qs, return_lse=True)
    ro, rl = O.attention_qpool(q, k, v, qs)
    assert o.shape == (Bo, Bi, Tn // qs, Hh, d)
    assert_bf16_close(to_f64(o), ro, f"O {case}")
    _lse_close(to_f64(lse), rl, f"lse {case}")
    assert T.device_error() == 0


def test_qpool_stride_one_is_plain_short_attention(T):
    q, k, v = (S.normal((4, 3, 64, 2, 96), 17, c) for c in range(3))
    a = T.mha_fwd_qpool(to_dev(q), to_dev(k), to_dev(v), 1)
    b = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v))
    assert bool((a.view(-1) == b.view(-1)).all())


def test_qpool_hiera_pooling_block_in_place(T):
    """Hiera's qkv(x).view(B, T, nw, 3, H, D) read in place (batch = (b,
    unit), seq stride nw * 3 * H * D): T = 64 tokens per unit pooled 4:1 to
    16, two heads of 96; the output written straight into Hiera's
    (B, Tq, nw, H, D) layout (tq slow, unit fast)."""
    import torch
    B, Tn, nw, H, D, qs = 4, 64, 9, 2, 96, 4
    Tq = Tn // qs
    tok = S.normal((B, Tn, nw, 3, H, D), 23, 0)
    t = to_dev(tok)
    q, k, v = (t[:, :, :, c].permute(0, 2, 1, 3, 4) for c in range(3))   # [B, nw, T, H, D]
    dst = torch.zeros((B, Tq, nw, H, D), dtype=torch.bfloat16, device="cuda")
    T.mha_fwd_qpool(q, k, v, qs, out=dst.permute(0, 2, 1, 3, 4))
    views = [tok[:, :, :, c].transpose(0, 2, 1, 3, 4) for c in range(3)]
    ro, _ = O.attention_qpool(*views, qs)
    assert_bf16_close(to_f64(dst.permute(0, 2, 1, 3, 4)), ro, "hiera pooling block")
    assert T.device_error() == 0


def test_qpool_many_units_per_cta(T):
    """More unit pairs than CTAs: stages and TMEM buffers are reused while
    pooled tiles keep arriving (2 x 311 units, odd pair count)."""
    q, k, v = (S.normal((2, 311, 64, 1, 96), 29, c) for c in range(3))
    o = T.mha_fwd_qpool(to_dev(q), to_dev(k), to_dev(v), 4)
    ro, _ = O.attention_qpool(q, k, v, 4)
    assert_bf16_close(to_f64(o), ro, "many units")
    assert T.device_error() == 0


def test_qpool_rejects_bad_args(T):
    import torch
    x = torch.zeros((1, 1, 64, 1, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        T.mha_fwd_qpool(x, x, x, 3)                                 # 3 does not divide 64
    big = torch.zeros((1, 1, 128, 1, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(T.IHAError):
        T.mha_fwd_qpool(big, big, big, 4)                           # T > 64
    f = torch.zeros((1, 1, 64, 1, 96), dtype=torch.float32, device="cuda")
    with pytest.raises(T.IHAError):
        T.mha_fwd_qpool(f, f, f, 4)                                 # bf16 only
