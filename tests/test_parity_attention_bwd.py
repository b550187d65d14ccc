"""GPU parity: attention backward (dQ, dK, dV) vs the oracle.

The forward runs on the GPU (its O and LSE feed the backward, as in a training
step); the oracle recomputes everything from Q, K, V and dO in float64.
Small shapes run the whole oracle (several key and query tiles, ragged tails,
every mask mode, d from 16 to 128); the pseudo-head window shape (80 heads,
N=4096, W=1024) checks three heads in full.  Tolerance: the bf16 rule widened
by the rounding of the bf16 MMA operands dS and P (helpers.assert_grad_close)."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from helpers import assert_grad_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_iha_gb300 as T
    T.lib()
    return T


def _run(T, B, N, Hh, d, mask, window, seed):
    q, k, v, g = (S.normal((B, N, Hh, d), seed, c) for c in range(4))
    qd, kd, vd, gd = (to_dev(a) for a in (q, k, v, g))
    o, lse = T.mha_fwd(qd, kd, vd, mask=mask, window=window, return_lse=True)
    dq, dk, dv = T.mha_bwd(qd, kd, vd, o, gd, lse, mask=mask, window=window)
    assert T.device_error() == 0
    return (q, k, v, g), (dq, dk, dv)


CASES = [  # (B, N, Hh, d, mask, window)
    (1, 300, 2, 128, O.MASK_CAUSAL, 0),
    (2, 257, 3, 64, O.MASK_NONE, 0),
    (1, 300, 2, 128, O.MASK_CAUSAL_WINDOW, 129),
    (1, 130, 4, 32, O.MASK_CAUSAL_WINDOW, 40),
    (1, 64, 1, 128, O.MASK_NONE, 0),
    (2, 513, 2, 128, O.MASK_CAUSAL, 0),
    (1, 200, 2, 96, O.MASK_NONE, 0),
    (1, 100, 2, 16, O.MASK_CAUSAL, 0),
    (1, 384, 3, 128, O.MASK_CAUSAL_WINDOW, 1),
    (1, 1, 1, 128, O.MASK_CAUSAL, 0),
]


@pytest.mark.parametrize("case", CASES)
def test_attention_bwd_small(T, case):
    B, N, Hh, d, mask, window = case
    (q, k, v, g), (dq, dk, dv) = _run(T, B, N, Hh, d, mask, window, seed=N + d + mask)
    rq, rk, rv = O.attention_bwd(q, k, v, g, mask, window)
    aq, ak, av = O.attention_bwd(q, k, v, g, mask, window, absolute=True)
    assert_grad_close(to_f64(dv), rv, av, N, f"dV {case}")
    assert_grad_close(to_f64(dk), rk, ak, N, f"dK {case}")
    assert_grad_close(to_f64(dq), rq, aq, N, f"dQ {case}")


def test_attention_bwd_dv_sum_identity(T):
    """sum_j dV_j = sum_i dO_i per head (rows of P sum to 1), on the GPU result."""
    (q, k, v, g), (dq, dk, dv) = _run(T, 1, 700, 3, 128, O.MASK_CAUSAL, 0, seed=5)
    lhs = to_f64(dv).sum(axis=1)
    rhs = S.bf16_bits_to_f32(g).astype(np.float64).sum(axis=1)
    np.testing.assert_allclose(lhs, rhs, atol=0.05 * np.sqrt(700))


def test_attention_bwd_pseudo_head_window_three_heads(T):
    """80 pseudo-heads, N=4096, d=128, window W=1024: heads 0, 41 and 79 in full."""
    sh, W = S.LLAMA_WINDOW, S.WINDOW_KEYS
    (q, k, v, g), (dq, dk, dv) = _run(T, sh.B, sh.N, sh.HP, sh.d, O.MASK_CAUSAL_WINDOW, W, seed=2)
    for h in (0, 41, 79):
        sl = (slice(None), slice(None), slice(h, h + 1))
        args = [np.ascontiguousarray(a[sl]) for a in (q, k, v, g)]
        rq, rk, rv = O.attention_bwd(*args, O.MASK_CAUSAL_WINDOW, W)
        aq, ak, av = O.attention_bwd(*args, O.MASK_CAUSAL_WINDOW, W, absolute=True)
        assert_grad_close(to_f64(dv[sl]), rv, av, sh.N, f"dV head {h}")
        assert_grad_close(to_f64(dk[sl]), rk, ak, sh.N, f"dK head {h}")
        assert_grad_close(to_f64(dq[sl]), rq, aq, sh.N, f"dQ head {h}")


def test_attention_bwd_rejects_bad_args(T):
    import torch
    q = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 8), dtype=torch.float32, device="cuda")
    L = T.lib()
    need = T.mha_bwd_workspace_bytes(1, 2, 8, 64)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = [torch.empty_like(q) for _ in range(3)]
    p = lambda t: t.data_ptr()
    # workspace too small
    assert L.mha_bwd(p(q), p(q), p(q), p(q), p(q), p(lse), *(p(t) for t in outs), p(ws), need - 1,
                     1, 2, 8, 64, 0.0, 1, 0, 1, None) == 1
    # d not a multiple of 16
    assert L.mha_bwd(p(q), p(q), p(q), p(q), p(q), p(lse), *(p(t) for t in outs), p(ws), need,
                     1, 2, 8, 40, 0.0, 1, 0, 1, None) == 2
    # an output aliasing an input
    assert L.mha_bwd(p(q), p(q), p(q), p(q), p(q), p(lse), p(q), p(outs[1]), p(outs[2]), p(ws),
                     need, 1, 2, 8, 64, 0.0, 1, 0, 1, None) == 1
    assert T.device_error() == 0


def test_attention_bwd_work_counter_slots_are_reused(T):
    """The backward's items (one key tile of one head) past the first wave
    come from a per-launch counter that the last CTA resets: 300 launches on
    two streams (every slot of the 256-entry counter table taken more than
    once) must reproduce the first launch's dK and dV bit for bit (each key
    tile's dK / dV is summed by one CTA in a fixed order) and its dQ to
    rounding (dQ is added by reductions in whatever order CTAs finish)."""
    import torch
    B, N, Hh, d, mask, window = 2, 1030, 48, 128, O.MASK_CAUSAL_WINDOW, 300
    q, k, v, g = (S.normal((B, N, Hh, d), 31, c) for c in range(4))
    qd, kd, vd, gd = (to_dev(a) for a in (q, k, v, g))
    o, lse = T.mha_fwd(qd, kd, vd, mask=mask, window=window, return_lse=True)
    dq0, dk0, dv0 = T.mha_bwd(qd, kd, vd, o, gd, lse, mask=mask, window=window)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [tuple(torch.empty_like(dq0) for _ in range(3)) for _ in range(2)]
    wss = [torch.empty(T.mha_bwd_workspace_bytes(B, Hh, N, d), dtype=torch.uint8, device="cuda")
           for _ in range(2)]
    for n in range(300):
        with torch.cuda.stream(streams[n & 1]):
            dq, dk, dv = outs[n & 1]
            T.mha_bwd(qd, kd, vd, o, gd, lse, mask=mask, window=window, dq=dq, dk=dk, dv=dv,
                      workspace=wss[n & 1])
        if n % 60 == 59 or n >= 298:
            torch.cuda.synchronize()
            for dq, dk, dv in outs:
                assert torch.equal(dk, dk0) and torch.equal(dv, dv0), f"launch {n}"
                # one bf16 ulp at most (2^-7 relative): the fp32 sums differ in order only
                diff = (dq.float() - dq0.float()).abs()
                assert bool((diff <= 2.0 ** -7 * dq0.float().abs() + 1e-6).all()), f"launch {n}"
    torch.cuda.synchronize()
    assert T.device_error() == 0
