"""GPU parity: attention forward (tcgen05 bf16 path and fp32 path) vs the oracle.

Small cases run the full oracle: several query / key tiles, ragged tails,
every mask mode, window edges (1, 127, 128, 129, N), head dims 32 / 64 / 96 /
128, Nq != Nk, and Hiera's (T outer, units inner) strided layout.  The
pseudo-head window shape (80 heads, N=4096, W=1024) and the long-context
causal shape (B=2, N=16384) check sampled rows, including the first and last
rows and rows at the window edge.
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from helpers import assert_bf16_close, assert_f32_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_iha_gb300 as T
    T.lib()
    return T


def _qkv(shape_q, shape_k, seed, dtype="bf16"):
    q = S.normal(shape_q, seed, 0, dtype=dtype)
    k = S.normal(shape_k, seed, 1, dtype=dtype)
    v = S.normal(shape_k, seed, 2, dtype=dtype)
    return q, k, v


def _lse_close(g, r, what):
    r = np.asarray(r)
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: lse finiteness differs"
    m = float(np.abs(g[fin] - r[fin]).max(initial=0.0))
    assert m <= 2e-3, f"{what}: lse max abs {m}"


CASES = [  # (B, N, Hh, d, mask, window)
    (1, 300, 3, 128, O.MASK_NONE, 0),
    (1, 300, 3, 128, O.MASK_CAUSAL, 0),
    (2, 300, 2, 128, O.MASK_CAUSAL_WINDOW, 1),
    (1, 300, 2, 128, O.MASK_CAUSAL_WINDOW, 127),
    (1, 300, 2, 128, O.MASK_CAUSAL_WINDOW, 128),
    (1, 300, 2, 128, O.MASK_CAUSAL_WINDOW, 129),
    (1, 300, 2, 128, O.MASK_CAUSAL_WINDOW, 300),
    (1, 513, 2, 64, O.MASK_CAUSAL, 0),
    (1, 200, 2, 96, O.MASK_NONE, 0),
    (1, 130, 4, 32, O.MASK_CAUSAL_WINDOW, 40),
    (1, 64, 1, 96, O.MASK_NONE, 0),
    (1, 1, 1, 128, O.MASK_CAUSAL, 0),
    (3, 257, 1, 16, O.MASK_CAUSAL, 0),
]


@pytest.mark.parametrize("case", CASES)
def test_attention_bf16_small(T, case):
    B, N, Hh, d, mask, window = case
    q, k, v = _qkv((B, N, Hh, d), (B, N, Hh, d), seed=N + d + mask)
    o, lse = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), mask=mask, window=window,
                       return_lse=True)
    ro, rl = O.attention(q[:, None], k[:, None], v[:, None], mask, window)
    assert_bf16_close(to_f64(o), ro[:, 0], f"O {case}")
    _lse_close(to_f64(lse)[:, 0], rl[:, 0], f"lse {case}")
    assert T.device_error() == 0


# Several work items per persistent CTA (more items than SMs), an odd number
# of query tiles (the last item has one tile), heads spread over groups.
MANY_ITEM_CASES = [  # (B, N, Hh, d, mask, window)
    (2, 1030, 48, 128, O.MASK_CAUSAL_WINDOW, 300),
    (1, 1100, 40, 128, O.MASK_CAUSAL, 0),
    (3, 390, 64, 64, O.MASK_NONE, 0),
]


@pytest.mark.parametrize("case", MANY_ITEM_CASES)
def test_attention_bf16_many_items_per_cta(T, case):
    B, N, Hh, d, mask, window = case
    q, k, v = _qkv((B, N, Hh, d), (B, N, Hh, d), seed=N + Hh)
    o, lse = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), mask=mask, window=window,
                       return_lse=True)
    ro, rl = O.attention(q[:, None], k[:, None], v[:, None], mask, window)
    assert_bf16_close(to_f64(o), ro[:, 0], f"O {case}")
    _lse_close(to_f64(lse)[:, 0], rl[:, 0], f"lse {case}")
    assert T.device_error() == 0


# Short sequences (Nq == Nk <= 64, no mask) take the packed kernel: two
# sequences per 128-row tile.  Edges: fewer than 64 tokens, d not a multiple
# of 16, an odd number of sequences (the last tile has one), several heads.
SHORT_CASES = [  # (Bo, Bi, T, Hh, d)
    (3, 1, 49, 2, 96),
    (1, 7, 64, 1, 128),
    (5, 1, 1, 3, 64),
    (2, 3, 33, 1, 40),
    (1, 1, 64, 1, 96),
    (4, 2, 64, 3, 16),
]


@pytest.mark.parametrize("case", SHORT_CASES)
def test_attention_bf16_short_sequences_packed(T, case):
    Bo, Bi, Tn, Hh, d = case
    q, k, v = _qkv((Bo, Bi, Tn, Hh, d), (Bo, Bi, Tn, Hh, d), seed=Tn + d + Hh)
    o, lse = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), return_lse=True)
    ro, rl = O.attention(q, k, v)
    assert_bf16_close(to_f64(o), ro, f"O {case}")
    _lse_close(to_f64(lse), rl, f"lse {case}")
    assert T.device_error() == 0


def test_attention_bf16_nq_ne_nk(T):
    q, _, _ = _qkv((2, 200, 3, 128), (2, 333, 3, 128), seed=7)
    _, k, v = _qkv((2, 333, 3, 128), (2, 333, 3, 128), seed=8)
    o, lse = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), return_lse=True)
    ro, rl = O.attention(q[:, None], k[:, None], v[:, None])
    assert_bf16_close(to_f64(o), ro[:, 0], "O nq!=nk")
    _lse_close(to_f64(lse)[:, 0], rl[:, 0], "lse nq!=nk")


def test_attention_bf16_hiera_layout_in_place(T):
    """Hiera's qkv(x).view(B, T, nw, 3, H, D) read in place: batch = (b, unit),
    seq stride = nw * 3 * H * D, no permute copies."""
    import torch
    B, Tn, nw, H, D = 2, 64, 5, 2, 96
    tok = S.normal((B, Tn, nw, 3, H, D), 9, 0)
    t = to_dev(tok)
    q, k, v = (t[:, :, :, c].permute(0, 2, 1, 3, 4) for c in range(3))   # [B, nw, T, H, D]
    o = T.mha_fwd(q, k, v)
    views = [tok[:, :, :, c].transpose(0, 2, 1, 3, 4) for c in range(3)]
    ro, _ = O.attention(*views)
    assert_bf16_close(to_f64(o), ro, "hiera layout")
    # output written into a strided destination as well
    dst = torch.zeros((B, Tn, nw, H, D), dtype=torch.bfloat16, device="cuda")
    T.mha_fwd(q, k, v, out=dst.permute(0, 2, 1, 3, 4))
    assert_bf16_close(to_f64(dst.permute(0, 2, 1, 3, 4)), ro, "hiera layout, strided out")


def test_attention_bf16_scale_argument(T):
    q, k, v = _qkv((1, 150, 2, 64), (1, 150, 2, 64), seed=10)
    o = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), mask=O.MASK_CAUSAL, scale=0.3)
    ro, _ = O.attention(q[:, None], k[:, None], v[:, None], O.MASK_CAUSAL, scale=0.3)
    assert_bf16_close(to_f64(o), ro[:, 0], "scale 0.3")


def test_attention_zero_query_gives_mean_of_visible_values(T):
    """Q = 0: every visible key gets the same weight (bit-level check of masking)."""
    N, W = 700, 129
    q = np.zeros((1, N, 1, 128), np.uint16)
    _, k, v = _qkv((1, N, 1, 128), (1, N, 1, 128), seed=12)
    o, lse = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), mask=O.MASK_CAUSAL_WINDOW, window=W,
                       return_lse=True)
    vf = S.bf16_bits_to_f32(v).astype(np.float64)[0, :, 0]
    ref = np.stack([vf[max(0, i - W + 1): i + 1].mean(axis=0) for i in range(N)])
    assert_bf16_close(to_f64(o)[0, :, 0], ref, "mean of window")
    cnt = np.minimum(np.arange(N) + 1, W)
    np.testing.assert_allclose(to_f64(lse)[0, 0, 0], np.log(cnt), atol=1e-4)


def test_attention_f32_tiny_layer(T):
    """fp32 path (tiny layer: 8 heads, N=128, d=32, no mask) at 1e-5."""
    for mask, window in [(O.MASK_NONE, 0), (O.MASK_CAUSAL, 0), (O.MASK_CAUSAL_WINDOW, 17)]:
        q, k, v = _qkv((1, 128, 8, 32), (1, 128, 8, 32), seed=0, dtype="f32")
        o, lse = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), mask=mask, window=window,
                           return_lse=True)
        ro, rl = O.attention(q[:, None], k[:, None], v[:, None], mask, window)
        assert_f32_close(to_f64(o), ro[:, 0], f"O f32 mask={mask}")
        assert_f32_close(to_f64(lse)[:, 0], rl[:, 0], f"lse f32 mask={mask}")


def _sample_rows(B, Hh, N, W, n, seed):
    g = np.random.default_rng(seed)
    rows = set()
    for i in (0, 1, 127, 128, 129, W - 1, W, W + 1, N - 129, N - 128, N - 1):
        if 0 <= i < N:
            rows.add((int(g.integers(B)), 0, int(g.integers(Hh)), i))
    while len(rows) < n:
        rows.add((int(g.integers(B)), 0, int(g.integers(Hh)), int(g.integers(N))))
    return np.array(sorted(rows), dtype=np.int64)


def _check_rows(o, lse, q, k, v, rows, mask, window, what):
    ro, rl = O.attention_rows(q[:, None], k[:, None], v[:, None], rows, mask, window)
    og = to_f64(o)
    lg = to_f64(lse)
    got = np.stack([og[b, i, h] for b, _, h, i in rows])
    gl = np.array([lg[b, 0, h, i] for b, _, h, i in rows])
    assert_bf16_close(got, ro, what)
    _lse_close(gl, rl, what)


def test_attention_pseudo_head_window_sampled(T):
    """80 pseudo-heads, N=4096, d=128, causal window W=1024 (fp32 LSE)."""
    sh, W = S.LLAMA_WINDOW, S.WINDOW_KEYS
    q, k, v = _qkv((sh.B, sh.N, sh.HP, sh.d), (sh.B, sh.N, sh.HP, sh.d), seed=0)
    o, lse = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), mask=O.MASK_CAUSAL_WINDOW, window=W,
                       return_lse=True)
    rows = _sample_rows(sh.B, sh.HP, sh.N, W, 192, 1)
    _check_rows(o, lse, q, k, v, rows, O.MASK_CAUSAL_WINDOW, W, "window 1024")


def test_attention_long_context_causal_sampled(T):
    """B=2, 80 pseudo-heads, N=16384, d=128, causal."""
    sh = S.LONG_CTX
    q, k, v = _qkv((sh.B, sh.N, sh.HP, sh.d), (sh.B, sh.N, sh.HP, sh.d), seed=3)
    o, lse = T.mha_fwd(to_dev(q), to_dev(k), to_dev(v), mask=O.MASK_CAUSAL, return_lse=True)
    rows = _sample_rows(sh.B, sh.HP, sh.N, sh.N, 96, 2)
    _check_rows(o, lse, q, k, v, rows, O.MASK_CAUSAL, 0, "causal 16384")


def test_attention_rejects_bad_args(T):
    import torch
    q = torch.zeros((1, 8, 1, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 9, 1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(T.IHAError) as e:
        T.mha_fwd(q, k, k, mask=O.MASK_CAUSAL)            # causal with Nq != Nk
    assert e.value.status == 2
    with pytest.raises(T.IHAError) as e:
        T.mha_fwd(q, q, q, mask=O.MASK_CAUSAL_WINDOW, window=0)
    assert e.value.status == 1
    big = torch.zeros((1, 8, 1, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(T.IHAError) as e:
        T.mha_fwd(big, big, big)
    assert e.value.status == 2
    wide = torch.zeros((1, 8, 3, 64), dtype=torch.bfloat16, device="cuda")[:, :, 1:]  # odd head offset ok
    T.mha_fwd(wide, wide, wide)
    odd = torch.zeros((1, 8, 1, 68), dtype=torch.bfloat16, device="cuda")[..., :64]   # seq stride 68
    with pytest.raises(T.IHAError) as e:
        T.mha_fwd(odd, odd, odd)
    assert e.value.status == 3
    assert T.device_error() == 0


def test_attention_work_counter_slots_are_reused(T):
    """Items past the first wave come from a per-launch counter that the last
    CTA resets: 600 launches (every slot of the counter table taken more than
    twice, on two streams) must all give the first launch's bits, and that
    launch the oracle's values."""
    import torch
    B, N, Hh, d, mask, window = 2, 1030, 48, 128, O.MASK_CAUSAL_WINDOW, 300
    q, k, v = _qkv((B, N, Hh, d), (B, N, Hh, d), seed=21)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    first = T.mha_fwd(qd, kd, vd, mask=mask, window=window)
    ro, _ = O.attention(q[:, None], k[:, None], v[:, None], mask, window)
    assert_bf16_close(to_f64(first), ro[:, 0], "first launch")
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(first) for _ in range(4)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for n in range(600):
        with torch.cuda.stream(streams[n & 1]):
            o = outs[n & 3]
            o.zero_()
            T.mha_fwd(qd, kd, vd, mask=mask, window=window, out=o)
        if n % 50 == 49 or n >= 596:
            torch.cuda.synchronize()
            for t in outs:
                assert torch.equal(t, first), f"launch {n}"
    torch.cuda.synchronize()
    assert T.device_error() == 0


@pytest.mark.parametrize("shape", [(1, 384, 3, 128), (2, 1030, 5, 64), (1, 4096, 4, 128)])
def test_attention_window_one_returns_v_exactly(T, shape):
    """W = 1: each query sees only its own key, the softmax has one term
    (P = 1), so O is V and lse the scaled self-score.  Holds at any size;
    catches a row maximum taken over masked scores (P rounded away from 1,
    O off by a bf16 ulp ~1e-2) that the bf16 tolerance would let through.
    The one allowed difference is the weight a masked key keeps in the
    FMA-pipe exponential, 2^-125 (about 1e-38) instead of 0."""
    import torch
    B, N, Hh, d = shape
    q, k, v = _qkv((B, N, Hh, d), (B, N, Hh, d), seed=N + Hh)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o, lse = T.mha_fwd(qd, kd, vd, mask=O.MASK_CAUSAL_WINDOW, window=1, return_lse=True)
    assert float((o.float() - vd.float()).abs().max()) <= 1e-30
    s = (qd.float() * kd.float()).sum(-1) / np.sqrt(d)          # [B, N, Hh]
    np.testing.assert_allclose(lse[:, 0].cpu().numpy(), s.permute(0, 2, 1).cpu().numpy(),
                               atol=2e-4, rtol=1e-5)
    assert T.device_error() == 0
