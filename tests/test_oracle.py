"""Pins for the oracle: values and identities fixed by the pages and by the
mathematics, each chosen so a plausible slip (a dropped term, a wrong sign, a
transposed operand, a wrong flattening) fails at least one test.

CPU only (no GPU marker).
"""
import math
import os

import numpy as np
import pytest

import oracle as O
import synthetic as S

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------- premix fwd
def test_premix_hand_example():
    """Hand-computed example from the definition (golden file)."""
    g = {r[0]: np.array([float(t) for t in r[1:]]) for r in _read_rows("premix_hand.txt")}
    x = g["X"].astype(np.float32).reshape(1, 1, 2, 2)
    w = g["W"].astype(np.float32).reshape(2, 2, 2)
    y = O.premix_fwd(x, w, P=2)
    np.testing.assert_array_equal(y.reshape(-1), g["Y"])
    dx = O.premix_bwd_dx(np.ones((1, 1, 4, 2), np.float32), w)
    np.testing.assert_array_equal(dx.reshape(-1), g["DX_ONES"])
    dw = O.premix_bwd_dw(np.ones((1, 1, 4, 2), np.float32), x, P=2)
    np.testing.assert_array_equal(dw.reshape(-1), g["DW_ONES"])


def test_premix_one_hot_copies_heads():
    """W[h,p,s] = [s == sigma(h,p)] makes pseudo-head h*P+p a copy of head sigma."""
    B, N, H, P, d = 2, 5, 5, 3, 8
    x = S.normal((B, N, H, d), seed=1, dtype="f32")
    sigma = lambda h, p: (3 * h + 2 * p + 1) % H
    w = np.zeros((H, P, H), np.float32)
    for h in range(H):
        for p in range(P):
            w[h, p, sigma(h, p)] = 1.0
    y = O.premix_fwd(x, w, P)
    for h in range(H):
        for p in range(P):
            np.testing.assert_array_equal(y[:, :, h * P + p, :], x[:, :, sigma(h, p), :])


def test_premix_identity_P1():
    x = S.normal((1, 7, 4, 16), seed=2, dtype="f32")
    y = O.premix_fwd(x, np.eye(4, dtype=np.float32).reshape(4, 1, 4), 1)
    np.testing.assert_array_equal(y, x)


def test_premix_linear_in_x_and_w():
    B, N, H, P, d = 1, 6, 4, 2, 8
    x1 = S.normal((B, N, H, d), 3, dtype="f32")
    x2 = S.normal((B, N, H, d), 4, dtype="f32")
    w1 = S.premix_weight(H, P, 5, 0)
    w2 = S.premix_weight(H, P, 6, 0)
    a, b = np.float32(0.5), np.float32(-2.0)
    lhs = O.premix_fwd((a * x1 + b * x2).astype(np.float32), w1, P)
    rhs = a * O.premix_fwd(x1, w1, P) + b * O.premix_fwd(x2, w1, P)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-6, atol=1e-6)
    lhs = O.premix_fwd(x1, (a * w1 + b * w2).astype(np.float32), P)
    rhs = a * O.premix_fwd(x1, w1, P) + b * O.premix_fwd(x1, w2, P)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-6, atol=1e-6)


# ----------------------------------------------------------------- premix bwd
@pytest.mark.parametrize("rope", [False, True])
def test_premix_dx_is_adjoint(rope):
    """<dY, premix(X)> == <premix_dx(dY), X> (the chain rule, through RoPE too)."""
    B, N, H, P, d = 2, 9, 5, 3, 16
    x = S.normal((B, N, H, d), 7, dtype="f32")
    dy = S.normal((B, N, H * P, d), 8, dtype="f32")
    w = S.premix_weight(H, P, 9, 0)
    lhs = float(np.sum(dy.astype(np.float64) * O.premix_fwd(x, w, P, rope=rope, rope_base=100.0)))
    rhs = float(np.sum(O.premix_bwd_dx(dy, w, rope=rope, rope_base=100.0) * x.astype(np.float64)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


@pytest.mark.parametrize("rope", [False, True])
def test_premix_dw_matches_difference_quotient(rope):
    """L(W) = <dY, premix_W(X)> is linear in W, so the central difference
    (L(W+E) - L(W-E)) / 2 is dL/dW along E exactly (up to rounding)."""
    B, N, H, P, d = 2, 6, 3, 2, 8
    x = S.normal((B, N, H, d), 10, dtype="f32")
    dy = S.normal((B, N, H * P, d), 11, dtype="f32")
    w = np.zeros((H, P, H))
    dw = O.premix_bwd_dw(dy, x, P, rope=rope, rope_base=50.0)

    def L(wm):
        return float(np.sum(dy.astype(np.float64) *
                            O.premix_fwd(x, wm.astype(np.float32), P, rope=rope, rope_base=50.0)))

    for h in range(H):
        for p in range(P):
            for s in range(H):
                E = np.zeros_like(w)
                E[h, p, s] = 1.0
                # L is linear, so L(W+E) - L(W-E) = L(E) - L(-E) = 2 L(E);
                # evaluating at +-E keeps every weight exact in float32.
                fd = (L(E) - L(-E)) / 2.0
                assert abs(fd - dw[h, p, s]) <= 1e-9 * max(1.0, abs(fd))


def test_premix_dw_pairs_with_forward():
    """<dW, dWdir> == <dY, premix_dWdir(X)> for a random direction."""
    B, N, H, P, d = 1, 11, 4, 3, 8
    x = S.normal((B, N, H, d), 13, dtype="f32")
    dy = S.normal((B, N, H * P, d), 14, dtype="f32")
    dir_ = S.premix_weight(H, P, 15, 0)
    dw = O.premix_bwd_dw(dy, x, P)
    lhs = float(np.sum(dw * dir_.astype(np.float64)))
    rhs = float(np.sum(dy.astype(np.float64) * O.premix_fwd(x, dir_, P)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


# ----------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity_and_pairs_keep_norm():
    x = S.normal((1, 6, 3, 16), 20, dtype="f32").astype(np.float64)
    y = O.rope(x, base=10000.0)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])
    half = 8
    nx = x[..., :half] ** 2 + x[..., half:] ** 2
    ny = y[..., :half] ** 2 + y[..., half:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12)
    np.testing.assert_allclose(O.rope(y, base=10000.0, inverse=True), x, atol=1e-12)


def test_rope_d2_rotates_by_position():
    """d = 2: inv_freq_0 = base^0 = 1, so position n rotates (1, 0) by n radians."""
    x = np.zeros((1, 4, 1, 2))
    x[..., 0] = 1.0
    y = O.rope(x, base=123.0)
    for n in range(4):
        np.testing.assert_allclose(y[0, n, 0], [math.cos(n), math.sin(n)], atol=1e-15)


def test_rope_equals_complex_multiplication():
    """Rotate-half RoPE == multiplying z_i = x_i + i*x_{i+d/2} by exp(i*n*base^(-2i/d))."""
    N, d, base = 9, 12, 500.0
    x = S.normal((1, N, 2, d), 21, dtype="f32").astype(np.float64)
    y = O.rope(x, base=base)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    theta = np.arange(N)[:, None] * base ** (-2.0 * np.arange(d // 2) / d)[None, :]
    zr = z * np.exp(1j * theta)[None, :, None, :]
    np.testing.assert_allclose(y[..., : d // 2], zr.real, atol=1e-12)
    np.testing.assert_allclose(y[..., d // 2:], zr.imag, atol=1e-12)


def test_rope_commutes_with_premix():
    """Premix mixes heads, RoPE mixes features: R(M X) == M(R X)."""
    B, N, H, P, d = 2, 7, 3, 2, 8
    x = S.normal((B, N, H, d), 22, dtype="f32")
    w = S.premix_weight(H, P, 23, 0)
    fused = O.premix_fwd(x, w, P, rope=True, rope_base=1000.0)
    after = O.rope(O.premix_fwd(x, w, P), base=1000.0)
    before = O.premix_fwd(O.rope(x.astype(np.float64), base=1000.0).astype(np.float32), w, P)
    np.testing.assert_allclose(fused, after, atol=1e-12)
    np.testing.assert_allclose(fused, before, atol=1e-5)   # x rounded to f32 after RoPE


# ----------------------------------------------------------------- attention
def _qkv(Bo, Bi, N, Hh, d, seed, Nk=None):
    Nk = N if Nk is None else Nk
    q = S.normal((Bo, Bi, N, Hh, d), seed, 0, dtype="f32")
    k = S.normal((Bo, Bi, Nk, Hh, d), seed, 1, dtype="f32")
    v = S.normal((Bo, Bi, Nk, Hh, d), seed, 2, dtype="f32")
    return q, k, v


def _visible_count(i, N, mask, window):
    if mask == 0:
        return N
    if mask == 1:
        return i + 1
    return min(i + 1, window)


@pytest.mark.parametrize("mask,window", [(0, 0), (1, 0), (2, 5), (2, 1)])
def test_attention_zero_query_is_mean_of_visible_values(mask, window):
    q, k, v = _qkv(1, 2, 17, 2, 8, 30)
    q[:] = 0
    o, lse = O.attention(q, k, v, mask, window)
    for i in range(17):
        lo = 0 if mask == 0 else (0 if mask == 1 else max(0, i - window + 1))
        hi = 17 if mask == 0 else i + 1
        np.testing.assert_allclose(o[:, :, i], v[:, :, lo:hi].astype(np.float64).mean(axis=2),
                                   atol=1e-12)
        np.testing.assert_allclose(lse[..., i], math.log(_visible_count(i, 17, mask, window)),
                                   atol=1e-12)


def test_attention_window_one_returns_own_value():
    q, k, v = _qkv(2, 1, 13, 3, 16, 31)
    o, lse = O.attention(q, k, v, O.MASK_CAUSAL_WINDOW, 1)
    np.testing.assert_array_equal(o, v.astype(np.float64))
    dots = np.einsum("abnhd,abnhd->abhn", q.astype(np.float64), k.astype(np.float64))
    np.testing.assert_allclose(lse, dots / 4.0, atol=1e-12)


def test_attention_causal_first_row_is_first_value():
    q, k, v = _qkv(1, 1, 9, 2, 8, 32)
    o, _ = O.attention(q, k, v, O.MASK_CAUSAL)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0].astype(np.float64))


def test_attention_none_is_invariant_to_key_permutation():
    q, k, v = _qkv(1, 1, 11, 2, 8, 33)
    perm = np.random.default_rng(0).permutation(11)
    o1, l1 = O.attention(q, k, v)
    o2, l2 = O.attention(q, np.ascontiguousarray(k[:, :, perm]), np.ascontiguousarray(v[:, :, perm]))
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


@pytest.mark.parametrize("mask,window,Nq,Nk", [(0, 0, 9, 14), (1, 0, 12, 12), (2, 4, 12, 12),
                                               (2, 100, 12, 12)])
def test_attention_matches_library_sdpa(mask, window, Nq, Nk):
    """Brute force against torch's float64 CPU SDPA with an explicit boolean mask,
    and lse against scipy's logsumexp of the masked scores."""
    torch = pytest.importorskip("torch")
    from scipy.special import logsumexp
    Bo, Bi, Hh, d = 2, 3, 2, 8
    q, k, v = _qkv(Bo, Bi, Nq, Hh, d, 34, Nk=Nk)
    o, lse = O.attention(q, k, v, mask, window)
    tq = torch.from_numpy(q.astype(np.float64)).permute(0, 1, 3, 2, 4)   # [Bo,Bi,Hh,N,d]
    tk = torch.from_numpy(k.astype(np.float64)).permute(0, 1, 3, 2, 4)
    tv = torch.from_numpy(v.astype(np.float64)).permute(0, 1, 3, 2, 4)
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    if mask == 0:
        allowed = torch.ones(Nq, Nk, dtype=torch.bool)
    elif mask == 1:
        allowed = j <= i
    else:
        allowed = (j <= i) & (i - j < window)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=allowed)
    np.testing.assert_allclose(o, ref.permute(0, 1, 3, 2, 4).numpy(), atol=1e-12)
    scores = (tq @ tk.transpose(-1, -2)).numpy() / math.sqrt(d)
    scores = np.where(allowed.numpy(), scores, -np.inf)
    np.testing.assert_allclose(lse, logsumexp(scores, axis=-1), atol=1e-12)


def test_attention_strided_views_match_dense():
    """Hiera's (T outer, nw inner) token layout read in place equals the dense copy."""
    B, T, nw, Hh, d = 2, 6, 3, 2, 8
    tok = S.normal((B, T, nw, 3, Hh, d), 35, dtype="f32")        # qkv(x).view(B,T,nw,3,H,D)
    views = [tok[:, :, :, c].transpose(0, 2, 1, 3, 4) for c in range(3)]   # [B, nw, T, H, d]
    dense = [np.ascontiguousarray(vw) for vw in views]
    o1, l1 = O.attention(*views)
    o2, l2 = O.attention(*dense)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_attention_rows_match_full():
    q, k, v = _qkv(2, 1, 21, 3, 8, 36)
    o, lse = O.attention(q, k, v, O.MASK_CAUSAL_WINDOW, 6)
    rows = np.array([[0, 0, 0, 0], [1, 0, 2, 20], [0, 0, 1, 7], [1, 0, 0, 5]])
    orow, lrow = O.attention_rows(q, k, v, rows, O.MASK_CAUSAL_WINDOW, 6)
    for r, (bo, bi, h, i) in enumerate(rows):
        np.testing.assert_array_equal(orow[r], o[bo, bi, i, h])
        assert lrow[r] == lse[bo, bi, h, i]


# ----------------------------------------------------------------- tile visits
def test_tile_matched_window_table():
    """The page's tile-matched WSL column follows from counting 128x128 KV-tile
    visits over H*P pseudo-heads of length N (window W = WSL + 1) against MHA
    causal over H heads: WSL = max(N/(2P) - 1, smallest WSL matching MHA)."""
    H, P = 20, 4
    for N, formula, matched in [tuple(int(t) for t in r) for r in _read_rows("wsl_table.txt")]:
        assert formula == N // (2 * P) - 1
        mha = O.tile_visits(N, H, O.MASK_CAUSAL, 0)
        visits = lambda wsl: O.tile_visits(N, H * P, O.MASK_CAUSAL_WINDOW, wsl + 1)
        lo, hi = 0, N
        while lo < hi:                      # visits are non-decreasing in WSL
            mid = (lo + hi) // 2
            if visits(mid) >= mha:
                hi = mid
            else:
                lo = mid + 1
        assert max(formula, lo) == matched, (N, lo, matched)


def test_tile_visits_small_brute_force():
    """Against a per-pair enumeration on small sizes."""
    for N, tq, tk, mask, window in [(37, 8, 8, 1, 0), (37, 8, 4, 2, 5), (16, 4, 4, 0, 0),
                                    (50, 16, 8, 2, 17)]:
        count = 0
        for a in range(0, N, tq):
            for b in range(0, N, tk):
                hit = False
                for i in range(a, min(a + tq, N)):
                    for j in range(b, min(b + tk, N)):
                        ok = mask == 0 or (j <= i and (mask == 1 or i - j < window))
                        hit |= ok
                count += hit
        assert O.tile_visits(N, 3, mask, window, tq, tk) == 3 * count


# ----------------------------------------------------------------- gather / scatter
def test_mu_index_map_4x4():
    rows = [[int(t) for t in r] for r in _read_rows("mu_index_4x4.txt")]
    x = np.arange(16, dtype=np.int32).reshape(1, 16, 1)
    keep = np.array([[0, 1, 2, 3]], np.int32)
    g = O.mu_gather(x, keep, 4, 4, 2, 2)
    for r in rows:
        assert list(g[0, r[0], :, 0]) == r[1:]


def test_mu_scatter_inverts_gather_and_leaves_rest():
    sh = S.MaskUnitShape(B=3, grid_h=16, grid_w=24, mu_h=4, mu_w=8, n_keep=5, C=6)
    x = S.normal((sh.B, sh.grid_h * sh.grid_w, sh.C), 40, dtype="bf16")
    keep = S.keep_units(sh.B, sh.n_units, sh.n_keep, 41)
    g = O.mu_gather(x, keep, sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w)
    canvas = np.full_like(x, 0x7FC0)                    # bf16 NaN pattern as "untouched"
    s = O.mu_scatter(g, keep, canvas, sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w)
    kept = s != 0x7FC0
    np.testing.assert_array_equal(s[kept], x[kept])
    # exactly n_keep * unit_tokens tokens per sample were written
    assert int(kept[..., 0].sum()) == sh.B * sh.n_keep * sh.unit_tokens
    np.testing.assert_array_equal(O.mu_gather(s, keep, sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w), g)


def test_keep_units_sorted_unique():
    keep = S.keep_units(128, 49, 20, 0)
    assert keep.shape == (128, 20)
    for row in keep:
        assert list(row) == sorted(set(row.tolist())) and 0 <= row.min() and row.max() < 49


# ----------------------------------------------------------------- bf16 rounding
def test_round_bf16_hand_ties():
    """Round-to-nearest-even onto the bf16 grid (8 significand bits): values
    between two neighbours go to the nearer one; exact halves go to the one
    with an even last significand bit."""
    u = 2.0 ** -7                       # bf16 ulp on [1, 2)
    cases = [
        (1.0, 1.0),
        (1.0 + u / 2, 1.0),             # tie, 1.0 is even -> stays
        (1.0 + 3 * u / 2, 1.0 + 2 * u),  # tie between odd 1+u and even 1+2u
        (1.0 + u / 2 + 2.0 ** -20, 1.0 + u),  # just above the tie -> up
        (1.0 + u / 2 - 2.0 ** -20, 1.0),      # just below the tie -> down
        (-(1.0 + 3 * u / 2), -(1.0 + 2 * u)),  # sign symmetric
        (3.0 + 2.0 ** -7, 3.0),         # ulp on [2, 4) is 2^-6: tie, 3.0 even
        (0.0, 0.0),
        (2.0 ** -130, 2.0 ** -130),     # subnormal with few bits is exact
        (255.5, 256.0),                 # ulp 1 on [128, 256): tie to even 256
        (254.5, 254.0),                 # tie to even 254
        (1e30, None),                   # large value, checked by bits below
    ]
    got = O.round_bf16(np.array([c[0] for c in cases]))
    for (x, want), g in zip(cases[:-1], got[:-1]):
        assert g == want, (x, g, want)
    # 1e30: checked against the bit pattern rounded by hand (no tie)
    f = int(np.array(1e30, np.float32).view(np.uint32))
    want = np.array((f + 0x8000) & 0xFFFF0000, np.uint32).view(np.float32)
    assert got[-1] == float(want)


def test_round_bf16_matches_torch_cast():
    """Cross-check on random values against torch's own float32 -> bfloat16 cast."""
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(7)
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-20, 20, 20000),
                        np.float32(1.0) + np.arange(512) * 2.0 ** -9]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(x.astype(np.float64)), ref)


# ----------------------------------------------------------------- RoPE position offset
@pytest.mark.parametrize("n0", [1, 5, 13])
def test_premix_pos0_window_equals_slice_of_full_sequence(n0):
    """A window starting at row n0 with pos0 = n0 reproduces rows n0.. of the
    whole-sequence result exactly (forward and input gradient)."""
    B, N, H, P, d = 2, 17, 3, 2, 16
    x = S.normal((B, N, H, d), 31, 0, dtype="f32")
    dy = S.normal((B, N, H * P, d), 31, 1, dtype="f32")
    w = S.premix_weight(H, P, 31, 2)
    full = O.premix_fwd(x, w, P, rope=True, rope_base=50.0)
    win = O.premix_fwd(np.ascontiguousarray(x[:, n0:]), w, P, rope=True, rope_base=50.0, pos0=n0)
    np.testing.assert_array_equal(win, full[:, n0:])
    fdx = O.premix_bwd_dx(dy, w, rope=True, rope_base=50.0)
    wdx = O.premix_bwd_dx(np.ascontiguousarray(dy[:, n0:]), w, rope=True, rope_base=50.0, pos0=n0)
    np.testing.assert_array_equal(wdx, fdx[:, n0:])
    # and without the offset the window would be rotated by the wrong angles
    wrong = O.premix_fwd(np.ascontiguousarray(x[:, n0:]), w, P, rope=True, rope_base=50.0)
    assert not np.allclose(wrong[:, 1:], full[:, n0 + 1:])


def test_premix_pos0_rotates_by_absolute_position():
    """pos0 = n0 equals the plain mix followed by RoPE at positions n0 + row,
    built from the d = 2 closed form (rotation by n radians when base^0 = 1)."""
    B, N, H, P, n0 = 1, 4, 2, 1, 6
    x = S.normal((B, N, H, 2), 32, 0, dtype="f32")
    w = S.premix_weight(H, P, 32, 1)
    y = O.premix_fwd(x, w, P, rope=True, rope_base=7.0, pos0=n0)
    m = O.premix_fwd(x, w, P)
    for n in range(N):
        c, s = math.cos(n0 + n), math.sin(n0 + n)
        a, b = m[0, n, :, 0], m[0, n, :, 1]
        np.testing.assert_allclose(y[0, n, :, 0], a * c - b * s, atol=1e-12)
        np.testing.assert_allclose(y[0, n, :, 1], b * c + a * s, atol=1e-12)


# ----------------------------------------------------------------- attention backward
def _bwd_inputs(B, N, Hh, d, seed):
    """bf16-valued inputs: q +- 2^-12 * u (u in {-1, 0, 1}) stays exact in fp32."""
    q, k, v, g = (S.bf16_bits_to_f32(S.normal((B, N, Hh, d), seed, c)) for c in range(4))
    return q, k, v, g


def _loss(q, k, v, g, mask, window):
    o, _ = O.attention(q[:, None], k[:, None], v[:, None], mask, window)
    return float(np.sum(o[:, 0] * g))


@pytest.mark.parametrize("mask,window", [(0, 0), (1, 0), (2, 3)])
def test_attention_bwd_matches_central_differences(mask, window):
    """<grad, u> equals the central difference of L = <dO, O> along u, for
    random sign directions u in q, k and v (the forward oracle is pinned on
    its own); the step is exact in fp32 because the inputs are bf16 values."""
    B, N, Hh, d = 1, 7, 2, 8
    q, k, v, g = _bwd_inputs(B, N, Hh, d, 51 + mask)
    dq, dk, dv = O.attention_bwd(q, k, v, g, mask, window)
    rng = np.random.default_rng(9)
    eps = 2.0 ** -12
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(3):
            u = rng.integers(-1, 2, size=x.shape).astype(np.float32)
            xp, xm = x + np.float32(eps) * u, x - np.float32(eps) * u
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name], args_m[name] = xp, xm
            fd = (_loss(args_p["q"], args_p["k"], args_p["v"], g, mask, window) -
                  _loss(args_m["q"], args_m["k"], args_m["v"], g, mask, window)) / (2 * eps)
            an = float(np.sum(grad * u))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, mask, fd, an)


@pytest.mark.parametrize("mask,window", [(0, 0), (1, 0), (2, 5)])
def test_attention_bwd_sums(mask, window):
    """Sum over keys of dV equals the sum over queries of dO (each row of P
    sums to 1); sum over keys of dK is 0 (shifting every key by one vector
    adds a constant to each row's scores, which softmax ignores)."""
    q, k, v, g = _bwd_inputs(2, 13, 3, 16, 61 + mask)
    _, dk, dv = O.attention_bwd(q, k, v, g, mask, window)
    np.testing.assert_allclose(dv.sum(axis=1), g.astype(np.float64).sum(axis=1), atol=1e-10)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-10)


def test_attention_bwd_single_visible_key_has_no_query_gradient():
    """A row that sees one key has a constant softmax: dQ = 0 there (causal
    row 0, every row of window 1), and window 1 passes dO straight to dV."""
    q, k, v, g = _bwd_inputs(1, 9, 2, 8, 71)
    dq, _, _ = O.attention_bwd(q, k, v, g, 1, 0)
    np.testing.assert_array_equal(dq[:, 0], 0.0)
    dq, dk, dv = O.attention_bwd(q, k, v, g, 2, 1)
    np.testing.assert_array_equal(dq, 0.0)
    np.testing.assert_array_equal(dk, 0.0)
    np.testing.assert_array_equal(dv, g.astype(np.float64))


def test_attention_bwd_absolute_terms_bound_the_gradients():
    """The absolute-term sums dominate the gradients element-wise and equal
    them when every term has one sign (here: dV with dO >= 0)."""
    q, k, v, g = _bwd_inputs(1, 11, 2, 8, 81)
    for mask, window in ((0, 0), (1, 0), (2, 4)):
        grads = O.attention_bwd(q, k, v, g, mask, window)
        absg = O.attention_bwd(q, k, v, g, mask, window, absolute=True)
        for a, b in zip(grads, absg):
            assert np.all(np.abs(a) <= b * (1 + 1e-12) + 1e-300)
    gp = np.abs(g)
    _, _, dv = O.attention_bwd(q, k, v, gp, 1, 0)
    _, _, av = O.attention_bwd(q, k, v, gp, 1, 0, absolute=True)
    np.testing.assert_allclose(dv, av, rtol=1e-12)


# ---------------------------------------------------------------- interleaved pseudo-tokens
def test_interleave_heads_orders_pseudo_tokens_n_major():
    """Row h*P + p of token n becomes pseudo-token (n, p) of head h; P = 1 is
    the identity."""
    B, N, H, P, d = 2, 3, 4, 3, 2
    y = np.arange(B * N * H * P * d, dtype=np.float64).reshape(B, N, H * P, d)
    z = O.interleave_heads(y, H, P)
    for b in range(B):
        for n in range(N):
            for h in range(H):
                for p in range(P):
                    np.testing.assert_array_equal(z[b, n, p, h], y[b, n, h * P + p])
    y1 = np.arange(24, dtype=np.float64).reshape(1, 3, 4, 2)
    np.testing.assert_array_equal(O.interleave_heads(y1, 4, 1)[:, :, 0], y1)


def test_joint_attention_brute_force():
    """The joint softmax, written out with loops on a tiny case: query
    pseudo-token m = n*P + p of head h sees keys m' <= m of the same head."""
    rng = np.random.default_rng(7)
    B, N, P, H, d = 2, 3, 2, 2, 4
    q, k, v = (rng.standard_normal((B, N, P, H, d)).astype(np.float32) for _ in range(3))
    o, lse = O.joint_attention(q, k, v, causal=True)
    scale = 1.0 / math.sqrt(d)
    M = N * P
    for b in range(B):
        for h in range(H):
            for m in range(M):
                n, p = divmod(m, P)
                s = np.array([scale * float(np.dot(q[b, n, p, h].astype(np.float64),
                                                   k[b, m2 // P, m2 % P, h].astype(np.float64)))
                              for m2 in range(m + 1)])
                w = np.exp(s - s.max())
                ref = sum(w[m2] * v[b, m2 // P, m2 % P, h].astype(np.float64)
                          for m2 in range(m + 1)) / w.sum()
                np.testing.assert_allclose(o[b, n, p, h], ref, rtol=1e-12, atol=1e-12)
                assert abs(lse[b, h, m] - (s.max() + math.log(w.sum()))) < 1e-12
    # no mask: every pseudo-token sees all N*P of its head
    o2, _ = O.joint_attention(q, k, v, causal=False)
    b, h, n, p = 1, 0, 0, 1
    s = np.array([scale * float(np.dot(q[b, n, p, h].astype(np.float64),
                                       k[b, m2 // P, m2 % P, h].astype(np.float64)))
                  for m2 in range(M)])
    w = np.exp(s - s.max())
    ref = sum(w[m2] * v[b, m2 // P, m2 % P, h].astype(np.float64) for m2 in range(M)) / w.sum()
    np.testing.assert_allclose(o2[b, n, p, h], ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- Hiera q_pool
def test_q_pool_stride_one_is_identity_and_blocks_are_the_slow_axis():
    """q_stride = 1 changes nothing.  With q_stride copies of one block stacked
    along the slow axis, the pool is that block, while a block made of
    rows repeated along the fast axis (t * q_stride + i) is not pooled back
    to itself (the stride is the outer axis of the unit's rows)."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 3, 12, 2, 5)).astype(np.float32)
    np.testing.assert_array_equal(O.q_pool(q, 1), q)
    blk = rng.standard_normal((2, 3, 4, 2, 5)).astype(np.float32)
    stacked = np.concatenate([blk, blk, blk], axis=2)          # rows i*4 + t
    np.testing.assert_array_equal(O.q_pool(stacked, 3), blk)
    fast = np.repeat(blk, 3, axis=2)                            # rows t*3 + i
    assert not np.array_equal(O.q_pool(fast, 3), blk)


def test_q_pool_takes_the_largest_block_value():
    """Block i filled with the value i (and a per-row offset): every pooled
    row is the last block's; the pool never leaves the inputs' values."""
    S_, Tq = 4, 5
    q = np.zeros((1, 2, S_ * Tq, 3, 8), np.float32)
    for i in range(S_):
        for t in range(Tq):
            q[:, :, i * Tq + t] = 10.0 * i + t
    pooled = O.q_pool(q, S_)
    for t in range(Tq):
        np.testing.assert_array_equal(pooled[:, :, t], 10.0 * (S_ - 1) + t)
    # bf16 bit patterns: the result is one of the inputs, exactly
    bits = (np.random.default_rng(1).integers(0, 0x7F00, (1, 1, 8, 1, 6))).astype(np.uint16)  # finite
    p = O.q_pool(bits, 2)
    widened = O._as_f32(bits)
    assert np.all((p == widened[:, :, :4]) | (p == widened[:, :, 4:]))


def test_attention_qpool_with_identical_blocks_is_plain_attention():
    """Queries made of q_stride identical blocks pool to the block, so the
    pooled attention equals plain attention of that block over all T keys;
    q_stride = 1 is plain attention."""
    rng = np.random.default_rng(5)
    Bo, Bi, Tq, Hh, d, S_ = 2, 3, 4, 2, 8, 4
    blk = rng.standard_normal((Bo, Bi, Tq, Hh, d)).astype(np.float32)
    k = rng.standard_normal((Bo, Bi, Tq * S_, Hh, d)).astype(np.float32)
    v = rng.standard_normal((Bo, Bi, Tq * S_, Hh, d)).astype(np.float32)
    q = np.concatenate([blk] * S_, axis=2)
    o, lse = O.attention_qpool(q, k, v, S_)
    ro, rl = O.attention(blk, k, v)
    np.testing.assert_allclose(o, ro, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, rl, rtol=1e-13, atol=1e-13)
    o1, _ = O.attention_qpool(q, k, v, 1)
    np.testing.assert_allclose(o1, O.attention(q, k, v)[0], rtol=1e-13, atol=1e-13)


_THREADS_SCRIPT = r"""
import sys, pickle
import numpy as np
sys.path.insert(0, sys.argv[1])
import oracle as O
import synthetic as S
B, N, H, P, d = 2, 37, 5, 3, 16
x = S.normal((B, N, H, d), 11, 0)
dy = S.normal((B, N, H * P, d), 11, 1)
w = S.premix_weight(H, P, 11, 2)
q, k, v, g = (S.normal((1, 45, 3, 16), 12, c) for c in range(4))
o, lse = O.attention(q[:, None], k[:, None], v[:, None], O.MASK_CAUSAL_WINDOW, 9)
grid = S.normal((2, 16, 6), 13, 0)
keep = S.keep_units(2, 4, 2, 13)
out = {
    "threads": O.num_threads(),
    "fwd": O.premix_fwd(x, w, P, rope=True),
    "dx": O.premix_bwd_dx(dy, w, rope=True),
    "dw": O.premix_bwd_dw(dy, x, P, rope=True),
    "o": o, "lse": lse,
    "bwd": O.attention_bwd(q, k, v, g, O.MASK_CAUSAL_WINDOW, 9),
    "gather": O.mu_gather(grid, keep, 4, 4, 2, 2),
}
sys.stdout.buffer.write(pickle.dumps(out))
"""


def test_oracle_does_not_depend_on_its_thread_count():
    """Every oracle output is computed by one thread in a fixed order, except
    dW, whose per-thread slabs are summed in slab order: so one thread and
    four give bit-identical results, and dW agrees to double rounding.  A
    race in any of the parallel loops would break this."""
    import os
    import pickle
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = []
    for n in ("1", "4"):
        env = dict(os.environ, OMP_NUM_THREADS=n)
        r = subprocess.run([sys.executable, "-c", _THREADS_SCRIPT, root], env=env,
                           capture_output=True, timeout=300)
        assert r.returncode == 0, r.stderr.decode()
        res.append(pickle.loads(r.stdout))
    a, b = res
    assert (a["threads"], b["threads"]) == (1, 4)
    for key in ("fwd", "dx", "o", "lse", "gather"):
        assert np.array_equal(a[key], b[key]), key
    for ga, gb in zip(a["bwd"], b["bwd"]):
        assert np.array_equal(ga, gb)
    np.testing.assert_allclose(a["dw"], b["dw"], rtol=1e-13, atol=1e-13 * np.abs(a["dw"]).max())
