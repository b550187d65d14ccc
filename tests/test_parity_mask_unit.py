"""GPU parity: mask-unit gather / scatter (bit-exact) and the Hiera-Base MAE
stage-1 step (gather -> mask-unit attention -> scatter) vs the oracle."""
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


def _bits(t):
    import torch
    return t.cpu().contiguous().view(torch.uint8).numpy()


GEOMS = [  # (B, grid_h, grid_w, mu_h, mu_w, n_keep, C, dtype)
    (3, 16, 24, 4, 8, 5, 96, np.uint16),     # 192-byte rows: 16-byte path
    (2, 8, 8, 2, 2, 16, 5, np.uint16),       # 10-byte rows: byte path
    (2, 12, 6, 3, 3, 1, 6, np.float32),      # 24-byte rows: 4-byte path
    (1, 4, 4, 2, 2, 4, 8, np.uint16),        # every unit kept
]


@pytest.mark.parametrize("geom", GEOMS)
def test_gather_scatter_bit_exact(T, geom):
    import torch
    B, gh, gw, mh, mw, nk, Cc, dt = geom
    sh = S.MaskUnitShape(B=B, grid_h=gh, grid_w=gw, mu_h=mh, mu_w=mw, n_keep=nk, C=Cc)
    x = S.normal((B, gh * gw, Cc), 21, 0, dtype="bf16" if dt == np.uint16 else "f32")
    keep = S.keep_units(B, sh.n_units, nk, 22)
    xd, kd = to_dev(x), to_dev(keep)
    g = T.mu_gather(xd, kd, gh, gw, mh, mw)
    ref = O.mu_gather(x, keep, gh, gw, mh, mw)
    np.testing.assert_array_equal(_bits(g), ref.view(np.uint8).reshape(_bits(g).shape))
    canvas = S.normal((B, gh * gw, Cc), 23, 0, dtype="bf16" if dt == np.uint16 else "f32")
    cd = to_dev(canvas)
    src = S.normal((B, nk, mh * mw, Cc), 24, 0, dtype="bf16" if dt == np.uint16 else "f32")
    T.mu_scatter(to_dev(src), kd, cd, gh, gw, mh, mw)
    ref = O.mu_scatter(src, keep, canvas, gh, gw, mh, mw)
    np.testing.assert_array_equal(_bits(cd), ref.view(np.uint8).reshape(_bits(cd).shape))
    assert T.device_error() == 0


def test_gather_flags_out_of_range_unit_and_skips_it(T):
    """A keep id >= units is skipped on the GPU and raises the device error word."""
    import torch
    x = to_dev(S.normal((1, 16, 8), 25, 0))
    keep = torch.tensor([[1, 4]], dtype=torch.int32, device="cuda")   # 4 units: id 4 is invalid
    out = torch.zeros((1, 2, 4, 8), dtype=torch.bfloat16, device="cuda")
    T.mu_gather(x, keep, 4, 4, 2, 2, out=out)
    assert T.device_error(clear=True) == 1
    assert torch.all(out[0, 1] == 0)
    assert T.device_error() == 0


def test_hiera_mae_stage1_step(T):
    """B=128, 56x56 tokens, 8x8 units, 20 kept per sample, C = d = 96, one head.
    Gather the kept units, attend within each 64-token unit (Q = K = V = the
    gathered tokens, no mask), scatter the result back; every stage against
    the oracle (attention for all 2560 units)."""
    import torch
    sh = S.HIERA_MU
    x = S.normal((sh.B, sh.grid_h * sh.grid_w, sh.C), 0, 0)
    keep = S.keep_units(sh.B, sh.n_units, sh.n_keep, 0)
    xd, kd = to_dev(x), to_dev(keep)
    g = T.mu_gather(xd, kd, sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w)
    gref = O.mu_gather(x, keep, sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w)
    np.testing.assert_array_equal(_bits(g), gref.view(np.uint8).reshape(_bits(g).shape))
    units = g.view(sh.B * sh.n_keep, 1, sh.unit_tokens, 1, sh.C)       # [Bo, Bi, T, Hh, d]
    o = T.mha_fwd(units, units, units)
    u = gref.reshape(sh.B * sh.n_keep, 1, sh.unit_tokens, 1, sh.C)
    ro, _ = O.attention(u, u, u)
    assert_bf16_close(to_f64(o), ro, "mask-unit attention")
    dec = torch.zeros_like(xd)
    T.mu_scatter(o.view(sh.B, sh.n_keep, sh.unit_tokens, sh.C), kd, dec, sh.grid_h, sh.grid_w,
                 sh.mu_h, sh.mu_w)
    obits = o.cpu().view(torch.int16).numpy().view(np.uint16).reshape(sh.B, sh.n_keep,
                                                                      sh.unit_tokens, sh.C)
    dref = O.mu_scatter(obits, keep, np.zeros_like(x), sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w)
    np.testing.assert_array_equal(_bits(dec), dref.view(np.uint8).reshape(_bits(dec).shape))
    assert T.device_error() == 0


FUSED_GEOMS = [  # (B, grid_h, grid_w, mu_h, mu_w, n_keep, C)
    (2, 16, 16, 8, 8, 2, 96),    # the stage-1 unit, an even number of units
    (3, 16, 24, 8, 8, 5, 128),   # odd unit count: the last pair has one unit
    (2, 12, 12, 4, 4, 7, 64),    # 16-token units (rows 16..63 of each half unused)
    (1, 8, 24, 4, 8, 3, 32),     # rectangular units, one 64-channel chunk
]


def _oracle_fused(x, keep, canvas, gh, gw, mh, mw):
    """gather -> attention inside each unit (Q = K = V) -> scatter, by the oracle."""
    B, G, Cc = x.shape
    nk = keep.shape[1]
    g = O.mu_gather(x, keep, gh, gw, mh, mw)
    u = g.reshape(B * nk, 1, mh * mw, 1, Cc)
    ro, _ = O.attention(u, u, u)
    return g, ro.reshape(B, nk, mh * mw, Cc)


@pytest.mark.parametrize("geom", FUSED_GEOMS)
def test_fused_gather_attention_scatter(T, geom):
    """One pass equals the three-op step: against the oracle on the kept
    tokens, bit-equal to gather -> mha_fwd -> scatter on the GPU, and every
    other canvas token untouched."""
    import torch
    B, gh, gw, mh, mw, nk, Cc = geom
    sh = S.MaskUnitShape(B=B, grid_h=gh, grid_w=gw, mu_h=mh, mu_w=mw, n_keep=nk, C=Cc)
    x = S.normal((B, gh * gw, Cc), 31, 0)
    keep = S.keep_units(B, sh.n_units, nk, 32)
    canvas = S.normal((B, gh * gw, Cc), 33, 0)           # sentinel values
    xd, kd, cd = to_dev(x), to_dev(keep), to_dev(canvas)
    T.mu_attention_fused(xd, kd, cd, gh, gw, mh, mw)
    torch.cuda.synchronize()
    assert T.device_error() == 0
    # kept tokens: the oracle's attention output, read back through its gather
    _, ro = _oracle_fused(x, keep, canvas, gh, gw, mh, mw)
    got_units = T.mu_gather(cd, kd, gh, gw, mh, mw)
    assert_bf16_close(to_f64(got_units), ro, f"fused {geom}")
    # every token of a unit not kept is unchanged
    ones = np.ones((B, gh * gw, 1), np.uint16)
    mark = O.mu_scatter(O.mu_gather(ones, keep, gh, gw, mh, mw), keep,
                        np.zeros((B, gh * gw, 1), np.uint16), gh, gw, mh, mw)
    kept = mark[..., 0] == 1
    cbits = _bits(cd).reshape(B, gh * gw, Cc * 2)
    ref_bits = canvas.view(np.uint8).reshape(B, gh * gw, Cc * 2)
    np.testing.assert_array_equal(cbits[~kept], ref_bits[~kept])
    # bit-equal to the three-launch GPU path
    g = T.mu_gather(xd, kd, gh, gw, mh, mw)
    un = g.view(B * nk, 1, mh * mw, 1, Cc)
    o = T.mha_fwd(un, un, un)
    c2 = to_dev(canvas)
    T.mu_scatter(o.view(B, nk, mh * mw, Cc), kd, c2, gh, gw, mh, mw)
    np.testing.assert_array_equal(_bits(cd), _bits(c2))
    assert T.device_error() == 0


def test_fused_flags_out_of_range_unit_and_skips_it(T):
    """An out-of-range kept-unit id skips that unit (its tokens untouched)
    and raises the device error word; the other unit is still computed."""
    import torch
    gh = gw = 16
    x = S.normal((1, gh * gw, 64), 34, 0)
    keep = np.array([[1, 99]], np.int32)  # 4 units: id 99 is invalid
    canvas = torch.zeros((1, gh * gw, 64), dtype=torch.bfloat16, device="cuda")
    T.mu_attention_fused(to_dev(x), to_dev(keep), canvas, gh, gw, 8, 8)
    torch.cuda.synchronize()
    assert T.device_error(clear=True) == 1
    _, ro = _oracle_fused(x, keep[:, :1], None, gh, gw, 8, 8)
    got = T.mu_gather(canvas, to_dev(keep[:, :1]), gh, gw, 8, 8)
    assert_bf16_close(to_f64(got), ro, "fused, valid unit")
    # only unit 1's 64 tokens were written
    assert int((canvas.view(-1, 64).abs().sum(dim=1) > 0).sum()) <= 64
    assert T.device_error() == 0


def test_fused_hiera_stage1_matches_three_launches(T):
    """B=128, 56x56 tokens, 8x8 units, 20 kept, C=96: bit-equal to gather ->
    mha_fwd -> scatter, and the oracle on a sample of units."""
    import torch
    sh = S.HIERA_MU
    x = S.normal((sh.B, sh.grid_h * sh.grid_w, sh.C), 0, 0)
    keep = S.keep_units(sh.B, sh.n_units, sh.n_keep, 0)
    xd, kd = to_dev(x), to_dev(keep)
    cd = torch.zeros_like(xd)
    T.mu_attention_fused(xd, kd, cd, sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w)
    g = T.mu_gather(xd, kd, sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w)
    un = g.view(sh.B * sh.n_keep, 1, sh.unit_tokens, 1, sh.C)
    o = T.mha_fwd(un, un, un)
    c2 = torch.zeros_like(xd)
    T.mu_scatter(o.view(sh.B, sh.n_keep, sh.unit_tokens, sh.C), kd, c2, sh.grid_h, sh.grid_w,
                 sh.mu_h, sh.mu_w)
    np.testing.assert_array_equal(_bits(cd), _bits(c2))
    b = np.array([0, 63, 127])
    _, ro = _oracle_fused(x[b], keep[b], None, sh.grid_h, sh.grid_w, sh.mu_h, sh.mu_w)
    bt = torch.as_tensor(b, device="cuda")
    got = T.mu_gather(cd[bt].contiguous(), kd[bt].contiguous(), sh.grid_h, sh.grid_w, sh.mu_h,
                      sh.mu_w)
    assert_bf16_close(to_f64(got), ro, "fused stage 1, samples 0 / 63 / 127")
    assert T.device_error() == 0
