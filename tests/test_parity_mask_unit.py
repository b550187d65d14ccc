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
