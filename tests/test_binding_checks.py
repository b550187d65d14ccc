"""GPU tests of the Python binding's host-side checks: every tensor's shape,
dtype, device and layout is validated before the library is called, so a
mismatched buffer raises and nothing is launched (outputs stay untouched)."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_iha_gb300 as T
    T.lib()
    return T


def _z(shape, dt=None):
    import torch
    return torch.zeros(shape, dtype=dt or torch.bfloat16, device="cuda")


def test_premix_mismatches_raise(T):
    import torch
    x, w = _z((1, 8, 4, 32)), _z((4, 2, 4), torch.float32)
    with pytest.raises(ValueError):
        T.premix_fwd(x, w.to(torch.bfloat16), 2)                  # w must be fp32
    with pytest.raises(ValueError):
        T.premix_fwd(x, _z((4, 3, 4), torch.float32), 2)          # w shape vs P
    out = torch.full((1, 8, 7, 32), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        T.premix_fwd(x, w, 2, out=out)                            # wrong out shape
    assert torch.all(out == 3.0)
    with pytest.raises(ValueError):
        T.premix_fwd(_z((1, 8, 8, 32))[:, :, ::2], w, 2)          # non-contiguous x
    with pytest.raises(ValueError):
        T.premix_bwd_dx(_z((1, 8, 9, 32)), w)                     # dy heads != H*P
    with pytest.raises(ValueError):
        T.premix_bwd_dw(_z((1, 8, 8, 16)), x, 2)                  # dy d != x d
    with pytest.raises(ValueError):
        T.premix_bwd(_z((1, 8, 8, 32)), x, w, dw=_z((4, 2, 4)))   # dw must be fp32
    assert T.device_error() == 0


def test_attention_mismatches_raise(T):
    import torch
    q = _z((1, 16, 2, 64))
    with pytest.raises(ValueError):
        T.mha_fwd(q, _z((1, 16, 3, 64)), _z((1, 16, 3, 64)))      # head count
    with pytest.raises(ValueError):
        T.mha_fwd(q, _z((1, 16, 2, 64)), _z((1, 17, 2, 64)))      # k / v lengths
    with pytest.raises(ValueError):
        T.mha_fwd(q, q, q.float())                                # dtype
    with pytest.raises(ValueError):
        T.mha_fwd(q, q, q, lse=_z((1, 1, 2, 15), torch.float32))  # lse size
    out = torch.full((1, 16, 2, 32), 5.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        T.mha_fwd(q, q, q, out=out)                               # out shape
    assert torch.all(out == 5.0)


def test_mask_unit_mismatches_raise(T):
    import torch
    x = _z((2, 64, 8))
    keep = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        T.mu_gather(x, keep.long(), 8, 8, 4, 4)                   # keep must be int32
    with pytest.raises(ValueError):
        T.mu_gather(x, keep, 8, 16, 4, 4)                         # grid vs tokens
    with pytest.raises(ValueError):
        T.mu_gather(x, keep[:1], 8, 8, 4, 4)                      # keep batch
    canvas = torch.full((2, 64, 8), 2.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        T.mu_scatter(_z((2, 3, 16, 4)), keep, canvas, 8, 8, 4, 4)  # src channels
    with pytest.raises(ValueError):
        T.mu_scatter(_z((2, 3, 8, 8)), keep, canvas, 8, 8, 4, 4)   # src tokens per unit
    assert torch.all(canvas == 2.0)
    assert T.device_error() == 0
