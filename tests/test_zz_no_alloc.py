"""GPU test of the allocation-free attention backward (mha_bwd_noalloc).

Some callers cannot give the library a device buffer and cannot call
cudaMalloc themselves (a plugin whose host program owns all device memory, a
path that must not risk the device synchronization an allocation can cause).
For them the backward has an entry point whose scratch is built into the
library.  Called through the C ABI, it must give the same gradients as the
workspace entry point, on two calls in a row (the second call reuses the
scratch the first one left behind), and it must refuse a problem whose
scratch would not fit, before launching anything.

The file name sorts last, so a run that stops at the first failure has run
every other test before this one; it also passes when run on its own.
"""
import ctypes as C

import pytest

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


def _noalloc(T, q, k, v, o, g, lse, dq, dk, dv, mask, window):
    import torch
    B, N, Hh, d = q.shape
    p = lambda t: C.c_void_p(t.data_ptr())
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return T.lib().mha_bwd_noalloc(p(q), p(k), p(v), p(o), p(g), p(lse), p(dq), p(dk), p(dv),
                                   B, Hh, N, d, 0.0, mask, window, T.BF16, stream)


def test_noalloc_backward_matches_workspace_backward_on_two_calls(T):
    import torch
    problems = [((1, 700, 4, 128), T.MASK_CAUSAL, 0, 3),
                ((2, 300, 3, 64), T.MASK_CAUSAL_WINDOW, 129, 4)]
    for shape, mask, window, seed in problems:
        q, k, v, g = (to_dev(S.normal(shape, seed, c)) for c in range(4))
        o, lse = T.mha_fwd(q, k, v, mask=mask, window=window, return_lse=True)
        ref = T.mha_bwd(q, k, v, o, g, lse, mask=mask, window=window)
        got = [torch.full_like(q, 7.0) for _ in range(3)]
        assert _noalloc(T, q, k, v, o, g, lse, *got, mask, window) == 0, \
            T.lib().iha_last_error().decode()
        torch.cuda.synchronize()
        assert T.device_error() == 0
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            assert_bf16_close(to_f64(a), to_f64(b), f"{name} {shape}")


def test_noalloc_backward_refuses_oversized_scratch(T):
    import torch
    shape = (1, 8192, 16, 128)          # needs about 67 MB of scratch
    assert T.mha_bwd_workspace_bytes(1, 16, 8192, 128) > 32 << 20
    z = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 16, 8192), dtype=torch.float32, device="cuda")
    out = [torch.full_like(z, 3.0) for _ in range(3)]
    status = _noalloc(T, z, z, z, z, z, lse, *out, T.MASK_CAUSAL, 0)
    assert status == 2
    assert "scratch" in T.lib().iha_last_error().decode()
    torch.cuda.synchronize()
    assert all(bool(torch.all(t == 3.0)) for t in out)
    assert T.device_error() == 0
